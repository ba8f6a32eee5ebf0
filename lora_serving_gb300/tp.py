"""Tensor-parallel LoRA delta: the adapter sharded like the base layer, one
exchange per projection on the small fp32 intermediate v [T][r].

TGI multi-LoRA page, "5. LoRA under tensor parallelism": the adapter's
matrices are split the way the base weight is, and the ranks meet on v.
Two layouts (the reading of the page's "A by column, B by row" used here):

* column-parallel projection (q/k/v, gate/up: the output columns split over
  the N ranks).  Rank i holds rows [i r/N, (i+1) r/N) of every A (a slice of
  the adapter's ranks) and the rows of B' for its output columns.  It forms
  its slice of v, ``all_gather`` assembles v in rank order, and it adds
  B'_i v to its output columns.
* row-parallel projection (o, down: the input split over the ranks).  Rank i
  holds the columns of A for its input slice and all of B'.  Its partial
  v_i = A_i x_i is summed by ``all_reduce``, and every rank adds B' v to the
  (replicated) output.

This module only shards and exchanges.  The steps that touch adapter
weights are passed in: on GPUs the library's kernels (``kernel_steps``), in
the CPU tests oracle functions.  With one rank no collective is issued.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.distributed as dist


def _split(n: int, world: int, rank: int) -> slice:
    if n % world:
        raise ValueError(f"{n} does not split evenly over {world} ranks")
    return slice(rank * n // world, (rank + 1) * n // world)


def _own(t):
    """A contiguous copy: a rank keeps only its shard."""
    return t.contiguous() if hasattr(t, "contiguous") else np.ascontiguousarray(t)


def shard_column(A, B, world: int, rank: int):
    """A [..][r][h_in], B [..][out][r] -> this rank's rows of A (ranks) and of B (outputs)."""
    return _own(A[..., _split(A.shape[-2], world, rank), :]), _own(B[..., _split(B.shape[-2], world, rank), :])


def shard_row(A, B, world: int, rank: int):
    """A [..][r][h_in], B [..][out][r] -> this rank's columns of A (inputs) and all of B."""
    return _own(A[..., _split(A.shape[-1], world, rank)]), B


def column_parallel(x, y_shard, A_shard, B_shard, shrink, expand, world: int = 1, group=None):
    """y_shard (this rank's output columns) += B'_shard v with v all-gathered
    from the ranks' slices.  shrink(x, A_shard) -> v slice [T][r/N] (fp32 or
    fp64 tensor); expand(y_shard, v, B_shard) -> updated y_shard."""
    v_part = shrink(x, A_shard).contiguous()
    if world > 1:
        parts = [torch.empty_like(v_part) for _ in range(world)]
        dist.all_gather(parts, v_part, group=group)
        v = torch.cat(parts, dim=1)
    else:
        v = v_part
    return expand(y_shard, v, B_shard)


def row_parallel(x_shard, y, A_shard, B, shrink, expand, world: int = 1, group=None):
    """y += B' v with v = sum over ranks of A_i x_i (all-reduced).
    shrink(x_shard, A_shard) -> partial v [T][r]; expand(y, v, B) -> updated y."""
    v = shrink(x_shard, A_shard).contiguous()
    if world > 1:
        dist.all_reduce(v, group=group)
    return expand(y, v, B)


def kernel_steps(lora_ids, n_slots: int, dev_status=None, stream=None):
    """shrink / expand steps on the library's per-token kernels (BGMV) for a
    batch with per-row slot ids ``lora_ids`` (device int32, -1 = base):
    stores are [n_slots][r][h_in] and [n_slots][w][r], v is fp32."""
    from . import abi

    def shrink(x, A_store):
        r, h_in = int(A_store.shape[1]), int(A_store.shape[2])
        v = torch.zeros(x.shape[0], r, dtype=torch.float32, device=x.device)
        abi.lora_bgmv_shrink(v, x, A_store, lora_ids, h_in=h_in, r_slot=r, n_slots=n_slots,
                             dev_status=dev_status, stream=stream)
        return v

    def expand(y, v, B_store):
        w, r = int(B_store.shape[1]), int(B_store.shape[2])
        abi.lora_bgmv_expand(y, 0, w, v.contiguous(), B_store.contiguous(), lora_ids, r_slot=r,
                             n_slots=n_slots, dev_status=dev_status, stream=stream)
        return y

    return shrink, expand
