"""Tensor-parallel LoRA on two gloo ranks (CPU): the sharding and the one
exchange per projection (all_gather for column-parallel, all_reduce for
row-parallel), with the weight-touching steps done by the oracle.  The
result must equal the oracle's unsharded delta: bit for bit for the
column-parallel form (every v entry is computed whole on one rank), within
the bf16 tolerance for the row-parallel form (v summed in another grouping).

The shards are taken from slot stores padded to the slot rank (zero rows of
A, zero columns of B beyond an adapter's rank), as the library lays them
out, so every rank owns the same number of v columns for every slot."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle as O
from helpers import check_bf16
from lora_serving_gb300 import tp

T, H_IN, OUT, WORLD = 9, 64, 48, 2
RANKS = [4, 8, 6]          # 6: a rank that does not split evenly, padded
R_SLOT = 8


def _problem():
    g = torch.Generator().manual_seed(41)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    A = [bits((torch.randn(r, H_IN, generator=g) * 0.2).to(torch.bfloat16)) for r in RANKS]
    B = [bits((torch.randn(OUT, r, generator=g) * 0.2).to(torch.bfloat16)) for r in RANKS]
    scales = [O.scale(2.0 * r, r, False) for r in RANKS]
    x = bits(torch.randn(T, H_IN, generator=g).to(torch.bfloat16))
    y = bits(torch.randn(T, OUT, generator=g).to(torch.bfloat16))
    ids = np.array([0, 1, -1, 2, 2, 0, 1, -1, 2], np.int32)
    return A, B, scales, x, y, ids


def _padded(A, B):
    Ap = [np.pad(a, ((0, R_SLOT - a.shape[0]), (0, 0))) for a in A]
    Bp = [np.pad(b, ((0, 0), (0, R_SLOT - b.shape[1]))) for b in B]
    return Ap, Bp


def _oracle_steps(ids, scales):
    """shrink / expand done by the oracle on per-slot lists of bf16 bits."""
    def shrink(x, A_list):
        dummy_B = [np.zeros((1, a.shape[0]), np.uint16) for a in A_list]
        return torch.from_numpy(O.shrink(ids, x, O.Adapters(A_list, dummy_B, scales)))

    def expand(y, v, B_list):
        dummy_A = [np.zeros((b.shape[1], 8), np.uint16) for b in B_list]
        return O.expand(ids, v.numpy(), y, 0, O.Adapters(dummy_A, B_list, scales))
    return shrink, expand


def _rank_main(rank, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        A, B, scales, x, y, ids = _problem()
        A, B = _padded(A, B)
        shrink, expand = _oracle_steps(ids, scales)
        # column-parallel: rows of A (ranks) and of B (outputs) split
        shards = [tp.shard_column(a, b, WORLD, rank) for a, b in zip(A, B)]
        cols = tp._split(OUT, WORLD, rank)
        y_col = tp.column_parallel(x, np.ascontiguousarray(y[:, cols]), [s[0] for s in shards],
                                   [s[1] for s in shards], shrink, expand, WORLD)
        parts = [torch.empty(T, OUT // WORLD, dtype=torch.int32) for _ in range(WORLD)]
        dist.all_gather(parts, torch.from_numpy(y_col.astype(np.int32)))   # gloo has no 16-bit ints
        y_col_full = torch.cat(parts, dim=1).numpy().astype(np.uint16)
        # row-parallel: columns of A (inputs) split, x split likewise, B whole
        ks = tp._split(H_IN, WORLD, rank)
        rshards = [tp.shard_row(a, b, WORLD, rank) for a, b in zip(A, B)]
        y_row = tp.row_parallel(np.ascontiguousarray(x[:, ks]), y, [s[0] for s in rshards],
                                [s[1] for s in rshards], shrink, expand, WORLD)
        q.put((rank, y_col_full, y_row))
    except BaseException as e:
        q.put((rank, None, repr(e)))
        raise
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.timeout(180)
def test_tp_two_gloo_ranks_match_the_unsharded_oracle():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(WORLD)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=150) for _ in range(WORLD)), key=lambda t: t[0])
    for p in procs:
        p.join(timeout=30)
    for rank, y_col, y_row in res:
        assert y_col is not None, f"rank {rank} failed: {y_row}"
    assert all(p.exitcode == 0 for p in procs)
    A, B, scales, x, y, ids = _problem()
    ref = O.apply_projection(ids, x, y, 0, O.Adapters(A, B, scales))
    for rank, y_col, y_row in res:
        np.testing.assert_array_equal(y_col, ref, err_msg=f"column-parallel, rank {rank}")
        check_bf16(y_row, ref, ids, y, f"row-parallel, rank {rank}")
    np.testing.assert_array_equal(res[0][2], res[1][2])   # every rank holds the same output


def test_shards_reject_uneven_splits():
    A = np.zeros((6, 64), np.uint16)
    B = np.zeros((48, 6), np.uint16)
    with pytest.raises(ValueError):
        tp.shard_column(A, B, 4, 0)
