"""Seeded synthetic workloads for the multi-LoRA delta (inputs only).

This module draws the inputs that both the CUDA library and the CPU oracle
consume; it holds none of the method's arithmetic (no scaling, folding,
padding, metadata or products).  bf16 tensors are returned as numpy
``uint16`` bit patterns.

Recipe (shapes follow the five workloads of the LoRA-serving pages' sizing):
  * weights: lora_A [r][h_in] and lora_B [out][r] per adapter and projection,
    i.i.d. N(0, 0.02^2) rounded to bf16 (B is non-zero, unlike peft's init);
  * x: N(0, 1) rounded to bf16, one matrix per projection group;
  * y_in: zeros ("delta" mode) or N(0, 1) in bf16 ("accumulate" mode);
  * base weights (the linear layer): the group's stacked W [out][h_in],
    i.i.d. N(0, 1/h_in) in bf16, so that x W^T is of order one;
  * adapter ids: per workload, see the builders below.
Draw order: batch structure (lengths, ids) -> adapters (slot, group,
projection; A then B) -> x per group -> y_in per group.  Every tensor is
drawn in chunks of 2^24 elements, each from its own torch generator seeded
by a hash of (workload seed, tensor tag, chunk index), so the values do not
depend on the number of threads.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
from dataclasses import dataclass, field

import numpy as np
import torch

_CHUNK = 1 << 24


def _seed_of(*key) -> int:
    """63-bit seed from a tuple of integers (sha256: the same on every machine)."""
    data = b"".join(int(k).to_bytes(16, "little", signed=True) for k in key)
    return int.from_bytes(hashlib.sha256(data).digest()[:8], "little") >> 1


def _tag(s: str) -> int:
    return int.from_bytes(hashlib.sha256(s.encode()).digest()[:8], "little") >> 1


class _Stream:
    """splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
    generators", 2014) for the batch-structure draws, so lengths and ids are
    the same on every machine and numpy version."""

    _M = (1 << 64) - 1

    def __init__(self, seed: int):
        self.s = int(seed) & self._M

    def u64(self) -> int:
        self.s = (self.s + 0x9E3779B97F4A7C15) & self._M
        z = self.s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & self._M
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & self._M
        return z ^ (z >> 31)

    def random(self, n: int) -> np.ndarray:
        return np.array([(self.u64() >> 11) * 2.0 ** -53 for _ in range(n)])

    def integers(self, lo: int, hi: int, n: int) -> np.ndarray:
        """Uniform in [lo, hi) (rejection-free multiply-shift; bias < 2^-32)."""
        span = hi - lo
        return np.array([lo + ((self.u64() >> 32) * span >> 32) for _ in range(n)], np.int64)

    def choice_p(self, p: np.ndarray, n: int) -> np.ndarray:
        cdf = np.cumsum(p)
        cdf[-1] = 1.0
        return np.searchsorted(cdf, self.random(n), side="right").astype(np.int64)

    def permutation(self, a: np.ndarray) -> np.ndarray:
        a = np.array(a, copy=True)
        for i in range(a.size - 1, 0, -1):   # Fisher-Yates
            j = int(self.integers(0, i + 1, 1)[0])
            a[i], a[j] = a[j], a[i]
        return a


def normal_bf16(shape, std: float, seed: int, tag: str) -> np.ndarray:
    """N(0, std^2) rounded to bf16 (torch's round-to-nearest-even), as uint16 bits."""
    n = int(np.prod(shape))
    out = torch.empty(n, dtype=torch.bfloat16)
    t = _tag(tag)

    def fill(c):
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = torch.Generator().manual_seed(_seed_of(seed, t, c))
        out[lo:hi] = (torch.randn(hi - lo, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)

    n_chunks = (n + _CHUNK - 1) // _CHUNK
    if n_chunks <= 1:
        for c in range(n_chunks):
            fill(c)
    else:
        with cf.ThreadPoolExecutor(max_workers=min(n_chunks, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.view(torch.int16).numpy().view(np.uint16).reshape(shape)


@dataclass
class Group:
    """Projections that share one input x (q/k/v, gate/up) or a single one."""
    name: str
    h_in: int
    projs: list  # [(name, width)]

    @property
    def ld_y(self) -> int:
        return sum(w for _, w in self.projs)

    @property
    def offsets(self):
        offs, o = [], 0
        for _, w in self.projs:
            offs.append(o)
            o += w
        return offs


@dataclass
class Workload:
    name: str
    seed: int
    groups: list
    ranks: np.ndarray          # true rank per adapter slot
    alphas: np.ndarray         # lora_alpha per slot
    rslora: np.ndarray         # bool per slot
    r_slot: int                # slot rank the store is padded to
    ids: np.ndarray            # int32 [T], -1 = base
    n_prefill: int
    seg_lens: list = field(default_factory=list)  # prefill request lengths, in order
    # filled by materialise()
    A: dict = field(default_factory=dict)   # (group, proj, slot) -> [r][h_in] bits
    B: dict = field(default_factory=dict)   # (group, proj, slot) -> [w][r] bits
    x: dict = field(default_factory=dict)   # group -> [T][h_in] bits
    y: dict = field(default_factory=dict)   # group -> [T][ld_y] bits
    y_mode: str = "delta"

    @property
    def n_slots(self) -> int:
        return len(self.ranks)

    @property
    def n_rows(self) -> int:
        return int(self.ids.size)

    def materialise(self, y_mode: str = "delta", groups=None, weights: bool = True, layer: int = 0):
        """Draws adapters, x and y_in (for the named groups, default all).
        ``layer`` > 0 draws an independent layer instance of the same shapes."""
        self.y_mode = y_mode
        names = [g.name for g in self.groups] if groups is None else list(groups)
        L = f"L{layer}" if layer else ""
        if weights:
            for k in range(self.n_slots):
                r = int(self.ranks[k])
                for g in self.groups:
                    if g.name not in names:
                        continue
                    for pname, w in g.projs:
                        self.A[(g.name, pname, k)] = normal_bf16((r, g.h_in), 0.02, self.seed, f"A{g.name}{pname}{k}{L}")
                        self.B[(g.name, pname, k)] = normal_bf16((w, r), 0.02, self.seed, f"B{g.name}{pname}{k}{L}")
        T = self.n_rows
        for g in self.groups:
            if g.name not in names:
                continue
            self.x[g.name] = normal_bf16((T, g.h_in), 1.0, self.seed, f"x{g.name}{L}")
        for g in self.groups:
            if g.name not in names:
                continue
            if y_mode == "delta":
                self.y[g.name] = np.zeros((T, g.ld_y), np.uint16)
            else:
                self.y[g.name] = normal_bf16((T, g.ld_y), 1.0, self.seed, f"y{g.name}{L}")
        return self

    def base_weight(self, group: str, layer: int = 0) -> np.ndarray:
        """The group's stacked base weight [sum of widths][h_in] (bf16 bits)."""
        g = next(g for g in self.groups if g.name == group)
        L = f"L{layer}" if layer else ""
        return normal_bf16((g.ld_y, g.h_in), 1.0 / np.sqrt(g.h_in), self.seed, f"W{g.name}{L}")


# ------------------------------------------------------------ workloads ----

def tiny() -> Workload:
    """hidden 256, one projection 256->256, 4 adapters of rank 8, alpha 16;
    prefill segments of 5/17/32 rows with ids 0/2/-1, then six decode tokens
    with ids [1,3,3,0,-1,2]; seed 0."""
    ids = np.array([0] * 5 + [2] * 17 + [-1] * 32 + [1, 3, 3, 0, -1, 2], np.int32)
    return Workload("tiny", 0, [Group("proj", 256, [("proj", 256)])],
                    np.full(4, 8), np.full(4, 16.0), np.zeros(4, bool), 8, ids, 54, [5, 17, 32])


def llama3b_decode(n_tokens: int = 64) -> Workload:
    """Llama-3.2-3B-shaped decode: hidden 3072, q 3072 / k,v 1024 (GQA) / o
    3072; 8 adapter slots, all rank 16, alpha 32; 64 decode tokens, each
    base-only with p = 0.1, else an adapter uniform over the 8; seed 1."""
    seed = 1
    g = _Stream(_seed_of(seed, _tag("ids")))
    base = g.random(n_tokens) < 0.1
    ids = np.where(base, -1, g.integers(0, 8, n_tokens)).astype(np.int32)
    groups = [Group("qkv", 3072, [("q", 3072), ("k", 1024), ("v", 1024)]),
              Group("o", 3072, [("o", 3072)])]
    return Workload("llama3b_decode", seed, groups, np.full(8, 16), np.full(8, 32.0),
                    np.zeros(8, bool), 16, ids, 0)


def mistral7b_prefill(n_seqs: int = 32) -> Workload:
    """Mistral-7B-shaped prefill: hidden 4096, q 4096 / k,v 1024 / o 4096 /
    gate,up 14336 / down 14336->4096; 16 adapters with ranks drawn i.i.d. from
    {8,16,32,64}, padded to 64; rsLoRA on the even-indexed half; alpha 16 for
    all; 32 sequences of lengths uniform in [64, 2048], each on an adapter
    uniform over the 16; contiguous segments; no base-only rows; seed 2."""
    seed = 2
    g = _Stream(_seed_of(seed, _tag("ids")))
    ranks = np.array([8, 16, 32, 64])[g.integers(0, 4, 16)]
    lens = g.integers(64, 2049, n_seqs)
    seq_ids = g.integers(0, 16, n_seqs)
    ids = np.repeat(seq_ids, lens).astype(np.int32)
    groups = [Group("qkv", 4096, [("q", 4096), ("k", 1024), ("v", 1024)]),
              Group("o", 4096, [("o", 4096)]),
              Group("gate_up", 4096, [("gate", 14336), ("up", 14336)]),
              Group("down", 14336, [("down", 4096)])]
    rs = (np.arange(16) % 2) == 0
    return Workload("mistral7b_prefill", seed, groups, ranks, np.full(16, 16.0), rs, 64, ids,
                    int(ids.size), [int(v) for v in lens])


def mixed(n_decode: int = 256, n_prefill_segs: int = 8) -> Workload:
    """Mixed continuous batch: hidden 4096, q/k/v/o Mistral-shaped; 64
    adapters of rank 16, alpha 32; 8 prefill requests of lengths uniform in
    [128, 1024] followed by 256 decode rows; each request is base-only with
    p = 0.2, else its adapter follows Zipf(s = 1.1) over popularity ranks
    1..64 (id = rank - 1); seed 3."""
    seed = 3
    g = _Stream(_seed_of(seed, _tag("ids")))
    pz = 1.0 / np.arange(1, 65) ** 1.1
    pz /= pz.sum()

    def draw(n):
        base = g.random(n) < 0.2
        return np.where(base, -1, g.choice_p(pz, n)).astype(np.int32)

    lens = g.integers(128, 1025, n_prefill_segs)
    pre = np.repeat(draw(n_prefill_segs), lens)
    dec = draw(n_decode)
    ids = np.concatenate([pre, dec]).astype(np.int32)
    groups = [Group("qkv", 4096, [("q", 4096), ("k", 1024), ("v", 1024)]),
              Group("o", 4096, [("o", 4096)])]
    return Workload("mixed", seed, groups, np.full(64, 16), np.full(64, 32.0), np.zeros(64, bool),
                    16, ids, int(pre.size), [int(v) for v in lens])


def stress70b(n_tokens: int = 512) -> Workload:
    """70B-shaped stress: hidden 8192, gate/up 8192->28672, down 28672->8192;
    128 adapters of rank 64, alpha 128 (above the BGMV cap, so SGMV); 512
    decode tokens whose ids are a seeded random permutation of each of the
    128 ids repeated 4 times (512 tokens cannot all be distinct over 128
    adapters: every adapter is touched, by 4 scattered tokens); seed 4."""
    seed = 4
    g = _Stream(_seed_of(seed, _tag("ids")))
    ids = g.permutation(np.repeat(np.arange(128), n_tokens // 128)).astype(np.int32)
    groups = [Group("gate_up", 8192, [("gate", 28672), ("up", 28672)]),
              Group("down", 28672, [("down", 8192)])]
    return Workload("stress70b", seed, groups, np.full(128, 64), np.full(128, 128.0),
                    np.zeros(128, bool), 64, ids, 0)


WORKLOADS = {
    "tiny": tiny,
    "llama3b_decode": llama3b_decode,
    "mistral7b_prefill": mistral7b_prefill,
    "mixed": mixed,
    "stress70b": stress70b,
}


def get(name: str, **kw) -> Workload:
    return WORKLOADS[name](**kw)
