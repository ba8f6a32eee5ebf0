"""Shared helpers for the parity tests: device transfer of bf16 bit arrays,
the oracle reference for a workload group, and the tolerance check.

Tolerance (the stated bar): against the fp64 oracle rounded to bf16, the
relative L2 error of the written outputs is <= 1e-3 and the max abs error is
<= 3e-2.  Reading used where one bf16 step exceeds 3e-2 (|y| >= 4, where
the spacing is 2^-5 = 0.03125): such an element may differ from the oracle by
at most one bf16 step; the count of such elements is returned.  Rows whose
id is -1 must be bit-identical to y_in.

One more figure, stricter than the stated bar: at least MIN_EXACT of the
adapter rows' elements must equal the oracle's value bit for bit.  A
kernel that forms y + delta in fp32 and rounds once agrees with the
correctly rounded fp64 result except where y lies within the fp32 error of
a rounding boundary (about 1e-4 of the elements).  The rel-L2 figure
alone is weak in accumulate mode, where y_in ~ N(0,1) dominates the norm:
a delta 0.1 % too large moves rel-L2 to only 8.5e-4 there, but leaves 10 %
of the elements one step off.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

REL_L2 = 1e-3
MAX_ABS = 3e-2
MIN_EXACT = 0.95


def to_dev(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_host(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def oracle_adapters(wl, group, pname):
    A = [wl.A[(group, pname, k)] for k in range(wl.n_slots)]
    B = [wl.B[(group, pname, k)] for k in range(wl.n_slots)]
    scales = [O.scale(float(wl.alphas[k]), int(wl.ranks[k]), bool(wl.rslora[k])) for k in range(wl.n_slots)]
    return O.Adapters(A, B, scales)


def oracle_group(wl, gname, rows=None):
    """Oracle output y for the group's rows (all, or the given row indices)."""
    g = next(g for g in wl.groups if g.name == gname)
    rows = np.arange(wl.n_rows) if rows is None else np.asarray(rows)
    ids = wl.ids[rows]
    x = wl.x[gname][rows]
    y = wl.y[gname][rows].copy()
    for (pname, _), off in zip(g.projs, g.offsets):
        y = O.apply_projection(ids, x, y, off, oracle_adapters(wl, gname, pname))
    return y


def oracle_group_all_rows(wl, gname, block: int = 256):
    """Oracle output y for every row of the group, row blocks computed on a
    thread pool over all host cores (the oracle's C calls release the GIL;
    each row's result depends on that row alone)."""
    import concurrent.futures as cf
    import os
    g = next(g for g in wl.groups if g.name == gname)
    ads = [oracle_adapters(wl, gname, pname) for pname, _ in g.projs]
    out = wl.y[gname].copy()

    def run(lo):
        hi = min(wl.n_rows, lo + block)
        y = wl.y[gname][lo:hi].copy()
        for ad, off in zip(ads, g.offsets):
            y = O.apply_projection(wl.ids[lo:hi], wl.x[gname][lo:hi], y, off, ad)
        out[lo:hi] = y

    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
        list(ex.map(run, range(0, wl.n_rows, block)))
    return out


def bf16_step(vals: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |vals| (2^(e-7) for |v| in [2^e, 2^(e+1)))."""
    a = np.abs(vals)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def check_bf16(got_bits, ref_bits, ids, yin_bits, what=""):
    """Asserts the tolerance on rows with id >= 0 and bit-identity elsewhere.
    Returns a dict of error figures."""
    got_bits = np.asarray(got_bits)
    ref_bits = np.asarray(ref_bits)
    base = np.asarray(ids) < 0
    if base.any():
        np.testing.assert_array_equal(got_bits[base], np.asarray(yin_bits)[base],
                                      err_msg=f"{what}: base-only rows changed")
    act = ~base
    if not act.any():
        return {"rel_l2": 0.0, "max_abs": 0.0, "n_big_step": 0, "n": 0, "exact": 1.0}
    got = O.bf16_to_f64(got_bits[act])
    ref = O.bf16_to_f64(ref_bits[act])
    err = np.abs(got - ref)
    den = np.sqrt(np.sum(ref * ref))
    rel = float(np.sqrt(np.sum(err * err)) / den) if den > 0 else float(np.sqrt(np.sum(err * err)))
    over = err > MAX_ABS
    big = over & (err <= bf16_step(ref) * (1 + 1e-9))
    bad = over & ~big
    n_big = int(big.sum())
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2} ({n_big} elements one bf16 step off)"
    assert not bad.any(), (f"{what}: {int(bad.sum())} elements off by more than "
                           f"max(3e-2, one bf16 step); worst {float(err.max()):.4g}; "
                           f"{n_big} elements one bf16 step off where the step exceeds 3e-2")
    exact = float(np.mean(got_bits[act] == ref_bits[act]))
    assert exact >= MIN_EXACT, (f"{what}: only {exact:.4f} of the adapter rows' elements equal the "
                                f"oracle's rounded value (at least {MIN_EXACT}); rel-L2 {rel:.3e}")
    return {"rel_l2": rel, "max_abs": float(err.max()), "n_big_step": n_big, "n": int(err.size), "exact": exact}


def shrink_bound(ids, x_bits, A_list, h_in):
    """Rigorous bound on fp32 accumulation error of v = A x: K * 2^-24 * sum |a||x|
    (the product of two bf16 values is exact in fp32).  A_list: [r][h_in] per slot."""
    absA = [np.asarray(a) & np.uint16(0x7FFF) for a in A_list]
    dummyB = [np.zeros((8, a.shape[0]), np.uint16) for a in A_list]
    ad = O.Adapters(absA, dummyB, np.ones(len(A_list)))
    s = O.shrink(ids, np.asarray(x_bits) & np.uint16(0x7FFF), ad)
    return h_in * 2.0 ** -24 * s + 1e-30
