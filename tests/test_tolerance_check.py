"""The parity check itself (tests/helpers.check_bf16), on the CPU: what it
accepts and what it rejects, with mistakes planted in the oracle's output.

Setting: one projection (4096 -> 1024), 4 adapters of rank 16, alpha 32,
weights N(0, 0.02^2) and x N(0, 1) in bf16, as in the Llama-3.2-3B-shaped
decode workload; y_in N(0, 1) (accumulate mode) or 0 (delta mode).
"""
import numpy as np
import pytest

import oracle as O
from helpers import MAX_ABS, REL_L2, bf16_step, check_bf16

T, H_IN, W, R, N_AD = 512, 4096, 1024, 16, 4


def _bf16(a):
    return O.f64_to_bf16(np.asarray(a, np.float64))


@pytest.fixture(scope="module")
def problem():
    rng = np.random.default_rng(7)
    A = [_bf16(rng.standard_normal((R, H_IN)) * 0.02) for _ in range(N_AD)]
    B = [_bf16(rng.standard_normal((W, R)) * 0.02) for _ in range(N_AD)]
    ad = O.Adapters(A, B, [O.scale(2.0 * R, R, False)] * N_AD)
    x = _bf16(rng.standard_normal((T, H_IN)))
    ids = rng.integers(-1, N_AD, T).astype(np.int32)
    y_in = _bf16(rng.standard_normal((T, W)))
    return ad, x, ids, y_in, rng


def _stated_bar(got, ref, act):
    g, r = O.bf16_to_f64(got[act]), O.bf16_to_f64(ref[act])
    err = np.abs(g - r)
    rel = np.sqrt((err ** 2).sum() / (r ** 2).sum())
    within = (err <= MAX_ABS) | (err <= bf16_step(r) * (1 + 1e-9))
    return rel <= REL_L2 and bool(within.all())


def test_fp32_delta_rounded_once_is_accepted(problem):
    """A delta formed in fp32 (v = A x, then B' v, as the kernels do) and
    rounded once with y_in passes, bit-identity fraction included."""
    ad, x, ids, y_in, _ = problem
    ref = O.apply_projection(ids, x, y_in, 0, ad)
    xf = O.bf16_to_f64(x).astype(np.float32)
    d = np.zeros((T, W), np.float32)
    for k in range(N_AD):
        m = ids == k
        Ak = O.bf16_to_f64(ad.A_cat[ad.A_off[k]:ad.A_off[k] + R * H_IN].reshape(R, H_IN)).astype(np.float32)
        Bp = O.bf16_to_f64(O.fold_B(ad.B_cat[ad.B_off[k]:ad.B_off[k] + W * R].reshape(W, R),
                                    ad.scale[k])).astype(np.float32)
        d[m] = (xf[m] @ Ak.T) @ Bp.T
    got = np.where((ids >= 0)[:, None], _bf16(O.bf16_to_f64(y_in) + d.astype(np.float64)), y_in)
    res = check_bf16(got, ref, ids, y_in, "fp32 delta")
    assert res["exact"] > 0.999


def test_small_delta_error_in_accumulate_mode_is_rejected(problem):
    """The oracle's delta made 0.1 % too large (planted on the CPU): it meets
    the stated rel-L2 and max-abs bar in accumulate mode, and the
    bit-identity fraction rejects it."""
    ad, x, ids, y_in, _ = problem
    ref = O.apply_projection(ids, x, y_in, 0, ad)
    d = O.delta(ids, x, ad)
    act = ids >= 0
    planted = np.where(act[:, None], _bf16(O.bf16_to_f64(y_in) + d * 1.001), y_in)
    assert _stated_bar(planted, ref, act)
    with pytest.raises(AssertionError, match="equal the oracle's rounded value"):
        check_bf16(planted, ref, ids, y_in, "planted")


def test_changed_base_row_is_rejected(problem):
    """A base-only row (id -1) must keep y_in bit for bit."""
    ad, x, ids, y_in, _ = problem
    ref = O.apply_projection(ids, x, y_in, 0, ad)
    got = ref.copy()
    t = int(np.flatnonzero(ids < 0)[0])
    got[t, 3] ^= np.uint16(1)
    with pytest.raises(AssertionError, match="base-only rows changed"):
        check_bf16(got, ref, ids, y_in, "base row")
