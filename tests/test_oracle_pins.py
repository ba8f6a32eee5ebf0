"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each test names what fixes the expected value: a closed form, a library
routine on a special case, brute force, the merged-weight identity
(W + s B A) x - W x = s B (A x) from the multi-LoRA serving note ("direct
answer", "interviewer follow-ups": merging gives the same model), or an
invariant the pages state (None / -1 rows run the base model, zero rank
padding from the TGI page's "weight preprocessing" section leaves results
unchanged).  A plausible slip in the oracle -- a dropped term, a wrong sign,
a transposed operand, a wrong row index, a double rounding -- fails at least
one of these.
"""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle as O


def _bits_of(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _rand_bf16(gen, shape, std=1.0):
    t = (torch.randn(*shape, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)
    return _bits_of(t)


# ---------------------------------------------------------------- bf16 ----

def test_bf16_roundtrip_exhaustive():
    """Every finite bf16 pattern survives bf16 -> double -> bf16 unchanged."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_to_f64(bits)
    finite = np.isfinite(vals)
    back = O.f64_to_bf16(vals[finite])
    np.testing.assert_array_equal(back, bits[finite])
    # bf16 -> double agrees with the hardware view of bf16 as the top half of binary32
    ref = (bits[finite].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    np.testing.assert_array_equal(vals[finite], ref)


def test_bf16_rne_matches_library_on_binary32_values():
    """On values exactly representable in binary32 there is no double rounding,
    so one RNE step to bf16 must agree with torch's binary32 -> bf16 (RNE)."""
    g = torch.Generator().manual_seed(123)
    f = torch.cat([
        torch.randn(200000, generator=g) * 3.0,
        torch.randn(20000, generator=g) * 1e-38,       # subnormal range
        torch.randn(20000, generator=g) * 1e38,        # near overflow
        torch.tensor([3.3961e38, -3.3961e38, 3.39e38, 1e-45, -1e-45, 0.0, -0.0]),
    ]).to(torch.float32)
    ref = _bits_of(f.to(torch.bfloat16))
    got = O.f64_to_bf16(f.numpy().astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_ties_to_even_and_single_rounding():
    # 1 + 2^-8 lies half-way between 1 and 1 + 2^-7: ties go to the even 1.0.
    assert O.f64_to_bf16([1 + 2.0 ** -8])[0] == 0x3F80
    # 1 + 3*2^-8 lies half-way between 1+2^-7 (odd) and 1+2^-6 (even).
    assert O.f64_to_bf16([1 + 3 * 2.0 ** -8])[0] == 0x3F82
    # Just above a tie must round up.  Going through binary32 first would lose
    # the 2^-40 and then round the resulting tie down to 1.0 (double rounding).
    assert O.f64_to_bf16([1 + 2.0 ** -8 + 2.0 ** -40])[0] == 0x3F81
    assert O.f64_to_bf16([-(1 + 2.0 ** -8 + 2.0 ** -40)])[0] == 0xBF81
    # smallest subnormal 2^-133; half of it is a tie that goes to +0
    assert O.f64_to_bf16([2.0 ** -133])[0] == 0x0001
    assert O.f64_to_bf16([2.0 ** -134])[0] == 0x0000
    assert O.f64_to_bf16([1.5 * 2.0 ** -133])[0] == 0x0002
    # largest finite (2 - 2^-7) 2^127; the tie above it overflows to inf
    assert O.f64_to_bf16([(2 - 2.0 ** -7) * 2.0 ** 127])[0] == 0x7F7F
    assert O.f64_to_bf16([(2 - 2.0 ** -8) * 2.0 ** 127])[0] == 0x7F80
    assert O.f64_to_bf16([float("inf")])[0] == 0x7F80
    assert O.f64_to_bf16([float("-inf")])[0] == 0xFF80
    assert (O.f64_to_bf16([float("nan")])[0] & 0x7F80) == 0x7F80


def test_bf16_rne_is_nearest_on_doubles():
    """Definition of round-to-nearest on arbitrary doubles: the result is at
    least as close as both bf16 neighbours."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal(50000) * np.exp(rng.uniform(-20, 20, 50000))
    b = O.f64_to_bf16(x)
    r = O.bf16_to_f64(b)
    up = O.bf16_to_f64((b.astype(np.int32) + 1).astype(np.uint16))
    dn = O.bf16_to_f64((b.astype(np.int32) - 1).astype(np.uint16))
    err = np.abs(r - x)
    assert np.all(err <= np.abs(up - x))
    assert np.all(err <= np.abs(dn - x))
    assert np.all(err <= np.abs(x) * 2.0 ** -8)


# ------------------------------------------------------------ scaling ----

@pytest.mark.parametrize("alpha,r,rs,expect", [
    (16, 8, False, 2.0),     # the tiny workload: lora_alpha 16, rank 8
    (32, 16, False, 2.0),    # the 3B decode workload: alpha 32, rank 16
    (16, 64, False, 0.25),
    (16, 64, True, 2.0),     # rsLoRA: alpha / sqrt(r) = 16 / 8
    (16, 16, True, 4.0),
])
def test_scale_closed_form(alpha, r, rs, expect):
    assert O.scale(alpha, r, rs) == expect


def test_scale_rslora_defining_property():
    for r in (8, 32, 128):
        s = O.scale(16.0, r, True)
        assert abs(s * s * r - 256.0) < 1e-12
        assert O.scale(16.0, r, False) * r == 16.0


def test_fold_power_of_two_is_exponent_shift():
    """Scaling normal bf16 values by 2 (or 1/4) adds 1 (or -2) to the binary
    exponent field and leaves sign and mantissa bits unchanged."""
    g = torch.Generator().manual_seed(7)
    B = _rand_bf16(g, (64, 16), std=0.02)
    B = B[(B & 0x7F80) > (3 << 7)].reshape(-1, 1)  # normal, away from subnormals
    np.testing.assert_array_equal(O.fold_B(B, 2.0), B + np.uint16(1 << 7))
    np.testing.assert_array_equal(O.fold_B(B, 0.25), B - np.uint16(2 << 7))


def test_fold_generic_scale_is_single_nearest_rounding():
    g = torch.Generator().manual_seed(8)
    B = _rand_bf16(g, (128, 8), std=0.02)
    s = 16 / math.sqrt(8)
    Bp = O.bf16_to_f64(O.fold_B(B, s))
    exact = s * O.bf16_to_f64(B)
    # bf16 keeps 8 significant bits: unit roundoff u = 2^-8
    assert np.all(np.abs(Bp - exact) <= np.abs(exact) * 2.0 ** -8 * (1 + 1e-12))
    # and the rounding actually happened at bf16 precision (not a no-op)
    assert np.any(Bp != exact)


# ----------------------------------------------------- delta: helpers ----

def _tiny_problem(seed, T=11, h_in=24, w=40, ranks=(4, 8, 3), with_base=True):
    g = torch.Generator().manual_seed(seed)
    n = len(ranks)
    A = [_rand_bf16(g, (r, h_in), 0.3) for r in ranks]
    B = [_rand_bf16(g, (w, r), 0.3) for r in ranks]
    alphas = [2.0 * r for r in ranks]
    scales = [O.scale(a, r, False) for a, r in zip(alphas, ranks)]
    x = _rand_bf16(g, (T, h_in))
    lo = -1 if with_base else 0
    ids = torch.randint(lo, n, (T,), generator=g).numpy().astype(np.int32)
    return A, B, scales, x, ids


def test_merged_weight_identity():
    """(W + B'A) x - W x equals the oracle's delta B'(A x) for every row."""
    for seed in range(4):
        A, B, scales, x, ids = _tiny_problem(seed)
        ad = O.Adapters(A, B, scales)
        d = O.delta(ids, x, ad)
        xd = O.bf16_to_f64(x)
        rng = np.random.default_rng(seed)
        W = rng.standard_normal((ad.w, ad.h_in))
        for t in range(len(ids)):
            k = ids[t]
            if k < 0:
                np.testing.assert_array_equal(d[t], 0.0)
                continue
            Bp = O.bf16_to_f64(O.fold_B(B[k], scales[k]))
            merged = W + Bp @ O.bf16_to_f64(A[k])
            ref = merged @ xd[t] - W @ xd[t]
            tol = 1e-12 * (np.abs(W) @ np.abs(xd[t]) + np.abs(Bp) @ np.abs(O.bf16_to_f64(A[k])) @ np.abs(xd[t]))
            assert np.all(np.abs(d[t] - ref) <= tol), (seed, t)


def test_brute_force_triple_loop():
    """Delta W = B'A formed entry by entry in plain Python, then Delta W x."""
    A, B, scales, x, ids = _tiny_problem(11, T=5, h_in=8, w=6, ranks=(2, 3))
    ad = O.Adapters(A, B, scales)
    d = O.delta(ids, x, ad)
    xd = O.bf16_to_f64(x)
    for t in range(len(ids)):
        k = ids[t]
        if k < 0:
            assert all(v == 0.0 for v in d[t])
            continue
        Ak = O.bf16_to_f64(A[k]).tolist()
        Bk = O.bf16_to_f64(B[k]).tolist()
        r = len(Ak)
        dW = [[0.0] * 8 for _ in range(6)]
        for c in range(6):
            for i in range(8):
                acc = 0.0
                for j in range(r):
                    # fold s into B' by the definition bf16_rne(s * B)
                    bp = float(O.bf16_to_f64(O.f64_to_bf16([scales[k] * Bk[c][j]]))[0])
                    acc += bp * Ak[j][i]
                dW[c][i] = acc
        for c in range(6):
            ref = sum(dW[c][i] * float(xd[t][i]) for i in range(8))
            assert abs(d[t][c] - ref) <= 1e-12 * (1 + abs(ref))


def test_zero_padding_invariance_bit_exact():
    """Zero-padding A's rows and B's columns to a slot rank gives bit-identical
    results (the scale still uses the true rank)."""
    A, B, scales, x, ids = _tiny_problem(21)
    r_slot = 8
    Ap = [np.vstack([a, np.zeros((r_slot - a.shape[0], a.shape[1]), np.uint16)]) for a in A]
    Bpd = [np.hstack([b, np.zeros((b.shape[0], r_slot - b.shape[1]), np.uint16)]) for b in B]
    d0 = O.delta(ids, x, O.Adapters(A, B, scales))
    d1 = O.delta(ids, x, O.Adapters(Ap, Bpd, scales))
    np.testing.assert_array_equal(d0, d1)
    g = torch.Generator().manual_seed(3)
    y = _rand_bf16(g, (len(ids), 50))
    np.testing.assert_array_equal(O.apply_projection(ids, x, y, 6, O.Adapters(A, B, scales)),
                                  O.apply_projection(ids, x, y, 6, O.Adapters(Ap, Bpd, scales)))


def test_base_rows_untouched_and_slice_only():
    A, B, scales, x, ids = _tiny_problem(31)
    ids[::3] = -1
    g = torch.Generator().manual_seed(4)
    y = _rand_bf16(g, (len(ids), 64))
    out = O.apply_projection(ids, x, y, 8, O.Adapters(A, B, scales))
    base = ids < 0
    np.testing.assert_array_equal(out[base], y[base])
    np.testing.assert_array_equal(out[:, :8], y[:, :8])
    np.testing.assert_array_equal(out[:, 48:], y[:, 48:])
    assert np.any(out[~base, 8:48] != y[~base, 8:48])


def test_apply_is_one_rounding_of_y_plus_delta():
    A, B, scales, x, ids = _tiny_problem(41)
    ad = O.Adapters(A, B, scales)
    g = torch.Generator().manual_seed(5)
    y = _rand_bf16(g, (len(ids), 40))
    out = O.apply_projection(ids, x, y, 0, ad)
    d = O.delta(ids, x, ad)
    act = ids >= 0
    ref = O.f64_to_bf16(O.bf16_to_f64(y[act]) + d[act])
    np.testing.assert_array_equal(out[act], ref)


def test_expand_of_shrink_equals_apply():
    A, B, scales, x, ids = _tiny_problem(51)
    ad = O.Adapters(A, B, scales)
    v = O.shrink(ids, x, ad)
    g = torch.Generator().manual_seed(6)
    y = _rand_bf16(g, (len(ids), 40))
    np.testing.assert_array_equal(O.expand(ids, v, y, 0, ad), O.apply_projection(ids, x, y, 0, ad))


def test_single_adapter_reduces_to_matmul():
    """All rows on one adapter: delta = X A^T B'^T, a plain library matmul."""
    A, B, scales, x, _ = _tiny_problem(61, T=9, ranks=(8,))
    ids = np.zeros(9, np.int32)
    ad = O.Adapters(A, B, scales)
    d = O.delta(ids, x, ad)
    Bp = O.bf16_to_f64(O.fold_B(B[0], scales[0]))
    ref = (O.bf16_to_f64(x) @ O.bf16_to_f64(A[0]).T) @ Bp.T
    np.testing.assert_allclose(d, ref, rtol=1e-12, atol=1e-14)


def test_row_permutation_equivariance_exact():
    A, B, scales, x, ids = _tiny_problem(71, T=17)
    ad = O.Adapters(A, B, scales)
    d = O.delta(ids, x, ad)
    p = np.random.default_rng(0).permutation(len(ids))
    dp = O.delta(ids[p], x[p], ad)
    np.testing.assert_array_equal(dp, d[p])


def test_rank_index_not_swapped():
    """A delta built only from rank component j must use row j of A with
    column j of B (an index swap between them changes the answer)."""
    h_in, w, r = 4, 3, 2
    A = np.zeros((r, h_in), np.uint16)
    B = np.zeros((w, r), np.uint16)
    one = O.f64_to_bf16([1.0])[0]
    two = O.f64_to_bf16([2.0])[0]
    A[0, 1] = one          # v0 = x1
    A[1, 2] = two          # v1 = 2 x2
    B[0, 0] = one          # d0 = v0
    B[2, 1] = one          # d2 = v1
    x = O.f64_to_bf16([[3.0, 5.0, 7.0, 11.0]])
    d = O.delta(np.array([0], np.int32), x, O.Adapters([A], [B], [1.0]))
    np.testing.assert_array_equal(d, [[5.0, 0.0, 14.0]])


# ----------------------------------------------------------- metadata ----

def _meta_brute(ids, P, n_slots):
    seg_starts, seg_slot = [], []
    pos = 0
    for key, grp in itertools.groupby(ids[:P].tolist()):
        seg_starts.append(pos)
        seg_slot.append(key)
        pos += len(list(grp))
    seg_starts.append(P)
    dec = list(range(P, len(ids)))
    order = sorted(dec, key=lambda row: (ids[row] == -1, ids[row], row))
    gseg_starts, gseg_slot = [], []
    for i, row in enumerate(order):
        if i == 0 or ids[row] != ids[order[i - 1]]:
            gseg_starts.append(i)
            gseg_slot.append(int(ids[row]))
    gseg_starts.append(len(order))
    return seg_starts, seg_slot, order, gseg_starts, gseg_slot


@pytest.mark.parametrize("seed", range(12))
def test_metadata_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    n_slots = int(rng.integers(1, 9))
    T = int(rng.integers(0, 60))
    P = int(rng.integers(0, T + 1))
    ids = rng.integers(-1, n_slots, T).astype(np.int32)
    if seed % 3 == 0 and P > 0:  # long runs, as prefill segments have
        ids[:P] = np.repeat(rng.integers(-1, n_slots, 4), (P + 3) // 4)[:P]
    got = O.build_metadata(ids, P, n_slots)
    ref = _meta_brute(ids, P, n_slots)
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, np.array(b, np.int32).reshape(a.shape))


def test_metadata_tiny_workload_layout():
    """Three prefill segments of 5/17/32 rows with ids 0/2/-1, then six decode
    rows with ids [1,3,3,0,-1,2] over 4 slots."""
    ids = np.array([0] * 5 + [2] * 17 + [-1] * 32 + [1, 3, 3, 0, -1, 2], np.int32)
    seg_starts, seg_slot, perm, gs, gslot = O.build_metadata(ids, 54, 4)
    np.testing.assert_array_equal(seg_starts, [0, 5, 22, 54])
    np.testing.assert_array_equal(seg_slot, [0, 2, -1])
    np.testing.assert_array_equal(perm, [57, 54, 59, 55, 56, 58])
    np.testing.assert_array_equal(gs, [0, 1, 2, 3, 5, 6])
    np.testing.assert_array_equal(gslot, [0, 1, 2, 3, -1])


def test_metadata_rejects_out_of_range_ids():
    with pytest.raises(ValueError):
        O.build_metadata(np.array([0, 4], np.int32), 1, 4)
    with pytest.raises(ValueError):
        O.build_metadata(np.array([-2], np.int32), 0, 4)


# --------------------------------------------------------------- merge ----
# The merged weight W' = bf16(W +/- B'A) ([MLS], interviewer follow-ups).

def _small_ints_bf16(rng, shape, lo, hi):
    """Small integers: exact in bf16, and every sum below stays exact too."""
    return O.f64_to_bf16(rng.integers(lo, hi + 1, shape).astype(np.float64))


def test_merge_zero_adapter_leaves_weight_bit_identical():
    g = torch.Generator().manual_seed(21)
    W = _rand_bf16(g, (24, 40))
    A = _rand_bf16(g, (5, 40))
    Bp = np.zeros((24, 5), np.uint16)
    for sign in (1, -1):
        np.testing.assert_array_equal(O.merge(W, A, Bp, sign), W)


def test_merge_rank_one_closed_form():
    """A = a e_i^T (one row), B' = b e_j: only W[j][i] moves, by sign * a * b, one rounding."""
    g = torch.Generator().manual_seed(3)
    W = _rand_bf16(g, (16, 32))
    a, b, i, j = 0.71875, -1.40625, 9, 4   # both exact in bf16
    A = np.zeros((1, 32), np.uint16)
    A[0, i] = O.f64_to_bf16(np.array([a]))[0]
    Bp = np.zeros((16, 1), np.uint16)
    Bp[j, 0] = O.f64_to_bf16(np.array([b]))[0]
    for sign in (1, -1):
        got = O.merge(W, A, Bp, sign)
        expect = W.copy()
        expect[j, i] = O.f64_to_bf16(np.array([O.bf16_to_f64(W[j:j + 1, i])[0] + sign * a * b]))[0]
        np.testing.assert_array_equal(got, expect)


def test_merge_then_unmerge_restores_exact_weights():
    """With small integers every value and sum is exact in bf16, so unmerge
    undoes merge bit for bit (a swapped sign or operand would not)."""
    rng = np.random.default_rng(11)
    W = _small_ints_bf16(rng, (12, 20), -40, 40)
    A = _small_ints_bf16(rng, (3, 20), -3, 3)
    Bp = _small_ints_bf16(rng, (12, 3), -3, 3)
    merged = O.merge(W, A, Bp, 1)
    # spot value by hand: an integer sum
    w = O.bf16_to_f64(W)
    expect = w + O.bf16_to_f64(Bp) @ O.bf16_to_f64(A)
    np.testing.assert_array_equal(O.bf16_to_f64(merged), expect)
    np.testing.assert_array_equal(O.merge(merged, A, Bp, -1), W)


def test_merged_weight_applied_equals_base_plus_delta():
    """W' x = W x + B'(A x) up to W's one rounding: the merge checked against
    the oracle's separate delta path (shrink then expand, per row)."""
    for seed in range(3):
        A, B, scales, x, ids = _tiny_problem(seed, ranks=(4, 8))
        ad = O.Adapters(A, B, scales)
        d = O.delta(ids, x, ad)
        g = torch.Generator().manual_seed(100 + seed)
        W = _rand_bf16(g, (ad.w, ad.h_in))
        xd = O.bf16_to_f64(x)
        for k in range(len(A)):
            Bp = O.fold_B(B[k], scales[k])
            merged = O.bf16_to_f64(O.merge(W, A[k], Bp, 1))
            # one bf16 rounding per weight: |error| <= 2^-9 |w'| per element
            for t in np.nonzero(ids == k)[0]:
                lhs = merged @ xd[t]
                rhs = O.bf16_to_f64(W) @ xd[t] + d[t]
                bound = 2.0 ** -8 * (np.abs(merged) @ np.abs(xd[t])) + 1e-12
                assert np.all(np.abs(lhs - rhs) <= bound), (seed, k, t)


# ------------------------------------------------------ linear layer ----

def test_linear_small_integers_equal_exact_integer_product():
    """With small integers and scale 1 every product and sum is exact, so the
    layer's output must equal x (W + B A)^T computed in integers for adapter
    rows and x W^T for base rows (a dropped delta, a wrong slot, a transposed
    operand or a sign slip would not)."""
    rng = np.random.default_rng(17)
    T, h_in, w, ranks = 11, 12, 9, (2, 3, 1)
    x = rng.integers(-1, 2, (T, h_in))
    W = rng.integers(-3, 4, (w, h_in))
    A = [rng.integers(-2, 3, (r, h_in)) for r in ranks]
    B = [rng.integers(-2, 3, (w, r)) for r in ranks]
    ids = np.array([0, -1, 1, 2, 2, 0, -1, 1, 0, 2, 1], np.int32)
    to_bits = lambda a: O.f64_to_bf16(a.astype(np.float64))
    ad = O.Adapters([to_bits(a) for a in A], [to_bits(b) for b in B],
                    [O.scale(float(r), r, False) for r in ranks])            # alpha = r: s = 1
    y_in = np.full((T, w + 5), 0x7FC0, np.uint16)                             # NaN: must not be read
    got = O.linear_projection(ids, to_bits(x), to_bits(W), y_in, 3, ad)
    expect = np.empty((T, w), np.int64)
    for t in range(T):
        Wt = W + (B[ids[t]] @ A[ids[t]] if ids[t] >= 0 else 0)
        expect[t] = Wt @ x[t]
    assert np.abs(expect).max() < 256                                         # exact in bf16
    np.testing.assert_array_equal(O.bf16_to_f64(got[:, 3:3 + w]), expect.astype(np.float64))
    np.testing.assert_array_equal(got[:, :3], y_in[:, :3])                    # outside the slice untouched
    np.testing.assert_array_equal(got[:, 3 + w:], y_in[:, 3 + w:])


def test_linear_rounds_once():
    """base = 1 + 2^-8 sits exactly halfway between two bf16 values; a delta
    of 2^-10 tips the single rounding up to 1 + 2^-7, where rounding the base
    first (ties to even: 1) and then adding the delta would give 1.  A base
    row keeps the tie and rounds to even."""
    one, eps8, eps10 = 1.0, 2.0 ** -8, 2.0 ** -10
    x = O.f64_to_bf16(np.array([[one, one], [one, one]]))
    W = O.f64_to_bf16(np.array([[one, eps8]]))
    A = [O.f64_to_bf16(np.array([[1.0, 0.0]]))]
    B = [O.f64_to_bf16(np.array([[eps10]]))]
    ad = O.Adapters(A, B, [O.scale(1.0, 1, False)])
    got = O.bf16_to_f64(O.linear_projection(np.array([0, -1], np.int32), x, W, np.zeros((2, 1), np.uint16), 0, ad))
    assert got[0, 0] == 1.0 + 2.0 ** -7
    assert got[1, 0] == 1.0


def test_linear_base_rows_equal_rounded_plain_product():
    """Rows with id -1 are bf16_rne of the plain product, checked against an
    independent fp64 matrix product."""
    g = torch.Generator().manual_seed(8)
    T, h_in, w = 6, 40, 24
    x, W = _rand_bf16(g, (T, h_in)), _rand_bf16(g, (w, h_in), 0.2)
    A, B = [_rand_bf16(g, (4, h_in))], [_rand_bf16(g, (w, 4))]
    ids = np.array([-1, 0, -1, -1, 0, -1], np.int32)
    ad = O.Adapters(A, B, [O.scale(8.0, 4, False)])
    got = O.linear_projection(ids, x, W, np.zeros((T, w), np.uint16), 0, ad)
    plain = O.f64_to_bf16(O.bf16_to_f64(x) @ O.bf16_to_f64(W).T)
    base = ids < 0
    np.testing.assert_array_equal(got[base], plain[base])
    assert (got[~base] != plain[~base]).any()                                 # adapter rows differ
