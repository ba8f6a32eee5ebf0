"""CPU tests of the C library's host side: exports, store preparation,
metadata builder, slot rank and argument validation (no kernel launches)."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle as O
from lora_serving_gb300 import abi, build, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    return abi.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "lora.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lora_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(_lib):
    declared = _declared_functions()
    assert set(declared) == set(abi.EXPORTS)
    for name in declared:
        assert hasattr(_lib, name), name


def test_status_strings(_lib):
    for code, name in abi.STATUS.items():
        assert abi.lora_status_string(code).startswith(name)


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("r,r_slot,alpha,rs", [(8, 8, 16, False), (16, 16, 32, False),
                                               (8, 64, 16, True), (32, 64, 16, True),
                                               (64, 64, 16, False), (5, 16, 7.0, False)])
def test_prepare_adapter_bit_exact_vs_oracle(r, r_slot, alpha, rs):
    g = torch.Generator().manual_seed(r * 100 + r_slot)
    h_in, out = 48, 40
    A = _bits((torch.randn(r, h_in, generator=g) * 0.02).to(torch.bfloat16))
    B = _bits((torch.randn(out, r, generator=g) * 0.02).to(torch.bfloat16))
    A_s, B_s = abi.lora_prepare_adapter(A, B, alpha, rs, r_slot)
    np.testing.assert_array_equal(A_s[:r], A)
    np.testing.assert_array_equal(A_s[r:], 0)
    np.testing.assert_array_equal(B_s[:, :r], O.fold_B(B, O.scale(alpha, r, rs)))
    np.testing.assert_array_equal(B_s[:, r:], 0)


def test_prepare_adapter_rounding_edge_cases():
    """Values whose scaled product sits on or next to a bf16 rounding tie, and
    subnormal/overflow products, fold exactly as the oracle's rounding."""
    vals = O.f64_to_bf16(np.array([1.0, 1 + 2 ** -7, -3.0, 1e-38, 3e38, 2 ** -126, 0.0, -0.0]))
    B = np.tile(vals, (3, 1)).T.copy()  # [8][3]
    A = np.zeros((3, 8), np.uint16)
    for alpha, rs in [(1.5, False), (3 * 1.0000001, True), (2.0 ** -10, False), (1e5, False)]:
        _, B_s = abi.lora_prepare_adapter(A, B, alpha, rs, 8)
        np.testing.assert_array_equal(B_s[:, :3], O.fold_B(B, O.scale(alpha, 3, rs)))


def test_prepare_adapter_rejects():
    A = np.zeros((16, 8), np.uint16)
    B = np.zeros((8, 16), np.uint16)
    with pytest.raises(abi.LoraError) as e:
        abi.lora_prepare_adapter(A, B, 32, False, 8)   # rank 16 > slot rank 8
    assert e.value.name == "LORA_ERR_RANK_EXCEEDS_SLOT"
    with pytest.raises(abi.LoraError) as e:
        abi.lora_prepare_adapter(A, B, 32, False, 20)  # slot rank not a multiple of 8
    assert e.value.name == "LORA_ERR_ALIGNMENT"


@pytest.mark.parametrize("seed", range(20))
def test_metadata_bit_exact_vs_oracle(seed):
    rng = np.random.default_rng(1000 + seed)
    n_slots = int(rng.integers(1, 12))
    T = int(rng.integers(0, 300))
    P = int(rng.integers(0, T + 1))
    ids = rng.integers(-1, n_slots, T).astype(np.int32)
    if seed % 2 and P:
        ids[:P] = np.repeat(rng.integers(-1, n_slots, 6), (P + 5) // 6)[:P]
    m = abi.lora_build_metadata(ids, P, n_slots)
    ref = O.build_metadata(ids, P, n_slots)
    for key, r in zip(("seg_starts", "seg_slot", "perm", "gseg_starts", "gseg_slot"), ref):
        np.testing.assert_array_equal(m[key], r, err_msg=key)
    lens = np.diff(ref[0])
    assert m["max_seg_len"] == (lens.max() if lens.size else 0)
    glens = np.diff(ref[3])
    assert m["max_gseg_len"] == (glens.max() if glens.size else 0)


@pytest.mark.parametrize("name", ["tiny", "llama3b_decode", "mistral7b_prefill", "mixed", "stress70b"])
def test_metadata_workloads_bit_exact(name):
    wl = synth.get(name)
    m = abi.lora_build_metadata(wl.ids, wl.n_prefill, wl.n_slots)
    ref = O.build_metadata(wl.ids, wl.n_prefill, wl.n_slots)
    for key, r in zip(("seg_starts", "seg_slot", "perm", "gseg_starts", "gseg_slot"), ref):
        np.testing.assert_array_equal(m[key], r, err_msg=key)


def test_metadata_rejects_bad_ids():
    with pytest.raises(abi.LoraError) as e:
        abi.lora_build_metadata(np.array([0, 5], np.int32), 1, 4)
    assert e.value.name == "LORA_ERR_SLOT_RANGE"


def _golden(name):
    rows = []
    for line in open(os.path.join(ROOT, "tests", "golden", name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line)
    return rows


def test_golden_slot_rank():
    """vLLM page, step 2: adapters of rank 16/32/64 -> max_lora_rank 64."""
    for row in _golden("slot_rank.txt"):
        lhs, rhs = row.split("->")
        assert abi.lora_slot_rank([int(v) for v in lhs.split()]) == int(rhs)
    assert abi.lora_slot_rank([5, 3]) == 8      # rounded up to the 8-wide vector
    assert abi.lora_slot_rank([]) == 0


def test_golden_param_count_closed_form():
    """Interview note: d*k -> r*(d+k) parameters per matrix, about 100x fewer.
    The store slot of one projection holds exactly r_slot*(h_in + out) values."""
    from lora_serving_gb300.store import GroupStore
    for row in _golden("param_count.txt"):
        d, k, r = (int(v) for v in row.split())
        st = GroupStore.__new__(GroupStore)
        st.h_in, st.r_slot, st.projs = k, r, [("p", d)]
        assert st.nbytes_slot() == 2 * r * (d + k)
        ratio = (d * k) / (r * (d + k))
        assert 30 <= ratio <= 300


def _null_stream():
    return 0


def test_kernel_entry_points_validate_before_launch():
    """Host-detectable errors come back before anything is enqueued, so these
    calls are safe without a GPU."""
    lib = abi.load()
    buf = (ctypes.c_uint8 * 4096)()
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    ids = base
    # NULL x
    assert lib.lora_bgmv_shrink(base, 16, 0, 64, base, ids, 4, 64, 16, 2, 0, 0) == 1
    # h_in not a multiple of 8
    assert lib.lora_bgmv_shrink(base, 16, base, 64, base, ids, 4, 60, 16, 2, 0, 0) == 5
    # r_slot beyond the fused limit
    assert lib.lora_bgmv_shrink(base, 1024, base, 64, base, ids, 4, 64, 1024, 2, 0, 0) == 3
    # misaligned y pointer
    assert lib.lora_bgmv_expand(base + 2, 64, 0, 64, base, 16, base, ids, 4, 16, 2, 0, 0) == 5
    # slice past the row
    assert lib.lora_bgmv_expand(base, 64, 32, 64, base, 16, base, ids, 4, 16, 2, 0, 0) == 2
    # r_slot above the per-slot maximum
    assert lib.lora_bgmv_expand(base, 64, 0, 64, base, 256, base, ids, 4, 256, 2, 0, 0) == 3
    # empty batches are a no-op
    assert lib.lora_bgmv_shrink(base, 16, base, 64, base, ids, 0, 64, 16, 2, 0, 0) == 0
    # SGMV with positions but no segments
    assert lib.lora_sgmv_shrink(base, 16, base, 64, base, 0, 0, 0, 0, 4, 4, 0, 64, 16, 2, 0, 0) == 6
    # lora_apply: no workspace
    projs = abi.make_projs([(base, base, 0, 64)])
    meta = abi.lora_meta_t()
    meta.lora_ids, meta.n_rows, meta.n_prefill = ids, 4, 0
    meta.perm, meta.gseg_starts, meta.gseg_slot, meta.n_gsegs = base, base, base, 1
    st = lib.lora_apply(base, 64, base, 64, 64, ctypes.addressof(projs), 1, 16, 2,
                        ctypes.addressof(meta), 0, 0, 0, 0, 0)
    assert st == 7
    # lora_apply: too many projections
    st = lib.lora_apply(base, 64, base, 64, 64, ctypes.addressof(projs), 5, 16, 2,
                        ctypes.addressof(meta), base, 1 << 20, 0, 0, 0)
    assert st == 1
    # lora_apply: projection slices that overlap in y
    both = abi.make_projs([(base, base, 0, 64), (base, base, 56, 64)])
    st = lib.lora_apply(base, 128, base, 64, 64, ctypes.addressof(both), 2, 16, 2,
                        ctypes.addressof(meta), base, 1 << 20, 0, 0, 0)
    assert st == 2
    # a slice whose end overflows int is past the row, not wrapped around
    assert lib.lora_bgmv_expand(base, 64, 2**31 - 8, 64, base, 16, base, ids, 4, 16, 2, 0, 0) == 2
    # bf16 hi/lo planes (rank padded to 64) + fp32 v + the expand's work-item
    # counter, each region rounded to 256 B
    planes = (2 * 10 * 3 * 64 * 2 + 255) // 256 * 256
    fp32 = (10 * 3 * 16 * 4 + 255) // 256 * 256
    assert lib.lora_apply_workspace_bytes(10, 3, 16) == planes + fp32 + 256


def test_linear_and_merge_batch_validate_before_launch():
    """lora_linear and lora_merge_batch reject host-detectable errors before
    any CUDA call, so these run without a GPU."""
    lib = abi.load()
    buf = (ctypes.c_uint8 * 8192)()
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    meta = abi.lora_meta_t()
    meta.lora_ids, meta.n_rows, meta.n_prefill = base, 4, 4
    meta.seg_starts, meta.seg_slot, meta.n_segs = base, base, 1
    tiles = abi.make_projs([(base, base, 0, 64), (base, base, 64, 64)])
    gap = abi.make_projs([(base, base, 0, 64), (base, base, 72, 56)])   # column 64..71 uncovered
    P = ctypes.addressof
    # projections that do not tile [0, n_out)
    assert lib.lora_linear(base, 128, base, 64, 64, base, 64, P(gap), 2, 16, 2, P(meta), base, 1 << 20, 0, 0) == 2
    # ld_w below h_in
    assert lib.lora_linear(base, 128, base, 64, 64, base, 32, P(tiles), 2, 16, 2, P(meta), base, 1 << 20, 0, 0) == 2
    # misaligned W
    assert lib.lora_linear(base, 128, base, 64, 64, base + 2, 64, P(tiles), 2, 16, 2, P(meta), base, 1 << 20,
                           0, 0) == 5
    # slot rank above 64 with decode rows
    meta.n_prefill = 2
    assert lib.lora_linear(base, 128, base, 64, 64, base, 64, P(tiles), 2, 128, 2, P(meta), base, 1 << 20,
                           0, 0) == 3
    meta.n_prefill = 4
    # no workspace
    assert lib.lora_linear(base, 128, base, 64, 64, base, 64, P(tiles), 2, 16, 2, P(meta), 0, 0, 0, 0) == 7
    # NULL W
    assert lib.lora_linear(base, 128, base, 64, 64, 0, 64, P(tiles), 2, 16, 2, P(meta), base, 1 << 20, 0, 0) == 1

    Ws = (ctypes.c_void_p * 2)(base, base + 2)
    As = (ctypes.c_void_p * 2)(base, base)
    Bs = (ctypes.c_void_p * 2)(base, base)
    ld = (ctypes.c_int * 2)(64, 64)
    out = (ctypes.c_int * 2)(32, 32)
    h_in = (ctypes.c_int * 2)(64, 64)
    # the second weight misaligned
    assert lib.lora_merge_batch(2, Ws, ld, out, h_in, As, Bs, 16, 1, 0) == 5
    # bad sign, NULL arrays, slot rank above the maximum
    assert lib.lora_merge_batch(1, Ws, ld, out, h_in, As, Bs, 16, 0, 0) == 1
    assert lib.lora_merge_batch(1, None, ld, out, h_in, As, Bs, 16, 1, 0) == 1
    assert lib.lora_merge_batch(1, Ws, ld, out, h_in, As, Bs, 136, 1, 0) == 3
    # nothing to do
    assert lib.lora_merge_batch(0, None, None, None, None, None, None, 16, 1, 0) == 0


def test_binding_refuses_host_tensors_for_kernel_arguments():
    """A host pointer handed to a kernel would be an illegal device address:
    the binding refuses host tensors before calling into the library."""
    import torch
    v = torch.zeros(4, 16)
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    A = torch.zeros(2, 16, 64, dtype=torch.bfloat16)
    ids = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        abi.lora_bgmv_shrink(v, x, A, ids, h_in=64, r_slot=16, n_slots=2, stream=0)
    W = torch.zeros(64, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        abi.lora_merge(W, A[0], torch.zeros(64, 16, dtype=torch.bfloat16), 1, stream=0)


def test_noalloc_rejects_before_any_cuda_call():
    """lora_apply_noalloc refuses a batch too large for its built-in scratch,
    and bad counts, before it looks up the scratch on a device."""
    lib = abi.load()
    buf = (ctypes.c_uint8 * 4096)()
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    projs = abi.make_projs([(base, base, 0, 64)])
    meta = abi.lora_meta_t()
    rows = abi.LORA_NOALLOC_SCRATCH_BYTES // (64 * 4) + 1   # fp32 v alone exceeds the scratch
    meta.lora_ids, meta.n_rows, meta.n_prefill = base, rows, 0
    P = ctypes.addressof
    assert lib.lora_apply_noalloc(base, 64, base, 64, 64, P(projs), 1, 64, 2, P(meta), 0, 0, 0) == 7
    assert lib.lora_apply_noalloc(base, 64, base, 64, 64, P(projs), 0, 64, 2, P(meta), 0, 0, 0) == 1
    meta.n_rows = -1
    assert lib.lora_apply_noalloc(base, 64, base, 64, 64, P(projs), 1, 64, 2, P(meta), 0, 0, 0) == 1
    # a bad rank is reported as lora_apply reports it, not as a scratch-size
    # failure (and the size arithmetic never sees a huge rank)
    meta.n_rows = rows
    assert lib.lora_apply_noalloc(base, 64, base, 64, 64, P(projs), 1, 2**31 - 1, 2, P(meta), 0, 0, 0) == 3
    assert lib.lora_apply_noalloc(base, 64, base, 64, 64, P(projs), 1, 12, 2, P(meta), 0, 0, 0) == 5
    assert lib.lora_apply_noalloc(base, 64, base, 64, 64, P(projs), 1, 64, 0, P(meta), 0, 0, 0) == 1
    assert lib.lora_apply_workspace_bytes(rows, 1, 2**31 - 1) == 0
    assert lib.lora_apply_workspace_bytes(rows, 5, 64) == 0
