"""GPU parity: every C-ABI kernel entry point against the fp64 oracle on the
same seeded inputs (tolerances in helpers.py), on all five workloads, plus
the edge cases the method has (empty batch, all-base batch, prefill-only,
decode-only, ranks above the BGMV cap, malformed ids and segments)."""
import os

import numpy as np
import pytest
import torch

import oracle as O
from helpers import (check_bf16, oracle_adapters, oracle_group, oracle_group_all_rows, shrink_bound, to_dev,
                     to_host)
from lora_serving_gb300 import abi, build, store, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    abi.load()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"


def _status():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _seeded_v(T, cols, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(T, cols, generator=g, dtype=torch.float32)


_CACHE = {}


def _wl(name, mode="delta", **kw):
    key = (name, mode, tuple(sorted(kw.items())))
    if key not in _CACHE:
        _CACHE.clear()
        _CACHE[key] = synth.get(name, **kw).materialise(mode)
    return _CACHE[key]


# ------------------------------------------------- standalone kernels ----

@pytest.mark.parametrize("name,group", [("tiny", "proj"), ("llama3b_decode", "qkv"), ("llama3b_decode", "o")])
def test_bgmv_shrink_vs_oracle(name, group):
    wl = _wl(name)
    st = store.GroupStore.from_workload(wl, group)
    g = next(g for g in wl.groups if g.name == group)
    x = to_dev(wl.x[group])
    ids = torch.from_numpy(wl.ids).cuda()
    for p, (pname, _) in enumerate(g.projs):
        v = torch.full((wl.n_rows, wl.r_slot), -7.0, device="cuda")
        s = _status()
        abi.lora_bgmv_shrink(v, x, st.A[p], ids, h_in=g.h_in, r_slot=wl.r_slot, n_slots=wl.n_slots, dev_status=s)
        torch.cuda.synchronize()
        assert abi.lora_read_device_status(s) == 0
        got = v.cpu().numpy().astype(np.float64)
        ad = oracle_adapters(wl, group, pname)
        ref = O.shrink(wl.ids, wl.x[group], ad, v_cols=wl.r_slot)
        bound = shrink_bound(wl.ids, wl.x[group], [wl.A[(group, pname, k)] for k in range(wl.n_slots)], g.h_in)
        act = wl.ids >= 0
        r = int(wl.ranks.max())
        assert np.all(np.abs(got[act, :r] - ref[act, :r]) <= bound[act, :r])
        assert np.all(got[~act] == -7.0), "base rows must not be written"


def test_bgmv_shrink_stacked_qkv():
    """q/k/v A stores stacked along rank give the three shrinks side by side."""
    wl = _wl("llama3b_decode")
    st = store.GroupStore.from_workload(wl, "qkv")
    A_stack = torch.cat(st.A, dim=1).contiguous()  # [n][3*r][h]
    x = to_dev(wl.x["qkv"])
    ids = torch.from_numpy(wl.ids).cuda()
    v = torch.zeros(wl.n_rows, 3 * wl.r_slot, device="cuda")
    abi.lora_bgmv_shrink(v, x, A_stack, ids, h_in=3072, r_slot=3 * wl.r_slot, n_slots=wl.n_slots)
    for p in range(3):
        v1 = torch.zeros(wl.n_rows, wl.r_slot, device="cuda")
        abi.lora_bgmv_shrink(v1, x, st.A[p], ids, h_in=3072, r_slot=wl.r_slot, n_slots=wl.n_slots)
        torch.testing.assert_close(v[:, p * wl.r_slot:(p + 1) * wl.r_slot], v1, rtol=0, atol=0)


@pytest.mark.parametrize("mode", ["delta", "accumulate"])
@pytest.mark.parametrize("name,group", [("tiny", "proj"), ("llama3b_decode", "qkv"), ("llama3b_decode", "o")])
def test_bgmv_expand_vs_oracle(name, group, mode):
    wl = _wl(name, mode)
    st = store.GroupStore.from_workload(wl, group)
    g = next(g for g in wl.groups if g.name == group)
    ids = torch.from_numpy(wl.ids).cuda()
    vcpu = _seeded_v(wl.n_rows, wl.r_slot, 99)
    v = vcpu.cuda()
    y = to_dev(wl.y[group])
    for p, ((pname, w), off) in enumerate(zip(g.projs, g.offsets)):
        abi.lora_bgmv_expand(y, off, w, v, st.B[p], ids, r_slot=wl.r_slot, n_slots=wl.n_slots)
    torch.cuda.synchronize()
    ref = wl.y[group].copy()
    for (pname, w), off in zip(g.projs, g.offsets):
        ref = O.expand(wl.ids, vcpu.numpy().astype(np.float64), ref, off, oracle_adapters(wl, group, pname))
    check_bf16(to_host(y), ref, wl.ids, wl.y[group], f"bgmv_expand {name}/{group}/{mode}")


@pytest.mark.parametrize("gather", [False, True])
def test_sgmv_shrink_expand_vs_oracle(gather):
    """Contiguous prefill segments of the tiny workload, or all its rows in
    the gather form (rows sorted by adapter through a permutation)."""
    wl = _wl("tiny", "accumulate")
    st = store.GroupStore.from_workload(wl, "proj")
    x = to_dev(wl.x["proj"])
    y = to_dev(wl.y["proj"])
    if gather:
        m = abi.lora_build_metadata(wl.ids, 0, wl.n_slots)
        starts, slots, perm, n_pos = m["gseg_starts"], m["gseg_slot"], m["perm"], wl.n_rows
        ng = m["n_gsegs"]
    else:
        m = abi.lora_build_metadata(wl.ids, wl.n_prefill, wl.n_slots)
        starts, slots, perm, n_pos = m["seg_starts"], m["seg_slot"], None, wl.n_prefill
        ng = m["n_segs"]
    d_starts = torch.from_numpy(starts).cuda()
    d_slots = torch.from_numpy(slots).cuda()
    d_perm = torch.from_numpy(perm).cuda() if perm is not None else None
    v = torch.zeros(wl.n_rows, wl.r_slot, device="cuda")
    s = _status()
    abi.lora_sgmv_shrink(v, x, st.A[0], d_starts, d_slots, ng, d_perm, n_pos, h_in=256,
                         r_slot=wl.r_slot, n_slots=wl.n_slots, dev_status=s)
    abi.lora_sgmv_expand(y, 0, 256, v, st.B[0], d_starts, d_slots, ng, d_perm, n_pos,
                         r_slot=wl.r_slot, n_slots=wl.n_slots, dev_status=s)
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(s) == 0
    covered = np.zeros(wl.n_rows, bool)
    covered[(perm if perm is not None else np.arange(n_pos))] = True
    ids_eff = np.where(covered, wl.ids, -1).astype(np.int32)
    ref = oracle_group(wl, "proj")
    ref[~covered] = wl.y["proj"][~covered]
    check_bf16(to_host(y), ref, ids_eff, wl.y["proj"], f"sgmv gather={gather}")


# ---------------------------------------------------------- lora_apply ----

def _run_apply(wl, group, meta=None, stat=None):
    g = next(g for g in wl.groups if g.name == group)
    st = store.GroupStore.from_workload(wl, group)
    meta = meta or store.BatchMeta(wl.ids, wl.n_prefill, wl.n_slots)
    ws = store.workspace_for(wl.n_rows, len(g.projs), wl.r_slot)
    x = to_dev(wl.x[group])
    y = to_dev(wl.y[group])
    s = stat if stat is not None else _status()
    store.apply(y, x, st, meta, ws, dev_status=s)
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(s) == 0
    return to_host(y)


@pytest.mark.parametrize("mode", ["delta", "accumulate"])
@pytest.mark.parametrize("name", ["tiny", "llama3b_decode", "mixed"])
def test_apply_full_workload(name, mode):
    wl = _wl(name, mode)
    for g in wl.groups:
        got = _run_apply(wl, g.name)
        ref = oracle_group(wl, g.name)
        check_bf16(got, ref, wl.ids, wl.y[g.name], f"{name}/{g.name}/{mode}")


@pytest.mark.parametrize("mode", ["delta", "accumulate"])
@pytest.mark.parametrize("name", ["mistral7b_prefill", "stress70b"])
def test_apply_full_size_all_rows(name, mode):
    """Full sizes, all groups, in the launch configuration the benchmark
    uses (the tensor-core SGMV kernels for the prefill batch, the two-launch
    grouped kernels for the stress batch): every element of every row is
    compared with the oracle, which runs over row blocks on all host cores."""
    wl = _wl(name, mode)
    for g in wl.groups:
        got = _run_apply(wl, g.name)
        ref = oracle_group_all_rows(wl, g.name)
        r = check_bf16(got, ref, wl.ids, wl.y[g.name], f"{name}/{g.name}/{mode}")
        assert r["n"] == int((wl.ids >= 0).sum()) * g.ld_y
        print(f"{name}/{g.name}/{mode}: {r['n']} elements, rel-L2 {r['rel_l2']:.2e}, max-abs "
              f"{r['max_abs']:.3g}, one bf16 step off where the step exceeds 3e-2: {r['n_big_step']}")


# ---------------------------------------------------------- edge cases ----

def _small(ids, n_prefill, n_slots=4, rank=8, h_in=64, widths=(64, 16, 16), seed=0, mode="accumulate",
           r_slot=None):
    ids = np.asarray(ids, np.int32)
    r_slot = r_slot or ((rank + 7) // 8 * 8)
    wl = synth.Workload("edge", seed, [synth.Group("g", h_in, [(f"p{i}", w) for i, w in enumerate(widths)])],
                        np.full(n_slots, rank), np.full(n_slots, 2.0 * rank), np.zeros(n_slots, bool),
                        r_slot, ids, n_prefill)
    return wl.materialise(mode)


def test_apply_empty_batch_is_noop():
    wl = _small(np.zeros(0, np.int32), 0)
    st = store.GroupStore.from_workload(wl, "g")
    meta = store.BatchMeta(wl.ids, 0, wl.n_slots)
    y = torch.zeros(1, 96, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(1, 64, dtype=torch.bfloat16, device="cuda")
    store.apply(y, x, st, meta, store.workspace_for(1, 3, 8))
    torch.cuda.synchronize()


def test_apply_all_base_rows_bit_identical():
    wl = _small([-1] * 7 + [-1] * 5, 7)
    got = _run_apply(wl, "g")
    np.testing.assert_array_equal(got, wl.y["g"])


@pytest.mark.parametrize("n_prefill", [0, 40])
def test_apply_decode_only_and_prefill_only(n_prefill):
    rng = np.random.default_rng(n_prefill)
    ids = rng.integers(-1, 4, 40).astype(np.int32)
    wl = _small(ids, n_prefill)
    got = _run_apply(wl, "g")
    check_bf16(got, oracle_group(wl, "g"), wl.ids, wl.y["g"], f"P={n_prefill}")


@pytest.mark.parametrize("rank", [40, 64, 128])
def test_apply_rank_above_bgmv_cap_uses_gather(rank):
    """Decode rows with r_slot > 32 take the SGMV gather route; up to the
    largest slot rank the kernels accept."""
    rng = np.random.default_rng(rank)
    ids = np.concatenate([np.repeat([2, 0, -1, 1], [9, 1, 3, 17]), rng.integers(-1, 4, 33)]).astype(np.int32)
    wl = _small(ids, 30, rank=rank, h_in=128, widths=(128, 24, 24))
    got = _run_apply(wl, "g")
    check_bf16(got, oracle_group(wl, "g"), wl.ids, wl.y["g"], f"rank={rank}")


def test_zero_padding_bit_identical_on_gpu():
    """The same adapters stored at slot rank 8 and 24 give identical bits."""
    rng = np.random.default_rng(3)
    ids = np.concatenate([np.repeat([1, 3], [12, 5]), rng.integers(-1, 4, 9)]).astype(np.int32)
    a = _small(ids, 17, rank=5, r_slot=8)
    b = _small(ids, 17, rank=5, r_slot=24)
    np.testing.assert_array_equal(_run_apply(a, "g"), _run_apply(b, "g"))


def test_bgmv_row_permutation_bit_exact():
    wl = _wl("llama3b_decode", "accumulate")
    p = np.random.default_rng(1).permutation(wl.n_rows)
    base = _run_apply(wl, "qkv")
    wl2 = synth.Workload(wl.name, wl.seed, wl.groups, wl.ranks, wl.alphas, wl.rslora, wl.r_slot,
                         wl.ids[p].copy(), 0)
    wl2.A, wl2.B = wl.A, wl.B
    wl2.x = {"qkv": wl.x["qkv"][p].copy()}
    wl2.y = {"qkv": wl.y["qkv"][p].copy()}
    np.testing.assert_array_equal(_run_apply(wl2, "qkv"), base[p])


def test_bad_slot_in_gather_groups_flagged_and_rows_skipped():
    """lora_apply's decode route reads the gather groups: a group naming a
    slot >= n_slots is flagged and its rows are left alone."""
    ids = np.array([0, 1, 2, 3, 1, 0], np.int32)
    wl = _small(ids, 0)
    st = store.GroupStore.from_workload(wl, "g")
    meta = store.BatchMeta(ids, 0, wl.n_slots)
    meta.gseg_slot.copy_(torch.tensor([0, 1, 9, 3], dtype=torch.int32))  # slot 2's group corrupted
    ws = store.workspace_for(6, 3, 8)
    y = to_dev(wl.y["g"])
    s = _status()
    store.apply(y, to_dev(wl.x["g"]), st, meta, ws, dev_status=s)
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(s) & abi.LORA_DEV_SLOT_OUT_OF_RANGE
    got = to_host(y)
    np.testing.assert_array_equal(got[2], wl.y["g"][2])
    ok = np.array([0, 1, 3, 4, 5])
    check_bf16(got[ok], oracle_group(wl, "g", ok), ids[ok], wl.y["g"][ok], "bad group slot")


@pytest.mark.parametrize("n_rows", [300, 1000])
def test_bgmv_per_row_ids_over_several_scan_rounds(n_rows):
    """The per-row-id calls group their rows on the device, each CTA scanning
    the ids 256 (shrink) or 128 (expand) at a time.  Batches longer than one
    round, with slot 0 holding more than 16 rows in every round: its runs of
    16 span rounds.  Shrink and expand against the oracle; base rows keep
    their v and y."""
    rng = np.random.default_rng(n_rows)
    ids = rng.integers(-1, 5, n_rows).astype(np.int32)
    ids[rng.random(n_rows) < 0.3] = 0
    wl = _small(ids, 0, n_slots=5, rank=16, h_in=512, widths=(320,), mode="accumulate")
    st = store.GroupStore.from_workload(wl, "g")
    d_ids = torch.from_numpy(wl.ids).cuda()
    v = torch.full((n_rows, wl.r_slot), -7.0, device="cuda")
    y = to_dev(wl.y["g"])
    s = _status()
    abi.lora_bgmv_shrink(v, to_dev(wl.x["g"]), st.A[0], d_ids, h_in=512, r_slot=wl.r_slot, n_slots=5, dev_status=s)
    abi.lora_bgmv_expand(y, 0, 320, v, st.B[0], d_ids, r_slot=wl.r_slot, n_slots=5, dev_status=s)
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(s) == 0
    act = wl.ids >= 0
    got_v = v.cpu().numpy().astype(np.float64)
    ad = oracle_adapters(wl, "g", "p0")
    ref_v = O.shrink(wl.ids, wl.x["g"], ad, v_cols=wl.r_slot)
    bound = shrink_bound(wl.ids, wl.x["g"], [wl.A[("g", "p0", k)] for k in range(5)], 512)
    assert np.all(np.abs(got_v[act] - ref_v[act]) <= bound[act])
    assert np.all(got_v[~act] == -7.0), "base rows must not be written"
    check_bf16(to_host(y), oracle_group(wl, "g"), wl.ids, wl.y["g"], f"bgmv ids n_rows={n_rows}")


def test_bad_row_id_flagged_in_per_token_kernels():
    """The per-token BGMV entry points read lora_ids: ids outside [-1, n_slots)
    are flagged and those rows skipped."""
    ids = np.array([0, 1, 2, 3, 1, 0], np.int32)
    wl = _small(ids, 0, widths=(64,))
    st = store.GroupStore.from_workload(wl, "g")
    bad = torch.tensor([0, 1, 9, 3, -5, 0], dtype=torch.int32, device="cuda")
    v = torch.zeros(6, 8, device="cuda")
    y = to_dev(wl.y["g"])
    s = _status()
    abi.lora_bgmv_shrink(v, to_dev(wl.x["g"]), st.A[0], bad, h_in=64, r_slot=8, n_slots=4, dev_status=s)
    abi.lora_bgmv_expand(y, 0, 64, v, st.B[0], bad, r_slot=8, n_slots=4, dev_status=s)
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(s) & abi.LORA_DEV_SLOT_OUT_OF_RANGE
    got = to_host(y)
    np.testing.assert_array_equal(got[[2, 4]], wl.y["g"][[2, 4]])
    ok = np.array([0, 1, 3, 5])
    check_bf16(got[ok], oracle_group(wl, "g", ok), ids[ok], wl.y["g"][ok], "bad id")


@pytest.mark.parametrize("flags", [0, abi.LORA_APPLY_X_READY, abi.LORA_APPLY_NO_PDL,
                                   abi.LORA_APPLY_X_READY | abi.LORA_APPLY_NO_PDL,
                                   abi.LORA_APPLY_X_READY | abi.LORA_APPLY_Y_READY])
def test_apply_orderings_give_identical_bits(flags):
    """The launch-ordering flags change when work may start, never the result;
    a chain of calls with PDL matches the same chain with plain ordering."""
    wl = _wl("llama3b_decode", "accumulate")
    base = _run_apply(wl, "qkv")
    g = wl.groups[0]
    st = store.GroupStore.from_workload(wl, g.name)
    meta = store.BatchMeta(wl.ids, 0, wl.n_slots)
    ws = store.workspace_for(wl.n_rows, 3, wl.r_slot)
    x = to_dev(wl.x[g.name])
    y = to_dev(wl.y[g.name])
    ys = [y.clone() for _ in range(4)]
    for yy in ys:  # back-to-back dependent-free calls, then one call that re-reads its own output
        store.apply(yy, x, st, meta, ws, flags=flags)
    store.apply(ys[0], x, st, meta, ws, flags=flags)
    torch.cuda.synchronize()
    for yy in ys[1:]:
        np.testing.assert_array_equal(to_host(yy), base)
    twice = _run_apply(wl, "qkv")  # fresh: one application
    st2 = store.GroupStore.from_workload(wl, g.name)
    y2 = to_dev(twice)
    store.apply(y2, x, st2, meta, ws, flags=abi.LORA_APPLY_NO_PDL)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(ys[0]), to_host(y2))


def test_bad_segment_table_flagged():
    ids = np.repeat([0, 1], [6, 6]).astype(np.int32)
    wl = _small(ids, 12)
    st = store.GroupStore.from_workload(wl, "g")
    meta = store.BatchMeta(ids, 12, wl.n_slots)
    meta.seg_starts.copy_(torch.tensor([0, 6, 9], dtype=torch.int32))  # ends short of 12 rows
    s = _status()
    y = to_dev(wl.y["g"])
    store.apply(y, to_dev(wl.x["g"]), st, meta, store.workspace_for(12, 3, 8), dev_status=s)
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(s) & abi.LORA_DEV_BAD_SEGMENT
    got = to_host(y)
    np.testing.assert_array_equal(got[9:], wl.y["g"][9:])


def test_host_rejects_before_enqueue():
    wl = _small(np.zeros(4, np.int32), 0)
    st = store.GroupStore.from_workload(wl, "g")
    meta = store.BatchMeta(wl.ids, 0, wl.n_slots)
    y = to_dev(wl.y["g"])
    with pytest.raises(abi.LoraError) as e:
        store.apply(y, to_dev(wl.x["g"]), st, meta, store.workspace_for(1, 1, 8)[:16])
    assert e.value.name == "LORA_ERR_WORKSPACE"
    np.testing.assert_array_equal(to_host(y), wl.y["g"])


@pytest.mark.parametrize("h_in,widths,rank,T,n_slots", [
    (4096, (4096, 1024, 1024, 1024), 32, 200, 8),   # 4 projections x rank 32: 128 ranks per row
    (28672, (8192,), 16, 40, 4),                    # long K: the cluster's K chunks pipeline in stages
    (3072, (3072,), 8, 100, 2),                     # ~50 rows per adapter: several 16-row units each
    (256, (256, 64, 64), 16, 7, 3),                 # fewer rows than one unit
    (8192, (28672, 28672), 16, 20, 4),              # wide outputs: several expand tiles per CTA
    (1024, (1024,), 24, 20, 4),                     # slot rank not a multiple of 16
    (8192, (28672, 28672), 64, 12, 4),              # rank 64 above the BGMV cap: gather groups, column parts
    (28672, (8192,), 64, 9, 3),                     # rank 64, long K (70B down projection shape)
    (2048, (2048, 512, 512), 40, 25, 3),            # rank 40: K padded to 48 in the expand
])
def test_apply_decode_fused_shapes(h_in, widths, rank, T, n_slots):
    rng = np.random.default_rng(h_in + T)
    ids = rng.integers(-1, n_slots, T).astype(np.int32)
    wl = _small(ids, 0, n_slots=n_slots, rank=rank, h_in=h_in, widths=widths, seed=T)
    got = _run_apply(wl, "g")
    check_bf16(got, oracle_group(wl, "g"), wl.ids, wl.y["g"], f"fused h_in={h_in} R={rank * len(widths)}")


@pytest.mark.parametrize("h_in,widths,rank,T,n_slots,n_prefill,ks", [
    (1024, (2056, 520), 8, 30, 3, 0, None),       # ragged last column block in both projections; rank 8
    (512, (4096, 256, 264), 24, 70, 2, 0, None),  # three pieces of 16 bytes per B' row; >16 rows per adapter
    (2048, (1536,), 40, 45, 4, 0, None),          # rank 40: the second piece of each lane half empty
    (8192, (3072, 3072), 64, 26, 5, 0, None),     # rank 64: two pieces per lane, odd rows swapped
    (256, (256, 64, 64), 16, 50, 3, 20, None),    # prefill rows (row-wise route) before the decode rows
    (1032, (512,), 16, 30, 3, 0, None),           # K ends 8 elements into a stage: ragged last k-step
    (4104, (1024, 1024), 32, 40, 6, 0, 4),        # K split over a 4-CTA cluster, ragged in the last CTA
    (3072, (512, 512, 512), 16, 33, 4, 0, 2),     # 48 ranks: three 16-rank blocks, 2-CTA clusters
])
def test_apply_decode_two_launch_form(h_in, widths, rank, T, n_slots, n_prefill, ks, monkeypatch):
    """The grouped shrink followed by the grouped expand (the form wide or
    weight-heavy calls take), forced on for shapes that span its edge cases."""
    monkeypatch.setenv("LORA_DECODE_TWO_LAUNCH", "1")
    if ks:
        monkeypatch.setenv("LORA_GROUPED_KS", str(ks))
    rng = np.random.default_rng(h_in + T + rank)
    ids = rng.integers(-1, n_slots, T).astype(np.int32)
    wl = _small(ids, n_prefill, n_slots=n_slots, rank=rank, h_in=h_in, widths=widths, seed=T)
    got = _run_apply(wl, "g")
    check_bf16(got, oracle_group(wl, "g"), wl.ids, wl.y["g"], f"two-launch h_in={h_in} r={rank}")


def test_two_launch_form_skewed_groups(monkeypatch):
    """One adapter with 100 rows beside 30 with one row each: units are
    numbered by the block-wide scan instead of (group, sub-unit)."""
    monkeypatch.setenv("LORA_DECODE_TWO_LAUNCH", "1")
    rng = np.random.default_rng(11)
    ids = rng.permutation(np.concatenate([np.zeros(100), np.arange(1, 31)])).astype(np.int32)
    wl = _small(ids, 0, n_slots=31, rank=16, h_in=1024, widths=(1024,), seed=5)
    got = _run_apply(wl, "g")
    check_bf16(got, oracle_group(wl, "g"), wl.ids, wl.y["g"], "skewed groups")


@pytest.mark.parametrize("flags", [0, abi.LORA_APPLY_X_READY, abi.LORA_APPLY_NO_PDL])
def test_two_launch_form_chained_calls_share_workspace(flags, monkeypatch):
    """Back-to-back calls on one workspace: each call's shrink stores v only
    after the previous call's expand has finished reading it."""
    monkeypatch.setenv("LORA_DECODE_TWO_LAUNCH", "1")
    rng = np.random.default_rng(7)
    ids = rng.integers(-1, 4, 40).astype(np.int32)
    wl = _small(ids, 0, n_slots=4, rank=16, h_in=1024, widths=(2048, 512), seed=3)
    st = store.GroupStore.from_workload(wl, "g")
    meta = store.BatchMeta(wl.ids, 0, wl.n_slots)
    # distinct inputs per call (rows rotated), so a call that stored v too
    # early would change another call's output
    xs = [to_dev(np.roll(wl.x["g"], i, axis=0)) for i in range(6)]
    refs = []
    for xx in xs:
        yy = to_dev(wl.y["g"])
        store.apply(yy, xx, st, meta, store.workspace_for(wl.n_rows, 2, wl.r_slot))
        torch.cuda.synchronize()
        refs.append(to_host(yy))
    ws = store.workspace_for(wl.n_rows, 2, wl.r_slot)
    ys = [to_dev(wl.y["g"]) for _ in range(6)]
    for xx, yy in zip(xs, ys):
        store.apply(yy, xx, st, meta, ws, flags=flags)
    torch.cuda.synchronize()
    for yy, ref in zip(ys, refs):
        np.testing.assert_array_equal(to_host(yy), ref)
    check_bf16(refs[0], oracle_group(wl, "g"), wl.ids, wl.y["g"], "chained")


@pytest.mark.parametrize("threads", [128, 256])
@pytest.mark.parametrize("h_in,widths,rank,T,n_slots", [
    (4096, (4096, 1024, 1024, 1024), 32, 200, 8),   # 4 tiles of 8 ranks per warp at 128 threads
    (1024, (1024,), 24, 20, 4),                     # slot rank not a multiple of 16
    (8192, (28672,), 16, 40, 4),                    # long K, wide output (no column parts)
])
def test_apply_decode_fused_thread_counts(h_in, widths, rank, T, n_slots, threads, monkeypatch):
    """The one-launch kernel in both CTA sizes (128 threads for large grids,
    256 for small ones) on the same shapes."""
    monkeypatch.setenv("LORA_DECODE_TWO_LAUNCH", "0")
    monkeypatch.setenv("LORA_FUSED_THREADS", str(threads))
    rng = np.random.default_rng(h_in + T + threads)
    ids = rng.integers(-1, n_slots, T).astype(np.int32)
    wl = _small(ids, 0, n_slots=n_slots, rank=rank, h_in=h_in, widths=widths, seed=T)
    got = _run_apply(wl, "g")
    check_bf16(got, oracle_group(wl, "g"), wl.ids, wl.y["g"], f"fused threads={threads} h_in={h_in}")


@pytest.mark.parametrize("two_launch", ["0", "1"])
def test_apply_decode_understated_longest_group_flagged(two_launch, monkeypatch):
    """The grids of the decode kernels are sized from the host's bound on the
    longest group.  Understated, some rows get no CTA: the call flags it (and
    the rows it did cover are still right)."""
    monkeypatch.setenv("LORA_DECODE_TWO_LAUNCH", two_launch)
    ids = np.concatenate([np.zeros(40), [1, 2, 3]]).astype(np.int32)   # 40 rows on slot 0: three units
    wl = _small(ids, 0)
    st = store.GroupStore.from_workload(wl, "g")
    meta = store.BatchMeta(ids, 0, wl.n_slots)
    assert meta.c.max_gseg_len == 40
    meta.c.max_gseg_len = 1                                            # grid of 4 units for 6
    s = _status()
    y = to_dev(wl.y["g"])
    store.apply(y, to_dev(wl.x["g"]), st, meta, store.workspace_for(43, 3, 8), dev_status=s)
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(s) & abi.LORA_DEV_BAD_SEGMENT
    if two_launch == "0":   # the scan numbers slot 0's units first: all 40 rows are covered
        got = to_host(y)
        ok = np.arange(40)
        check_bf16(got[ok], oracle_group(wl, "g", ok), ids[ok], wl.y["g"][ok], "covered rows")
    # a correct bound: no flag
    meta.c.max_gseg_len = 40
    s2 = _status()
    store.apply(to_dev(wl.y["g"]), to_dev(wl.x["g"]), st, meta, store.workspace_for(43, 3, 8), dev_status=s2)
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(s2) == 0


def test_apply_decode_bad_permutation_flagged():
    """A corrupted gather permutation is flagged and its group's rows skipped."""
    ids = np.array([0, 1, 0, 1, 0, 1], np.int32)
    wl = _small(ids, 0)
    st = store.GroupStore.from_workload(wl, "g")
    meta = store.BatchMeta(ids, 0, wl.n_slots)
    meta.perm.copy_(torch.tensor([0, 2, 77, 1, 3, 5], dtype=torch.int32))  # slot 0's group has row 77
    s = _status()
    y = to_dev(wl.y["g"])
    store.apply(y, to_dev(wl.x["g"]), st, meta, store.workspace_for(6, 3, 8), dev_status=s)
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(s) & abi.LORA_DEV_BAD_SEGMENT
    got = to_host(y)
    np.testing.assert_array_equal(got[[0, 2, 4]], wl.y["g"][[0, 2, 4]])
    ok = np.array([1, 3, 5])
    check_bf16(got[ok], oracle_group(wl, "g", ok), ids[ok], wl.y["g"][ok], "slot 1 rows")


# ------------------------------------------- tensor-core SGMV (tcgen05) ----

def _segments(lens, slots):
    return np.concatenate([np.full(n, s, np.int32) for n, s in zip(lens, slots)])


@pytest.mark.parametrize("h_in,widths,rank,lens,slots", [
    (256, (256,), 16, [300, 5, 129, 64], [1, 2, -1, 3]),                 # tiles crossing segment ends
    (512, (512, 128, 128), 32, [70, 200, 128], [0, 3, 1]),               # q/k/v stack: 96 ranks
    (1024, (1024,), 64, [64, 640, 1], [2, 2, 0]),                        # same slot twice, 1-row segment
    (320, (320, 40, 40), 16, [130, 90], [3, 0]),                         # widths not multiples of 128
    (4096, (2048, 2048), 128, [256, 100], [1, 0]),                       # r_slot 128: two K blocks per plane
    (8200, (4096,), 16, [200], [2]),                                     # h_in not a multiple of 64
])
@pytest.mark.parametrize("mode", ["delta", "accumulate"])
@pytest.mark.parametrize("order", ["default", "dynamic"])
def test_apply_prefill_tensor_core(h_in, widths, rank, lens, slots, mode, order, monkeypatch):
    """Prefill segments of >= 64 rows take the tcgen05 shrink/expand route;
    "dynamic": the expand takes its work items from the call's counter even
    for these small items (the order it uses for large ones)."""
    if order == "dynamic":
        monkeypatch.setenv("LORA_TC_EXPAND_DYNAMIC", "2")
    ids = _segments(lens, slots)
    rng = np.random.default_rng(h_in)
    ids = np.concatenate([ids, rng.integers(-1, 4, 9).astype(np.int32)])   # plus some decode rows
    wl = _small(ids, int(sum(lens)), rank=rank, h_in=h_in, widths=widths, seed=rank, mode=mode)
    got = _run_apply(wl, "g")
    check_bf16(got, oracle_group(wl, "g"), wl.ids, wl.y["g"], f"tc h_in={h_in} rank={rank}")


@pytest.mark.parametrize("ks", [1, 2, 8])
@pytest.mark.parametrize("h_in,widths,rank,lens,slots", [
    (1024, (1024,), 64, [64, 640, 1], [2, 2, 0]),                        # 16 K blocks over the cluster
    (8200, (4096,), 16, [200], [2]),                                     # ragged last K block, uneven split
    (512, (512, 128, 128), 32, [70, 200, 128], [0, 3, 1]),               # 96 ranks: 6 column groups per row
])
def test_tensor_core_shrink_cluster_split(h_in, widths, rank, lens, slots, ks, monkeypatch):
    """The tensor-core shrink with K split over a cluster of ks CTAs per row
    tile (partials summed through distributed shared memory) and without."""
    monkeypatch.setenv("LORA_TC_SHRINK_KS", str(ks))
    ids = _segments(lens, slots)
    wl = _small(ids, int(sum(lens)), rank=rank, h_in=h_in, widths=widths, seed=rank + ks, mode="accumulate")
    got = _run_apply(wl, "g")
    check_bf16(got, oracle_group(wl, "g"), wl.ids, wl.y["g"], f"tc ks={ks} h_in={h_in}")


@pytest.mark.parametrize("grid,chunk", [(1, 2), (3, 1), (5, 4)])
def test_tensor_core_expand_few_ctas_walk_many_items(grid, chunk, monkeypatch):
    """The persistent expand on one, three or five CTAs with short work items:
    the TMA ring, the v-slice buffers and both accumulators wrap around many
    times and must stay in step (segments of several row tiles, base rows,
    widths that leave partial output tiles)."""
    monkeypatch.setenv("LORA_TC_EXPAND_GRID", str(grid))
    monkeypatch.setenv("LORA_TC_EXPAND_CHUNK", str(chunk))
    ids = _segments([300, 5, 129, 260, 64], [1, 2, -1, 3, 0])
    wl = _small(ids, int(ids.size), rank=32, h_in=256, widths=(384, 72, 72), seed=grid, mode="accumulate")
    got = _run_apply(wl, "g")
    check_bf16(got, oracle_group(wl, "g"), wl.ids, wl.y["g"], f"tc expand grid={grid} chunk={chunk}")


@pytest.mark.parametrize("ks", [1, 4])
def test_sgmv_shrink_tensor_core_fp32(ks, monkeypatch):
    """lora_sgmv_shrink on long contiguous segments (tensor-core route) gives
    fp32 v within the fp32 accumulation bound of the oracle's, with K whole
    or split over a cluster."""
    monkeypatch.setenv("LORA_TC_SHRINK_KS", str(ks))
    lens, slots = [150, 80, 300], [2, -1, 0]
    ids = _segments(lens, slots)
    wl = _small(ids, ids.size, rank=32, h_in=1024, widths=(64,), seed=9)
    st = store.GroupStore.from_workload(wl, "g")
    m = abi.lora_build_metadata(wl.ids, wl.n_prefill, wl.n_slots)
    v = torch.full((wl.n_rows, 32), -3.0, device="cuda")
    s = _status()
    abi.lora_sgmv_shrink(v, to_dev(wl.x["g"]), st.A[0], torch.from_numpy(m["seg_starts"]).cuda(),
                         torch.from_numpy(m["seg_slot"]).cuda(), m["n_segs"], None, wl.n_prefill, h_in=1024,
                         r_slot=32, n_slots=wl.n_slots, max_seg_len=m["max_seg_len"], dev_status=s)
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(s) == 0
    got = v.cpu().numpy().astype(np.float64)
    ad = oracle_adapters(wl, "g", "p0")
    ref = O.shrink(wl.ids, wl.x["g"], ad, v_cols=32)
    bound = shrink_bound(wl.ids, wl.x["g"], [wl.A[("g", "p0", k)] for k in range(wl.n_slots)], 1024)
    act = wl.ids >= 0
    assert np.all(np.abs(got[act] - ref[act]) <= bound[act])
    assert np.all(got[~act] == -3.0), "rows of slot -1 segments must not be written"


# ------------------------------------------------------ merge / unmerge ----

def _merge_case(out, h_in, r, r_slot, seed, std_w=1.0):
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn(out, h_in, generator=g) * std_w).to(torch.bfloat16)
    A = torch.zeros(r_slot, h_in, dtype=torch.bfloat16)
    A[:r] = (torch.randn(r, h_in, generator=g) * 0.05).to(torch.bfloat16)
    Bp = torch.zeros(out, r_slot, dtype=torch.bfloat16)
    Bp[:, :r] = (torch.randn(out, r, generator=g) * 0.05).to(torch.bfloat16)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return W, A, Bp, bits(W), bits(A[:r]), bits(Bp[:, :r])


@pytest.mark.parametrize("out,h_in,r,r_slot", [
    (300, 520, 13, 16),      # ragged row and column tiles; padding ranks
    (4096, 1024, 64, 64),    # full tiles, rank 64
    (70, 136, 100, 128),     # rank above 64: eight K steps
])
@pytest.mark.parametrize("sign", [1, -1])
def test_merge_vs_oracle(out, h_in, r, r_slot, sign):
    """W' = bf16(W + sign B'A) against the fp64 oracle: the kernel's fp32 sum
    may move a value across a rounding boundary, so elements agree within one
    bf16 step and nearly all bit for bit."""
    W, A, Bp, Wb, Ab, Bb = _merge_case(out, h_in, r, r_slot, seed=out + r)
    ref = O.bf16_to_f64(O.merge(Wb, Ab, Bb, sign))
    Wd = W.cuda()
    abi.lora_merge(Wd, A.cuda(), Bp.cuda(), sign)
    torch.cuda.synchronize()
    got = O.bf16_to_f64(to_host(Wd))
    # fp32 sum of r products plus W: error <= (r + 1) 2^-24 (sum |B'||A| + |W|);
    # then the one rounding may land one bf16 step (<= 2^-7 |value|) apart
    E = (r + 1) * 2.0 ** -24 * (np.abs(O.bf16_to_f64(Bb)) @ np.abs(O.bf16_to_f64(Ab)) + np.abs(O.bf16_to_f64(Wb)))
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * (np.abs(ref) + E) + E)
    assert (got != ref).mean() < 1e-3


def test_merge_full_size_gate_shape():
    """The benchmark's largest merge launch shape, every element: a
    Mistral-7B gate weight (14336 x 4096) with a rank-64 adapter, merged and
    then unmerged on the GPU, each against the fp64 oracle applied to the
    same input (row blocks over the host cores).  Bound as in
    test_merge_vs_oracle."""
    import concurrent.futures as cf
    out, h_in, r = 14336, 4096, 64
    W, A, Bp, Wb, Ab, Bb = _merge_case(out, h_in, r, r, seed=14336)
    Wd = W.cuda()
    Ad, Bd = A.cuda(), Bp.cuda()
    absA = np.abs(O.bf16_to_f64(Ab))

    def check(before_bits, after_bits, sign, what):
        def block(i0):
            i1 = min(out, i0 + 512)
            ref = O.bf16_to_f64(O.merge(before_bits[i0:i1], Ab, Bb[i0:i1], sign))
            got = O.bf16_to_f64(after_bits[i0:i1])
            E = (r + 1) * 2.0 ** -24 * (np.abs(O.bf16_to_f64(Bb[i0:i1])) @ absA +
                                        np.abs(O.bf16_to_f64(before_bits[i0:i1])))
            bad = int(np.sum(np.abs(got - ref) > 2.0 ** -7 * (np.abs(ref) + E) + E))
            return bad, int(np.sum(got != ref))
        with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as ex:
            res = list(ex.map(block, range(0, out, 512)))
        bad = sum(b for b, _ in res)
        diff = sum(d for _, d in res)
        assert bad == 0, f"{what}: {bad} elements outside the bound"
        assert diff < 1e-3 * out * h_in, f"{what}: {diff} elements differ from the oracle"

    abi.lora_merge(Wd, Ad, Bd, 1)
    torch.cuda.synchronize()
    merged = to_host(Wd)
    check(Wb, merged, 1, "merge")
    abi.lora_merge(Wd, Ad, Bd, -1)
    torch.cuda.synchronize()
    check(merged, to_host(Wd), -1, "unmerge")


def test_merge_unmerge_round_trip_exact():
    """Small integers: every value and sum is exact, so the merged weight
    equals the oracle's bit for bit and unmerge restores W bit for bit."""
    rng = np.random.default_rng(5)
    out, h_in, r = 200, 264, 8
    Wb = O.f64_to_bf16(rng.integers(-40, 41, (out, h_in)).astype(np.float64))
    Ab = O.f64_to_bf16(rng.integers(-3, 4, (r, h_in)).astype(np.float64))
    Bb = O.f64_to_bf16(rng.integers(-3, 4, (out, r)).astype(np.float64))
    Wd, Ad, Bd = to_dev(Wb), to_dev(Ab), to_dev(Bb)
    abi.lora_merge(Wd, Ad, Bd, 1)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(Wd), O.merge(Wb, Ab, Bb, 1))
    abi.lora_merge(Wd, Ad, Bd, -1)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(Wd), Wb)


@pytest.mark.parametrize("n", [5, 37])
def test_merge_batch_equals_single_merges_and_oracle(n):
    """n weights of assorted shapes (37: two launches) folded in one call:
    bit for bit what n single lora_merge calls give, and within the single
    kernel's bound of the oracle; a repeat with sign -1 takes them back
    out the same way."""
    rng = np.random.default_rng(n)
    shapes = [(int(rng.integers(1, 40)) * 8, int(rng.integers(1, 50)) * 8) for _ in range(n)]
    r, r_slot = 12, 16
    cases = [_merge_case(o, h, r, r_slot, seed=100 + i) for i, (o, h) in enumerate(shapes)]
    Wb_dev = [c[0].cuda() for c in cases]
    Ws_dev = [c[0].cuda() for c in cases]
    As = [c[1].cuda() for c in cases]
    Bs = [c[2].cuda() for c in cases]
    for sign in (1, -1):
        abi.lora_merge_batch(Wb_dev, As, Bs, sign)
        for W, A, B in zip(Ws_dev, As, Bs):
            abi.lora_merge(W, A, B, sign)
        torch.cuda.synchronize()
        for i in range(n):
            np.testing.assert_array_equal(to_host(Wb_dev[i]), to_host(Ws_dev[i]), err_msg=f"weight {i} sign {sign}")
    # the first merge against the oracle
    Wd = [c[0].cuda() for c in cases]
    abi.lora_merge_batch(Wd, As, Bs, 1)
    torch.cuda.synchronize()
    for i, (W, A, Bp, Wb, Ab, Bb) in enumerate(cases):
        ref = O.bf16_to_f64(O.merge(Wb, Ab, Bb, 1))
        got = O.bf16_to_f64(to_host(Wd[i]))
        E = (r + 1) * 2.0 ** -24 * (np.abs(O.bf16_to_f64(Bb)) @ np.abs(O.bf16_to_f64(Ab)) + np.abs(O.bf16_to_f64(Wb)))
        assert np.all(np.abs(got - ref) <= 2.0 ** -7 * (np.abs(ref) + E) + E), i


def test_merge_batch_rejects_before_enqueue():
    W, A, Bp, *_ = _merge_case(64, 128, 8, 16, seed=1)
    Wd, Ad, Bd = W.cuda(), A.cuda(), Bp.cuda()
    keep = to_host(Wd).copy()
    with pytest.raises(abi.LoraError) as e:
        abi.lora_merge_batch([Wd, Wd[:, 1:]], [Ad, Ad[:, 1:]], [Bd, Bd], 1)   # second weight misaligned
    assert e.value.name in ("LORA_ERR_ALIGNMENT", "LORA_ERR_SHAPE")
    with pytest.raises(abi.LoraError) as e:
        abi.lora_merge_batch([Wd], [Ad], [Bd], 2)
    assert e.value.name == "LORA_ERR_INVALID_ARG"
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_host(Wd), keep)   # nothing ran


def test_binding_checks_dtype_and_layout():
    """Arguments of the wrong element type, or operands whose columns are not
    contiguous, are refused by the binding before any launch."""
    wl = _small(np.array([0, 1, 0, 1], np.int32), 0, widths=(64,))
    st = store.GroupStore.from_workload(wl, "g")
    x = to_dev(wl.x["g"])
    ids = torch.from_numpy(wl.ids).cuda()
    v = torch.zeros(4, 8, device="cuda")
    with pytest.raises(ValueError, match="float32"):
        abi.lora_bgmv_shrink(v.double(), x, st.A[0], ids, h_in=64, r_slot=8, n_slots=4)
    with pytest.raises(ValueError, match="int32"):
        abi.lora_bgmv_shrink(v, x, st.A[0], ids.long(), h_in=64, r_slot=8, n_slots=4)
    with pytest.raises(ValueError, match="unit column stride"):
        abi.lora_bgmv_shrink(v, x.t(), st.A[0], ids, h_in=64, r_slot=8, n_slots=4)
    torch.cuda.synchronize()
    assert torch.all(v == 0)


def test_merge_rejects_bad_arguments_before_enqueue():
    W = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(64, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(abi.LoraError) as e:
        abi.lora_merge(W, A, B, 0)
    assert e.value.name == "LORA_ERR_INVALID_ARG"
    with pytest.raises(abi.LoraError) as e:
        abi.lora_merge(W[:, 1:], A[:, 1:], B, 1)    # unaligned W and h_in not a multiple of 8
    assert e.value.name in ("LORA_ERR_ALIGNMENT", "LORA_ERR_SHAPE")
    big = torch.zeros(136, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(abi.LoraError) as e:
        abi.lora_merge(W, big, B, 1)               # slot rank above the limit
    assert e.value.name == "LORA_ERR_RANK_EXCEEDS_SLOT"


# ------------------------------------------------------ adapter slots ----

def test_slot_manager_feeds_the_stores_end_to_end():
    """Six adapters through three GPU slots over several batches: the manager
    maps each batch's adapter ids to slots, loading what is missing by async
    copies on the stream, and lora_apply then matches the oracle computed
    from the adapters by id (true ranks, unpadded, scale folded by the oracle)."""
    h_in, projs, r_slot, n_slots = 128, [("q", 128), ("k", 32), ("v", 32)], 16, 3
    ranks = [4, 8, 16, 12, 16, 8]
    g = torch.Generator().manual_seed(12)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    A = {(k, p): bits((torch.randn(r, h_in, generator=g) * 0.1).to(torch.bfloat16))
         for k, r in enumerate(ranks) for p in range(len(projs))}
    B = {(k, p): bits((torch.randn(w, r, generator=g) * 0.1).to(torch.bfloat16))
         for k, r in enumerate(ranks) for p, (_, w) in enumerate(projs)}
    st = store.GroupStore(h_in, projs, n_slots, r_slot)
    m = abi.SlotManager([h_in] * len(projs), [w for _, w in projs], n_slots, r_slot, max_cpu=6,
                        A_stores=st.A, B_stores=st.B)
    for k, r in enumerate(ranks):
        m.register(k, [A[k, p] for p in range(len(projs))], [B[k, p] for p in range(len(projs))], r, 2.0 * r,
                   use_rslora=(k % 2 == 1))
    ads = [O.Adapters([A[k, p] for k in range(len(ranks))], [B[k, p] for k in range(len(ranks))],
                      [O.scale(2.0 * r, r, k % 2 == 1) for k, r in enumerate(ranks)]) for p in range(len(projs))]
    batches = [[0, 1, 2, 0, -1, 1], [3, 0, 3, 3], [4, 5, 3, -1, 5], [1, 2, 1], [5, 4, 0, 0]]
    stream = torch.cuda.current_stream()
    for n, ids in enumerate(batches):
        ids = np.array(ids, np.int32)
        slots = m.acquire(ids, stream=stream)
        x = bits((torch.randn(len(ids), h_in, generator=g)).to(torch.bfloat16))
        y = bits((torch.randn(len(ids), st.ld_y, generator=g)).to(torch.bfloat16))
        yd = to_dev(y)
        meta = store.BatchMeta(slots, 0, n_slots)
        store.apply(yd, to_dev(x), st, meta, store.workspace_for(len(ids), len(projs), r_slot), stream=stream)
        torch.cuda.synchronize()
        ref = y.copy()
        for p, off in enumerate(st.offsets):
            ref = O.apply_projection(ids, x, ref, off, ads[p])
        check_bf16(to_host(yd), ref, ids, y, f"slot batch {n}")
    s = m.stats()
    assert s["loads"] == 10 and s["slot_evictions"] == 7 and s["hits"] == 3, s
    m.close()


# ------------------------------------------------- tensor-parallel steps ----

@pytest.mark.parametrize("world", [2, 4])
def test_tensor_parallel_kernel_steps_two_layouts(world):
    """The sharded stores through the library's BGMV kernels (tp.kernel_steps),
    with the ranks run one after another on this device and the exchange on
    v done by a device concatenation (all_gather) or sum (all_reduce): both
    layouts must match the oracle's unsharded delta."""
    from lora_serving_gb300 import tp
    h_in, w, r_slot, n_slots, T = 256, 128, 32, 4, 37     # a rank's slice of v: 32 / world >= 8 columns
    ranks = [4, 32, 20, 8]
    g = torch.Generator().manual_seed(21)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    A = [bits((torch.randn(r, h_in, generator=g) * 0.1).to(torch.bfloat16)) for r in ranks]
    B = [bits((torch.randn(w, r, generator=g) * 0.1).to(torch.bfloat16)) for r in ranks]
    alphas = [2.0 * r for r in ranks]
    st = store.GroupStore(h_in, [("q", w)], n_slots, r_slot).load_slots(
        {k: [(A[k], B[k], alphas[k], False)] for k in range(n_slots)})
    ids = torch.randint(-1, n_slots, (T,), generator=g, dtype=torch.int32)
    x = bits(torch.randn(T, h_in, generator=g).to(torch.bfloat16))
    y = bits(torch.randn(T, w, generator=g).to(torch.bfloat16))
    ids_np = ids.numpy()
    ref = O.apply_projection(ids_np, x, y, 0, O.Adapters(A, B, [O.scale(a, r, False) for a, r in zip(alphas, ranks)]))
    s = _status()
    shrink, expand = tp.kernel_steps(ids.cuda(), n_slots, dev_status=s)
    xd, yd = to_dev(x), to_dev(y)

    # column-parallel: each rank's slice of v, gathered in rank order
    shards = [tp.shard_column(st.A[0], st.B[0], world, i) for i in range(world)]
    v = torch.cat([shrink(xd, a) for a, _ in shards], dim=1)
    cols = [tp._split(w, world, i) for i in range(world)]
    y_col = torch.cat([expand(yd[:, c].contiguous(), v, b) for c, (_, b) in zip(cols, shards)], dim=1)
    # row-parallel: partial v from each input slice, summed
    ks = [tp._split(h_in, world, i) for i in range(world)]
    rshards = [tp.shard_row(st.A[0], st.B[0], world, i) for i in range(world)]
    v_sum = sum(shrink(xd[:, k].contiguous(), a) for k, (a, _) in zip(ks, rshards))
    y_row = expand(yd.clone(), v_sum, rshards[0][1])
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(s) == 0
    check_bf16(to_host(y_col), ref, ids_np, y, f"column-parallel over {world}")
    check_bf16(to_host(y_row), ref, ids_np, y, f"row-parallel over {world}")


def test_slot_loads_spanning_several_gather_launches_land_exactly():
    """Twelve adapters of four projections loaded by one acquire: 96 pieces,
    so the gather takes two launches.  Every slot must then hold exactly the
    prepared adapter (scale folded, ranks padded), bit for bit, and slots
    the batch did not load keep their previous contents."""
    projs = [(128, 96), (64, 40), (256, 128), (72, 24)]   # (h_in, width): uneven sizes, multiples of 8
    n_slots, r_slot, n_ad = 14, 16, 12
    A_st = [torch.full((n_slots, r_slot, h), 7.0, dtype=torch.bfloat16, device="cuda") for h, _ in projs]
    B_st = [torch.full((n_slots, w, r_slot), 7.0, dtype=torch.bfloat16, device="cuda") for _, w in projs]
    m = abi.SlotManager([h for h, _ in projs], [w for _, w in projs], n_slots, r_slot, max_cpu=n_slots,
                        A_stores=A_st, B_stores=B_st)
    g = torch.Generator().manual_seed(31)
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    ranks = [4 + (k % 4) * 4 for k in range(n_ad)]
    prepared = {}
    for k, r in enumerate(ranks):
        A = [bits(torch.randn(r, h, generator=g).to(torch.bfloat16)) for h, _ in projs]
        B = [bits(torch.randn(w, r, generator=g).to(torch.bfloat16)) for _, w in projs]
        m.register(k, A, B, r, 2.0 * r, use_rslora=(k % 3 == 0))
        prepared[k] = [abi.lora_prepare_adapter(A[p], B[p], 2.0 * r, k % 3 == 0, r_slot) for p in range(len(projs))]
    slots = m.acquire(np.arange(n_ad), stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert len(set(slots.tolist())) == n_ad and m.stats()["loads"] == n_ad
    for k in range(n_ad):
        for p in range(len(projs)):
            np.testing.assert_array_equal(to_host(A_st[p][slots[k]]), prepared[k][p][0], err_msg=f"A adapter {k} proj {p}")
            np.testing.assert_array_equal(to_host(B_st[p][slots[k]]), prepared[k][p][1], err_msg=f"B adapter {k} proj {p}")
    untouched = sorted(set(range(n_slots)) - set(slots.tolist()))
    for p in range(len(projs)):
        for sl in untouched:
            assert bool((A_st[p][sl] == 7.0).all()) and bool((B_st[p][sl] == 7.0).all())
    m.close()
