"""lora_apply_noalloc: the entry point for callers that cannot allocate device
memory when they call in (an engine whose KV-cache pool has taken nearly all
free HBM, a plug-in restricted to its host's memory pool).  It must give the
same result as lora_apply with a workspace, call after call, while keeping
its scratch in the library's own built-in array.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test.
"""
import numpy as np
import pytest
import torch

from helpers import check_bf16, to_dev, to_host
from lora_serving_gb300 import abi, build, store, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    abi.load()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"


def _problem(name, mode):
    wl = synth.get(name).materialise(mode, groups=[synth.get(name).groups[0].name])
    g = wl.groups[0]
    st = store.GroupStore.from_workload(wl, g.name)
    meta = store.BatchMeta(wl.ids, wl.n_prefill, wl.n_slots)
    return wl, g, st, meta


def _with_workspace(wl, g, st, meta):
    y = to_dev(wl.y[g.name])
    ws = store.workspace_for(wl.n_rows, len(g.projs), wl.r_slot)
    store.apply(y, to_dev(wl.x[g.name]), st, meta, ws)
    torch.cuda.synchronize()
    return to_host(y)


def _no_alloc(wl, g, st, meta):
    y = to_dev(wl.y[g.name])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    abi.lora_apply_noalloc(y, to_dev(wl.x[g.name]), g.h_in, st.c_projs(), st.r_slot, st.n_slots, meta.c,
                           dev_status=status)
    torch.cuda.synchronize()
    assert abi.lora_read_device_status(status) == 0
    return to_host(y)


def test_no_alloc_matches_workspace_entry_point_twice():
    """Two calls in a row on different batches (prefill segments through the
    scratch-using route, decode rows through the fused one): each matches
    lora_apply with a caller-allocated workspace."""
    for name, mode in (("mixed", "accumulate"), ("tiny", "delta")):
        wl, g, st, meta = _problem(name, mode)
        ref = _with_workspace(wl, g, st, meta)
        got = _no_alloc(wl, g, st, meta)
        check_bf16(got, ref, wl.ids, wl.y[g.name], f"no-alloc vs workspace, {name}")
        np.testing.assert_array_equal(got, ref)   # same kernels, same order: same bits


def test_no_alloc_back_to_back_on_one_stream():
    """The mixed and the tiny batch enqueued one after the other on one
    stream with no synchronisation between them: the second call's kernels
    may start early (programmatic dependent launch) while the first call
    still uses the shared scratch, and must still see only their own
    intermediate values.  Both results match the workspace entry point bit
    for bit."""
    probs = [_problem("mixed", "accumulate"), _problem("tiny", "delta")]
    refs = [_with_workspace(*p) for p in probs]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ys = []
    for flags in (0, abi.LORA_APPLY_X_READY):
        outs = []
        for wl, g, st, meta in probs:
            y = to_dev(wl.y[g.name])
            x = to_dev(wl.x[g.name])
            outs.append((y, x))
        torch.cuda.synchronize()
        for (wl, g, st, meta), (y, x) in zip(probs, outs):
            abi.lora_apply_noalloc(y, x, g.h_in, st.c_projs(), st.r_slot, st.n_slots, meta.c, flags=flags,
                                   dev_status=status)
        torch.cuda.synchronize()
        ys.append([to_host(y) for y, _ in outs])
    assert abi.lora_read_device_status(status) == 0
    for got in ys:
        for (wl, g, _, _), out, ref in zip(probs, got, refs):
            np.testing.assert_array_equal(out, ref, err_msg=f"back-to-back no-alloc call, {wl.name}")


def test_no_alloc_rejects_batches_beyond_its_scratch():
    rows = abi.LORA_NOALLOC_SCRATCH_BYTES // (3 * 64 * 4) + 1
    ids = np.zeros(rows, np.int32)
    meta = store.BatchMeta(ids, rows, 4)
    st = store.GroupStore(64, [("q", 64), ("k", 64), ("v", 64)], 4, 64)
    y = torch.zeros(rows, 192, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(rows, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(abi.LoraError) as e:
        abi.lora_apply_noalloc(y, x, 64, st.c_projs(), 64, 4, meta.c)
    assert e.value.name == "LORA_ERR_WORKSPACE"
