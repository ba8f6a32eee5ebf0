"""The bounded-wait path of the kernels (LORA_DEV_TIMEOUT), exercised on the
GPU without a fault: the library's test hook LORA_TEST_STALL arms one
kernel's first copy barrier for 16 bytes more than its copies deliver, so
that wait runs out after its limit while every copy still lands.  A call
must then return, report LORA_DEV_TIMEOUT, leave the rows that kernel owns
at y_in, finish the rows other kernels own correctly, and leave the device
usable: the next call on the same stream (tensor memory allocated again)
matches the oracle.

vLLM offline LoRA page, "limits": a failure is reported, never a hang."""
import time

import numpy as np
import pytest
import torch

from helpers import check_bf16, oracle_group, to_dev, to_host
from lora_serving_gb300 import abi, build, store, synth

pytestmark = pytest.mark.gpu

STALL = {"shrink_tc": 1, "expand_tc": 2, "fused_decode": 3}


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    abi.load()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"


def _case(h_in):
    """Prefill segments of 130, 70 and 20 rows (ids 1, 0, -1): the tensor-core
    SGMV kernels; then six decode rows: the one-launch decode kernel."""
    ids = np.array([1] * 130 + [0] * 70 + [-1] * 20 + [2, -1, 0, 1, 1, 3], np.int32)
    wl = synth.Workload("timeout", 9, [synth.Group("g", h_in, [("q", 256), ("k", 64)])], np.full(4, 16),
                        np.full(4, 32.0), np.zeros(4, bool), 16, ids, 220)
    return wl.materialise("accumulate")


def _call(wl, st, meta, ws, stream):
    y = to_dev(wl.y["g"])
    x = to_dev(wl.x["g"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        store.apply(y, x, st, meta, ws, dev_status=status)
    stream.synchronize()
    return to_host(y), abi.lora_read_device_status(status), time.perf_counter() - t0


@pytest.mark.parametrize("variant", [None, "shrink_ks_1", "expand_dynamic"])
@pytest.mark.parametrize("kernel", list(STALL))
def test_stalled_copy_reports_timeout_and_returns(kernel, variant, monkeypatch):
    if variant == "shrink_ks_1" and kernel != "shrink_tc":
        pytest.skip("the cluster split only concerns the shrink")
    if variant == "expand_dynamic" and kernel != "expand_tc":
        pytest.skip("the work-item order only concerns the expand")
    if variant == "shrink_ks_1":
        monkeypatch.setenv("LORA_TC_SHRINK_KS", "1")   # one CTA per row tile (no cluster)
    if variant == "expand_dynamic":
        monkeypatch.setenv("LORA_TC_EXPAND_DYNAMIC", "2")   # items from the call's counter
    wl = _case(h_in=1024)   # 16 K blocks: the shrink splits K over a cluster unless told not to
    st = store.GroupStore.from_workload(wl, "g")
    meta = store.BatchMeta(wl.ids, wl.n_prefill, wl.n_slots)
    ws = store.workspace_for(wl.n_rows, 2, wl.r_slot)
    stream = torch.cuda.Stream()
    ref = oracle_group(wl, "g")
    prefill = np.arange(wl.n_rows) < wl.n_prefill

    monkeypatch.setenv("LORA_TEST_STALL", str(STALL[kernel]))
    got, status, secs = _call(wl, st, meta, ws, stream)
    monkeypatch.delenv("LORA_TEST_STALL")
    assert status & abi.LORA_DEV_TIMEOUT, f"{kernel}: status {status:#x}"
    assert status == abi.LORA_DEV_TIMEOUT, f"{kernel}: unexpected bits {status:#x}"
    assert secs < 10.0, f"{kernel}: the call took {secs:.1f} s"
    # rows of the kernel that timed out keep y_in; the others are complete
    owned = prefill if kernel in ("shrink_tc", "expand_tc") else ~prefill
    np.testing.assert_array_equal(got[owned], wl.y["g"][owned], err_msg=f"{kernel}: rows it owns were written")
    other = ~owned
    check_bf16(got[other], ref[other], wl.ids[other], wl.y["g"][other], f"{kernel}: rows of the other kernels")

    # the device is usable afterwards: a normal call on the same stream
    got2, status2, _ = _call(wl, st, meta, ws, stream)
    assert status2 == 0
    check_bf16(got2, ref, wl.ids, wl.y["g"], f"{kernel}: the call after the timeout")
