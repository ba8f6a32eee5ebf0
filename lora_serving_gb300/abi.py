"""Thin ctypes binding of ``liblora.so`` (the C ABI declared in include/lora.h).

Argument marshalling only: every function here has the name of the C entry
point it calls, takes torch tensors (device memory for kernel entry points,
host numpy arrays for the host helpers), reads their pointers and leading
dimensions, and raises ``LoraError`` on a non-OK status.  There is no
fallback: if the CUDA library is missing the import fails loudly.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblora.so")

LORA_MAX_RANK = 128
LORA_BGMV_MAX_RANK = 32
LORA_MAX_PROJ = 4
LORA_DEV_SLOT_OUT_OF_RANGE = 0x1
LORA_DEV_BAD_SEGMENT = 0x2
LORA_APPLY_X_READY = 0x1
LORA_APPLY_NO_PDL = 0x2
LORA_APPLY_Y_READY = 0x4
LORA_DEV_TIMEOUT = 0x4

STATUS = {
    0: "LORA_OK", 1: "LORA_ERR_INVALID_ARG", 2: "LORA_ERR_SHAPE",
    3: "LORA_ERR_RANK_EXCEEDS_SLOT", 4: "LORA_ERR_SLOT_RANGE", 5: "LORA_ERR_ALIGNMENT",
    6: "LORA_ERR_METADATA", 7: "LORA_ERR_WORKSPACE", 8: "LORA_ERR_CUDA",
}

# Every symbol include/lora.h declares.
EXPORTS = (
    "lora_bgmv_shrink", "lora_bgmv_expand", "lora_sgmv_shrink", "lora_sgmv_expand",
    "lora_apply", "lora_apply_workspace_bytes", "lora_build_metadata",
    "lora_prepare_adapter", "lora_slot_rank", "lora_read_device_status", "lora_status_string",
    "lora_kernel_launch_count", "lora_apply_noalloc", "lora_merge", "lora_merge_batch", "lora_linear",
    "lora_slots_create", "lora_slots_destroy", "lora_slots_register", "lora_slots_acquire",
    "lora_slots_slot_of", "lora_slots_stats",
)
LORA_NOALLOC_SCRATCH_BYTES = 16 << 20


class LoraError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        self.name = STATUS.get(status, str(status))
        super().__init__(f"{fn} returned {self.name}")


class lora_proj_t(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p),
                ("out_off", ctypes.c_int), ("width", ctypes.c_int)]


class lora_meta_t(ctypes.Structure):
    _fields_ = [("lora_ids", ctypes.c_void_p), ("n_rows", ctypes.c_int), ("n_prefill", ctypes.c_int),
                ("seg_starts", ctypes.c_void_p), ("seg_slot", ctypes.c_void_p), ("n_segs", ctypes.c_int),
                ("max_seg_len", ctypes.c_int),
                ("perm", ctypes.c_void_p), ("gseg_starts", ctypes.c_void_p), ("gseg_slot", ctypes.c_void_p),
                ("n_gsegs", ctypes.c_int), ("max_gseg_len", ctypes.c_int)]


_lib = None


def load(path: str | None = None):
    """Loads liblora.so once.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing: run lora_serving_gb300.build.build()")
    lib = ctypes.CDLL(path)
    P, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "lora_bgmv_shrink": [P, i32, P, i32, P, P, i32, i32, i32, i32, P, P],
        "lora_bgmv_expand": [P, i32, i32, i32, P, i32, P, P, i32, i32, i32, P, P],
        "lora_sgmv_shrink": [P, i32, P, i32, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, P, P],
        "lora_sgmv_expand": [P, i32, i32, i32, P, i32, P, P, P, i32, P, i32, i32, i32, i32, i32, P, P],
        "lora_apply": [P, i32, P, i32, i32, P, i32, i32, i32, P, P, sz, ctypes.c_uint32, P, P],
        "lora_apply_noalloc": [P, i32, P, i32, i32, P, i32, i32, i32, P, ctypes.c_uint32, P, P],
        "lora_apply_workspace_bytes": [i32, i32, i32],
        "lora_build_metadata": [P, i32, i32, i32, P, P, P, P, P, P, P, P, P],
        "lora_prepare_adapter": [P, P, i32, i32, i32, ctypes.c_double, i32, i32, P, P],
        "lora_slot_rank": [P, i32],
        "lora_read_device_status": [P, P, P],
        "lora_status_string": [i32],
        "lora_merge": [P, i32, i32, i32, P, P, i32, i32, P],
        "lora_merge_batch": [i32, P, P, P, P, P, P, i32, i32, P],
        "lora_linear": [P, i32, P, i32, i32, P, i32, P, i32, i32, i32, P, P, sz, P, P],
        "lora_slots_create": [i32, P, P, P, P, i32, i32, i32, P],
        "lora_slots_register": [P, ctypes.c_int64, P, P, i32, ctypes.c_double, i32],
        "lora_slots_acquire": [P, P, i32, P, P],
        "lora_slots_slot_of": [P, ctypes.c_int64],
        "lora_slots_stats": [P, P],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.lora_apply_workspace_bytes.restype = ctypes.c_size_t
    lib.lora_status_string.restype = ctypes.c_char_p
    lib.lora_kernel_launch_count.argtypes = []
    lib.lora_kernel_launch_count.restype = ctypes.c_uint64
    lib.lora_slots_destroy.argtypes = [P]
    lib.lora_slots_destroy.restype = None
    _lib = lib
    return lib


def _check(fn: str, st: int):
    if st != 0:
        raise LoraError(fn, st)


def _p(t) -> int:
    """Device/host pointer of a torch tensor, numpy array or raw int (0 = NULL)."""
    if t is None:
        return 0
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _ld(t) -> int:
    return int(t.stride(0))


_DTYPES = {"bf16": "torch.bfloat16", "f32": "torch.float32", "i32": "torch.int32"}


def _dev(t, name: str, dtype: str | None = None, mat: bool = False) -> int:
    """Device pointer of a kernel argument, after the checks the C ABI cannot
    make: a torch tensor on a CUDA device (a host pointer handed to a kernel
    is an illegal address), of the element type the kernel reads, and for
    row-major operands (mat) 2-D with unit column stride, so that the row
    stride is the leading dimension.  None (NULL) and raw integer pointers
    pass unchecked."""
    if t is None or isinstance(t, int):
        return _p(t)
    if not getattr(t, "is_cuda", False):
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and str(t.dtype) != _DTYPES[dtype]:
        raise ValueError(f"{name} must be {_DTYPES[dtype]}, got {t.dtype}")
    if mat and (t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1)):
        raise ValueError(f"{name} must be 2-D with unit column stride")
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ------------------------------------------------------------ kernels ----

def lora_bgmv_shrink(v, x, A, lora_ids, *, h_in, r_slot, n_slots, dev_status=None, stream=None):
    n_rows = int(lora_ids.numel())
    _check("lora_bgmv_shrink", load().lora_bgmv_shrink(
        _dev(v, "v", "f32", True), _ld(v), _dev(x, "x", "bf16", True), _ld(x), _dev(A, "A", "bf16"),
        _dev(lora_ids, "lora_ids", "i32"), n_rows, h_in, r_slot, n_slots, _dev(dev_status, "dev_status", "i32"),
        _stream(stream)))


def lora_bgmv_expand(y, y_off, width, v, B, lora_ids, *, r_slot, n_slots, dev_status=None,
                     stream=None, v_col=0):
    n_rows = int(lora_ids.numel())
    vp = _dev(v, "v", "f32", True) + 4 * v_col
    _check("lora_bgmv_expand", load().lora_bgmv_expand(
        _dev(y, "y", "bf16", True), _ld(y), y_off, width, vp, _ld(v), _dev(B, "B", "bf16"),
        _dev(lora_ids, "lora_ids", "i32"), n_rows, r_slot, n_slots, _dev(dev_status, "dev_status", "i32"),
        _stream(stream)))


def lora_sgmv_shrink(v, x, A, seg_starts, seg_slot, n_segs, row_perm, n_pos, *, h_in, r_slot,
                     n_slots, max_seg_len=0, dev_status=None, stream=None):
    _check("lora_sgmv_shrink", load().lora_sgmv_shrink(
        _dev(v, "v", "f32", True), _ld(v), _dev(x, "x", "bf16", True), _ld(x), _dev(A, "A", "bf16"),
        _dev(seg_starts, "seg_starts", "i32"), _dev(seg_slot, "seg_slot", "i32"), n_segs,
        _dev(row_perm, "row_perm", "i32"), n_pos, int(x.shape[0]), max_seg_len, h_in, r_slot, n_slots,
        _dev(dev_status, "dev_status", "i32"), _stream(stream)))


def lora_sgmv_expand(y, y_off, width, v, B, seg_starts, seg_slot, n_segs, row_perm, n_pos, *,
                     r_slot, n_slots, max_seg_len=0, dev_status=None, stream=None, v_col=0):
    vp = _dev(v, "v", "f32", True) + 4 * v_col
    _check("lora_sgmv_expand", load().lora_sgmv_expand(
        _dev(y, "y", "bf16", True), _ld(y), y_off, width, vp, _ld(v), _dev(B, "B", "bf16"),
        _dev(seg_starts, "seg_starts", "i32"), _dev(seg_slot, "seg_slot", "i32"), n_segs,
        _dev(row_perm, "row_perm", "i32"), n_pos, int(y.shape[0]), max_seg_len, r_slot, n_slots,
        _dev(dev_status, "dev_status", "i32"), _stream(stream)))


def make_projs(projs):
    """projs: sequence of (A_store, B_store, out_off, width) -> ctypes array."""
    arr = (lora_proj_t * len(projs))()
    for i, (A, B, off, w) in enumerate(projs):
        arr[i].A, arr[i].B, arr[i].out_off, arr[i].width = _p(A), _p(B), int(off), int(w)
    return arr


def lora_apply(y, x, h_in, projs, r_slot, n_slots, meta, workspace, *, flags=0, dev_status=None,
               stream=None):
    """projs: ctypes array from make_projs(); meta: lora_meta_t; workspace: device tensor;
    flags: LORA_APPLY_* bits."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("lora_apply", load().lora_apply(
        _dev(y, "y", "bf16", True), _ld(y), _dev(x, "x", "bf16", True), _ld(x), h_in, ctypes.addressof(projs),
        len(projs), r_slot, n_slots, ctypes.addressof(meta), _dev(workspace, "workspace"), ws_bytes, int(flags),
        _dev(dev_status, "dev_status", "i32"), _stream(stream)))


def lora_apply_noalloc(y, x, h_in, projs, r_slot, n_slots, meta, *, flags=0, dev_status=None, stream=None):
    """lora_apply with the library's built-in scratch instead of a workspace
    (for callers that cannot allocate device memory when they call in)."""
    _check("lora_apply_noalloc", load().lora_apply_noalloc(
        _dev(y, "y", "bf16", True), _ld(y), _dev(x, "x", "bf16", True), _ld(x), h_in, ctypes.addressof(projs),
        len(projs), r_slot, n_slots, ctypes.addressof(meta), int(flags), _dev(dev_status, "dev_status", "i32"),
        _stream(stream)))


def lora_linear(y, x, h_in, W, projs, r_slot, n_slots, meta, workspace, *, dev_status=None, stream=None):
    """y[:, off_p + c] = bf16(x W^T + B'_p (A_p x)) for every projection of
    projs (ctypes array from make_projs(), tiling W's rows in order); W is
    the stacked base weight [n_out][h_in] (row stride ld); y is written."""
    ws_bytes = workspace.numel() * workspace.element_size()
    _check("lora_linear", load().lora_linear(
        _dev(y, "y", "bf16", True), _ld(y), _dev(x, "x", "bf16", True), _ld(x), h_in, _dev(W, "W", "bf16", True),
        _ld(W), ctypes.addressof(projs), len(projs), r_slot, n_slots, ctypes.addressof(meta),
        _dev(workspace, "workspace"), ws_bytes, _dev(dev_status, "dev_status", "i32"), _stream(stream)))


def lora_merge(W, A, B, sign, *, stream=None):
    """W [out][h_in] (row stride ld) += sign * B A, one bf16 rounding; A is one
    adapter slot [r_slot][h_in] of the A store, B the same slot [out][r_slot]
    of the scaled B store; sign +1 merges, -1 unmerges."""
    out, h_in = int(W.shape[0]), int(W.shape[1])
    r_slot = int(A.shape[0])
    _check("lora_merge", load().lora_merge(_dev(W, "W", "bf16", True), _ld(W), out, h_in, _dev(A, "A", "bf16", True),
                                           _dev(B, "B", "bf16", True), r_slot, int(sign), _stream(stream)))


def lora_merge_batch(Ws, As, Bs, sign, *, stream=None):
    """lora_merge over every (W, A, B) of the lists in one launch (per 32);
    all A share the slot rank (their row count)."""
    n = len(Ws)
    P = ctypes.c_void_p
    arr_w, arr_a, arr_b = (P * max(1, n))(), (P * max(1, n))(), (P * max(1, n))()
    ld = (ctypes.c_int * max(1, n))()
    out = (ctypes.c_int * max(1, n))()
    h_in = (ctypes.c_int * max(1, n))()
    for i, (W, A, B) in enumerate(zip(Ws, As, Bs)):
        arr_w[i] = _dev(W, f"Ws[{i}]", "bf16", True)
        arr_a[i], arr_b[i] = _dev(A, f"As[{i}]", "bf16", True), _dev(B, f"Bs[{i}]", "bf16", True)
        ld[i], out[i], h_in[i] = _ld(W), int(W.shape[0]), int(W.shape[1])
    r_slot = int(As[0].shape[0]) if n else 8
    _check("lora_merge_batch", load().lora_merge_batch(n, arr_w, ld, out, h_in, arr_a, arr_b, r_slot, int(sign),
                                                       _stream(stream)))


class lora_slot_stats_t(ctypes.Structure):
    _fields_ = [("registered", ctypes.c_uint64), ("host_evictions", ctypes.c_uint64), ("hits", ctypes.c_uint64),
                ("loads", ctypes.c_uint64), ("slot_evictions", ctypes.c_uint64)]


class SlotManager:
    """The adapter slot manager (lora_slots_*): a host cache of prepared
    adapters feeding the GPU slots of the stores.  A_stores / B_stores: one
    device tensor per projection ([n_slots][r_slot][h_in], [n_slots][w][r_slot]),
    or None for the policy alone."""

    def __init__(self, h_in, width, n_slots, r_slot, max_cpu, A_stores=None, B_stores=None):
        self.n_proj = len(h_in)
        hi = (ctypes.c_int * self.n_proj)(*h_in)
        wd = (ctypes.c_int * self.n_proj)(*width)
        if A_stores is not None:
            self._a = (ctypes.c_void_p * self.n_proj)(*[_dev(t, "A_stores", "bf16") for t in A_stores])
            self._b = (ctypes.c_void_p * self.n_proj)(*[_dev(t, "B_stores", "bf16") for t in B_stores])
            a, b = ctypes.addressof(self._a), ctypes.addressof(self._b)
        else:
            a = b = 0
        self._h = ctypes.c_void_p()
        _check("lora_slots_create", load().lora_slots_create(self.n_proj, ctypes.addressof(hi), ctypes.addressof(wd),
                                                             a, b, n_slots, r_slot, max_cpu, ctypes.byref(self._h)))

    def close(self):
        if self._h:
            load().lora_slots_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def register(self, adapter_id, A_list, B_list, r, alpha, use_rslora=False):
        """A_list[p]: host uint16 bits [r][h_in_p]; B_list[p]: [w_p][r] (unscaled)."""
        A = [np.ascontiguousarray(a, dtype=np.uint16) for a in A_list]
        B = [np.ascontiguousarray(b, dtype=np.uint16) for b in B_list]
        ap = (ctypes.c_void_p * self.n_proj)(*[a.ctypes.data for a in A])
        bp = (ctypes.c_void_p * self.n_proj)(*[b.ctypes.data for b in B])
        _check("lora_slots_register", load().lora_slots_register(self._h, int(adapter_id), ctypes.addressof(ap),
                                                                 ctypes.addressof(bp), int(r), float(alpha),
                                                                 int(bool(use_rslora))))

    def acquire(self, adapter_ids, stream=0) -> np.ndarray:
        """Adapter ids of a batch (-1 = base) -> slot ids, loading what is missing."""
        ids = np.ascontiguousarray(adapter_ids, dtype=np.int64)
        out = np.empty(ids.size, np.int32)
        st = stream if isinstance(stream, int) else _stream(stream)
        _check("lora_slots_acquire", load().lora_slots_acquire(self._h, ids.ctypes.data, int(ids.size),
                                                               out.ctypes.data, st))
        return out

    def slot_of(self, adapter_id) -> int:
        return int(load().lora_slots_slot_of(self._h, int(adapter_id)))

    def stats(self) -> dict:
        s = lora_slot_stats_t()
        _check("lora_slots_stats", load().lora_slots_stats(self._h, ctypes.byref(s)))
        return {f: int(getattr(s, f)) for f, _ in s._fields_}


def lora_apply_workspace_bytes(n_rows, n_proj, r_slot) -> int:
    return int(load().lora_apply_workspace_bytes(n_rows, n_proj, r_slot))


def lora_read_device_status(dev_status, stream=None) -> int:
    out = ctypes.c_int32(0)
    _check("lora_read_device_status", load().lora_read_device_status(
        _dev(dev_status, "dev_status", "i32"), ctypes.addressof(out), _stream(stream)))
    return out.value


# ------------------------------------------------------- host helpers ----

def lora_build_metadata(ids: np.ndarray, n_prefill: int, n_slots: int):
    """Returns dict of int32 arrays seg_starts, seg_slot, perm, gseg_starts,
    gseg_slot and ints n_segs, max_seg_len, n_gsegs, max_gseg_len."""
    ids = np.ascontiguousarray(ids, np.int32)
    T = ids.size
    D = T - n_prefill
    seg_starts = np.zeros(n_prefill + 1, np.int32)
    seg_slot = np.zeros(max(n_prefill, 1), np.int32)
    perm = np.zeros(max(D, 1), np.int32)
    gseg_starts = np.zeros(n_slots + 2, np.int32)
    gseg_slot = np.zeros(n_slots + 1, np.int32)
    S, MS, G, MG = (ctypes.c_int(0) for _ in range(4))
    _check("lora_build_metadata", load().lora_build_metadata(
        _p(ids), T, n_prefill, n_slots, _p(seg_starts), _p(seg_slot), ctypes.addressof(S),
        ctypes.addressof(MS), _p(perm), _p(gseg_starts), _p(gseg_slot), ctypes.addressof(G),
        ctypes.addressof(MG)))
    s, g = S.value, G.value
    return dict(seg_starts=seg_starts[: s + 1].copy(), seg_slot=seg_slot[:s].copy(), n_segs=s,
                max_seg_len=MS.value, perm=perm[:D].copy(), gseg_starts=gseg_starts[: g + 1].copy(),
                gseg_slot=gseg_slot[:g].copy(), n_gsegs=g, max_gseg_len=MG.value)


def lora_prepare_adapter(A: np.ndarray, B: np.ndarray, alpha: float, use_rslora: bool, r_slot: int,
                         A_slot_out: np.ndarray | None = None, B_slot_out: np.ndarray | None = None):
    """A [r][h_in], B [out][r] (uint16 bf16 bits) -> padded (A_slot, B'_slot)."""
    A = np.ascontiguousarray(A, np.uint16)
    B = np.ascontiguousarray(B, np.uint16)
    r, h_in = A.shape
    out = B.shape[0]
    if B.shape[1] != r:
        raise ValueError("lora_B must be [out][r] with the rank of lora_A")
    if A_slot_out is None:
        A_slot_out = np.empty((r_slot, h_in), np.uint16)
    if B_slot_out is None:
        B_slot_out = np.empty((out, r_slot), np.uint16)
    assert A_slot_out.flags.c_contiguous and B_slot_out.flags.c_contiguous
    _check("lora_prepare_adapter", load().lora_prepare_adapter(
        _p(A), _p(B), r, h_in, out, float(alpha), int(bool(use_rslora)), r_slot,
        _p(A_slot_out), _p(B_slot_out)))
    return A_slot_out, B_slot_out


def lora_slot_rank(ranks) -> int:
    arr = np.ascontiguousarray(ranks, np.int32)
    return int(load().lora_slot_rank(_p(arr), arr.size))


def lora_kernel_launch_count() -> int:
    return int(load().lora_kernel_launch_count())


def lora_status_string(status: int) -> str:
    return load().lora_status_string(status).decode()
