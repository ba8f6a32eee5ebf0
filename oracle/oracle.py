"""ctypes wrapper around ``lora_oracle.c`` -- TEST INFRASTRUCTURE ONLY.

The C file holds every step of the arithmetic; this module only builds the
library with gcc, marshals numpy arrays and lays out the per-slot adapter
buffers.  Sources are cited in the C file's header: the TGI multi-LoRA page
(section "implementation 3. weight preprocessing", "4. SGMV and BGMV"), the
vLLM offline per-request LoRA page (steps 2 and 3) and the multi-LoRA serving
interview note ("direct answer", "interviewer follow-ups").

bf16 values travel as ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_LIB = os.path.join(_HERE, "liblora_oracle.so")
_lock = threading.Lock()
_lib = None

__all__ = [
    "build", "bf16_to_f64", "f64_to_bf16", "scale", "fold_B", "build_metadata",
    "Adapters", "shrink", "delta", "apply_projection", "expand", "merge", "linear_projection",
]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (strict IEEE double, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
            "-Wall", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm",
        ])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_bf16_to_double.restype = f64
            lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_double_to_bf16.restype = ctypes.c_uint16
            lib.oracle_double_to_bf16.argtypes = [f64]
            lib.oracle_bf16_to_double_array.argtypes = [P, P, i64]
            lib.oracle_double_to_bf16_array.argtypes = [P, P, i64]
            lib.oracle_scale.restype = f64
            lib.oracle_scale.argtypes = [f64, i32, i32]
            lib.oracle_fold_B.argtypes = [P, i32, i32, f64, P]
            lib.oracle_build_metadata.restype = i32
            lib.oracle_build_metadata.argtypes = [P, i32, i32, i32, P, P, P, P, P, P, P]
            lib.oracle_shrink.argtypes = [i32, P, P, i64, i32, P, P, P, P, i64, i32]
            lib.oracle_delta.argtypes = [i32, P, P, i64, i32, i32, P, P, P, P, P, P, P, i64]
            lib.oracle_apply_projection.argtypes = [i32, P, P, i64, i32, P, i64, i32, i32,
                                                    P, P, P, P, P, P]
            lib.oracle_expand.argtypes = [i32, P, P, i64, P, i64, i32, i32, P, P, P, P]
            lib.oracle_merge.argtypes = [P, i64, i32, i32, P, i64, P, i64, i32, i32, P]
            lib.oracle_linear_projection.argtypes = [i32, P, P, i64, i32, P, i64, P, i64, i32, i32,
                                                     P, P, P, P, P, P]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def bf16_to_f64(bits) -> np.ndarray:
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float64)
    _load().oracle_bf16_to_double_array(_ptr(bits), _ptr(out), bits.size)
    return out


def f64_to_bf16(vals) -> np.ndarray:
    vals = _c(vals, np.float64)
    out = np.empty(vals.shape, np.uint16)
    _load().oracle_double_to_bf16_array(_ptr(vals), _ptr(out), vals.size)
    return out


def scale(alpha: float, r: int, use_rslora: bool) -> float:
    return _load().oracle_scale(float(alpha), int(r), int(bool(use_rslora)))


def fold_B(B_bits, s: float) -> np.ndarray:
    B_bits = _c(B_bits, np.uint16)
    out_, r = B_bits.shape
    Bp = np.empty_like(B_bits)
    _load().oracle_fold_B(_ptr(B_bits), out_, r, float(s), _ptr(Bp))
    return Bp


def build_metadata(ids, n_prefill: int, n_slots: int):
    """Returns (seg_starts, seg_slot, perm, gseg_starts, gseg_slot) as int32 arrays."""
    ids = _c(ids, np.int32)
    T = ids.size
    seg_starts = np.zeros(n_prefill + 1, np.int32)
    seg_slot = np.zeros(max(n_prefill, 1), np.int32)
    perm = np.zeros(max(T - n_prefill, 1), np.int32)
    gseg_starts = np.zeros(n_slots + 2, np.int32)
    gseg_slot = np.zeros(n_slots + 1, np.int32)
    S = ctypes.c_int(0)
    G = ctypes.c_int(0)
    rc = _load().oracle_build_metadata(
        _ptr(ids), T, int(n_prefill), int(n_slots), _ptr(seg_starts), _ptr(seg_slot),
        ctypes.addressof(S), _ptr(perm), _ptr(gseg_starts), _ptr(gseg_slot), ctypes.addressof(G))
    if rc != 0:
        raise ValueError(f"oracle_build_metadata rejected the ids (code {rc})")
    s, g = S.value, G.value
    return (seg_starts[: s + 1].copy(), seg_slot[:s].copy(), perm[: T - n_prefill].copy(),
            gseg_starts[: g + 1].copy(), gseg_slot[:g].copy())


class Adapters:
    """Per-slot adapter matrices of one projection, laid out for the C oracle.

    ``A[k]`` is ``[r_k][h_in]`` and ``B[k]`` is ``[w][r_k]`` (peft orientation),
    both bf16 bit patterns, unscaled.  ``scales[k]`` is s_k.  A slot may be
    ``None`` (no adapter loaded there).
    """

    def __init__(self, A_list, B_list, scales):
        n = len(A_list)
        self.h_in = next(a.shape[1] for a in A_list if a is not None)
        self.w = next(b.shape[0] for b in B_list if b is not None)
        self.rp = np.zeros(n, np.int32)
        self.scale = np.zeros(n, np.float64)
        self.A_off = np.zeros(n, np.int64)
        self.B_off = np.zeros(n, np.int64)
        a_parts, b_parts = [], []
        ao = bo = 0
        for k in range(n):
            if A_list[k] is None:
                continue
            A = _c(A_list[k], np.uint16)
            B = _c(B_list[k], np.uint16)
            assert A.shape[1] == self.h_in and B.shape[0] == self.w and A.shape[0] == B.shape[1]
            self.rp[k] = A.shape[0]
            self.scale[k] = float(scales[k])
            self.A_off[k], self.B_off[k] = ao, bo
            a_parts.append(A.ravel())
            b_parts.append(B.ravel())
            ao += A.size
            bo += B.size
        self.A_cat = np.concatenate(a_parts) if a_parts else np.zeros(1, np.uint16)
        self.B_cat = np.concatenate(b_parts) if b_parts else np.zeros(1, np.uint16)


def shrink(ids, x_bits, ad: Adapters, v_cols: int | None = None) -> np.ndarray:
    """v[t][j] = (A_k x_t)[j] in fp64 (zero beyond rank and for base rows)."""
    ids = _c(ids, np.int32)
    x_bits = _c(x_bits, np.uint16)
    T = ids.size
    v_cols = int(ad.rp.max()) if v_cols is None else v_cols
    v = np.zeros((T, max(v_cols, 1)), np.float64)
    _load().oracle_shrink(T, _ptr(ids), _ptr(x_bits), x_bits.shape[1], ad.h_in, _ptr(ad.rp),
                          _ptr(ad.A_cat), _ptr(ad.A_off), _ptr(v), v.shape[1], v_cols)
    return v[:, :v_cols]


def delta(ids, x_bits, ad: Adapters) -> np.ndarray:
    """The unrounded fp64 delta B'_k (A_k x_t) of one projection, [T][w]."""
    ids = _c(ids, np.int32)
    x_bits = _c(x_bits, np.uint16)
    T = ids.size
    d = np.zeros((T, ad.w), np.float64)
    _load().oracle_delta(T, _ptr(ids), _ptr(x_bits), x_bits.shape[1], ad.h_in, ad.w,
                         _ptr(ad.rp), _ptr(ad.scale), _ptr(ad.A_cat), _ptr(ad.A_off),
                         _ptr(ad.B_cat), _ptr(ad.B_off), _ptr(d), ad.w)
    return d


def apply_projection(ids, x_bits, y_bits, off: int, ad: Adapters) -> np.ndarray:
    """Returns a copy of y with bf16_rne(y + delta) written into [off, off+w)."""
    ids = _c(ids, np.int32)
    x_bits = _c(x_bits, np.uint16)
    y = np.array(y_bits, dtype=np.uint16, copy=True, order="C")
    T = ids.size
    _load().oracle_apply_projection(T, _ptr(ids), _ptr(x_bits), x_bits.shape[1], ad.h_in,
                                    _ptr(y), y.shape[1], int(off), ad.w, _ptr(ad.rp),
                                    _ptr(ad.scale), _ptr(ad.A_cat), _ptr(ad.A_off),
                                    _ptr(ad.B_cat), _ptr(ad.B_off))
    return y


def expand(ids, v, y_bits, off: int, ad: Adapters) -> np.ndarray:
    """The expand step alone, from a given intermediate v (fp64, [T][>= r])."""
    ids = _c(ids, np.int32)
    v = _c(v, np.float64)
    y = np.array(y_bits, dtype=np.uint16, copy=True, order="C")
    T = ids.size
    _load().oracle_expand(T, _ptr(ids), _ptr(v), v.shape[1], _ptr(y), y.shape[1], int(off),
                          ad.w, _ptr(ad.rp), _ptr(ad.scale), _ptr(ad.B_cat), _ptr(ad.B_off))
    return y


def linear_projection(ids, x_bits, W_bits, y_bits, off: int, ad: Adapters) -> np.ndarray:
    """Returns a copy of y with bf16_rne(x W^T + delta) written into
    [off, off+w); W is this projection's base weight [w][h_in] (bf16 bits)."""
    ids = _c(ids, np.int32)
    x_bits = _c(x_bits, np.uint16)
    W = _c(W_bits, np.uint16)
    assert W.shape == (ad.w, ad.h_in)
    y = np.array(y_bits, dtype=np.uint16, copy=True, order="C")
    _load().oracle_linear_projection(ids.size, _ptr(ids), _ptr(x_bits), x_bits.shape[1], ad.h_in, _ptr(W),
                                     W.shape[1], _ptr(y), y.shape[1], int(off), ad.w, _ptr(ad.rp),
                                     _ptr(ad.scale), _ptr(ad.A_cat), _ptr(ad.A_off), _ptr(ad.B_cat),
                                     _ptr(ad.B_off))
    return y


def merge(W_bits, A_bits, Bp_bits, sign: int) -> np.ndarray:
    """W' = bf16_rne(W + sign * B' A) (sign +1 merge, -1 unmerge); W [out][h_in],
    A [r][h_in], B' [out][r], all bf16 bits; the true rank r is A's row count."""
    lib = _load()
    W = _c(W_bits, np.uint16)
    A = _c(A_bits, np.uint16)
    Bp = _c(Bp_bits, np.uint16)
    out, h_in = W.shape
    r = A.shape[0]
    assert A.shape == (r, h_in) and Bp.shape == (out, r) and sign in (1, -1)
    res = np.empty_like(W)
    lib.oracle_merge(_ptr(W), h_in, out, h_in, _ptr(A), h_in, _ptr(Bp), r, r, sign, _ptr(res))
    return res
