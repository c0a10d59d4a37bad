"""ctypes wrapper around the fp64 CPU oracle in ``oracle.c``.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``. The product path never imports it.

Inputs are numpy arrays: ``float32``, ``float64``, ``float16``, or
``uint16`` holding raw bf16 bit patterns. Every function returns float64 results unless it is a
rounding helper.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32, BF16, F64, F16 = 0, 1, 2, 3

_lib = None


class Welford(ctypes.Structure):
    _fields_ = [("n", ctypes.c_double), ("mean", ctypes.c_double), ("m2", ctypes.c_double)]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        vp, i64, i32, dbl = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.oracle_row_moments.argtypes = [vp, i32, i64, ctypes.POINTER(dbl), ctypes.POINTER(dbl)]
        L.oracle_ln_fwd.argtypes = [vp, vp, vp, i32, i64, i64, dbl, vp, vp, vp]
        L.oracle_rms_fwd.argtypes = [vp, vp, i32, i64, i64, dbl, vp, vp]
        L.oracle_round_f32.argtypes = [vp, vp, i64]
        L.oracle_round_bf16.argtypes = [vp, vp, i64]
        L.oracle_round_f16.argtypes = [vp, vp, i64]
        L.oracle_quant_e4m3.argtypes = [vp, i64, dbl, vp]
        L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_value.restype = dbl
        L.oracle_welford_update.argtypes = [ctypes.POINTER(Welford), dbl]
        L.oracle_chan_combine.argtypes = [ctypes.POINTER(Welford)] * 3
        L.oracle_add_round.argtypes = [vp, vp, i32, i64, vp]
        L.oracle_ln_bwd.argtypes = [vp, vp, vp, i32, i64, i64, dbl, vp, vp, vp]
        L.oracle_rms_bwd.argtypes = [vp, vp, vp, i32, i64, i64, dbl, vp, vp]
        for f in ("oracle_row_moments", "oracle_ln_fwd", "oracle_rms_fwd", "oracle_round_f32",
                  "oracle_round_bf16", "oracle_welford_update", "oracle_chan_combine", "oracle_add_round",
                  "oracle_ln_bwd", "oracle_rms_bwd", "oracle_round_f16", "oracle_quant_e4m3"):
            getattr(L, f).restype = None
        L.oracle_abi_version.restype = ctypes.c_int
        _lib = L
    return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float64:
        return F64
    if a.dtype == np.float16:
        return F16
    raise TypeError(f"oracle inputs must be float32, float64, float16 or uint16 (bf16 bits), got {a.dtype}")


def _c(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def eps_as_f32(eps: float) -> float:
    """The ABI passes eps as fp32; the oracle uses that fp32 value widened."""
    return float(np.float32(eps))


def row_moments(x: np.ndarray):
    """(mean, biased variance) of a 1-D row, two-pass in fp64."""
    x = _c(x)
    m, v = ctypes.c_double(), ctypes.c_double()
    lib().oracle_row_moments(_ptr(x), _dtype_code(x), x.size, ctypes.byref(m), ctypes.byref(v))
    return m.value, v.value


def ln_fwd(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float):
    """LayerNorm forward of a 2-D array. Returns (y, mean, rstd) in float64."""
    x, gamma, beta = _c(x), _c(gamma), _c(beta)
    M, N = x.shape
    code = _dtype_code(x)
    assert _dtype_code(gamma) == code and _dtype_code(beta) == code
    assert gamma.size == N and beta.size == N
    y = np.empty((M, N), np.float64)
    mean = np.empty(M, np.float64)
    rstd = np.empty(M, np.float64)
    lib().oracle_ln_fwd(_ptr(x), _ptr(gamma), _ptr(beta), code, M, N, float(eps),
                        _ptr(y), _ptr(mean), _ptr(rstd))
    return y, mean, rstd


def rms_fwd(x: np.ndarray, w: np.ndarray, eps: float):
    """RMSNorm forward of a 2-D array. Returns (y, rstd) in float64."""
    x, w = _c(x), _c(w)
    M, N = x.shape
    code = _dtype_code(x)
    assert _dtype_code(w) == code and w.size == N
    y = np.empty((M, N), np.float64)
    rstd = np.empty(M, np.float64)
    lib().oracle_rms_fwd(_ptr(x), _ptr(w), code, M, N, float(eps), _ptr(y), _ptr(rstd))
    return y, rstd


def round_f32(v: np.ndarray) -> np.ndarray:
    v = _c(np.asarray(v, np.float64))
    out = np.empty(v.shape, np.float32)
    lib().oracle_round_f32(_ptr(v), _ptr(out), v.size)
    return out


def round_bf16(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16, nearest-even; returns raw uint16 bit patterns."""
    v = _c(np.asarray(v, np.float64))
    out = np.empty(v.shape, np.uint16)
    lib().oracle_round_bf16(_ptr(v), _ptr(out), v.size)
    return out


def round_f16(v: np.ndarray) -> np.ndarray:
    """Round fp64 values to IEEE fp16, nearest-even; returns float16."""
    v = _c(np.asarray(v, np.float64))
    out = np.empty(v.shape, np.uint16)
    lib().oracle_round_f16(_ptr(v), _ptr(out), v.size)
    return out.view(np.float16)


def quant_e4m3(y: np.ndarray, scale: float) -> np.ndarray:
    """E4M3 codes (uint8) of y / scale: nearest-even, saturating at 448."""
    y = _c(np.asarray(y, np.float64))
    q = np.empty(y.shape, np.uint8)
    lib().oracle_quant_e4m3(_ptr(y), y.size, float(scale), _ptr(q))
    return q


def e4m3_values(q: np.ndarray) -> np.ndarray:
    """Values of E4M3 codes (float64; NaN for 0x7F/0xFF)."""
    table = np.array([lib().oracle_e4m3_value(c) for c in range(256)])
    return table[np.asarray(q, np.uint8)]


def add_round(x: np.ndarray, r: np.ndarray) -> np.ndarray:
    """Residual add h = x + r rounded to the inputs' type (same shape)."""
    x, r = _c(x), _c(r)
    code = _dtype_code(x)
    assert _dtype_code(r) == code and x.shape == r.shape
    h = np.empty_like(x)
    lib().oracle_add_round(_ptr(x), _ptr(r), code, x.size, _ptr(h))
    return h


def ln_fwd_add(x, r, gamma, beta, eps):
    """Fused residual add + LayerNorm: returns (h, y, mean, rstd)."""
    h = add_round(x, r)
    return (h,) + ln_fwd(h, gamma, beta, eps)


def rms_fwd_add(x, r, w, eps):
    """Fused residual add + RMSNorm: returns (h, y, rstd)."""
    h = add_round(x, r)
    return (h,) + rms_fwd(h, w, eps)


def ln_bwd(dy: np.ndarray, x: np.ndarray, gamma: np.ndarray, eps: float):
    """LayerNorm backward of a 2-D array given the upstream gradient dy.
    Returns (dx, dgamma, dbeta) in float64."""
    dy, x, gamma = _c(dy), _c(x), _c(gamma)
    M, N = x.shape
    code = _dtype_code(x)
    assert _dtype_code(dy) == code and _dtype_code(gamma) == code and dy.shape == x.shape and gamma.size == N
    dx = np.empty((M, N), np.float64)
    dg = np.empty(N, np.float64)
    db = np.empty(N, np.float64)
    lib().oracle_ln_bwd(_ptr(dy), _ptr(x), _ptr(gamma), code, M, N, float(eps), _ptr(dx), _ptr(dg), _ptr(db))
    return dx, dg, db


def rms_bwd(dy: np.ndarray, x: np.ndarray, w: np.ndarray, eps: float):
    """RMSNorm backward of a 2-D array. Returns (dx, dw) in float64."""
    dy, x, w = _c(dy), _c(x), _c(w)
    M, N = x.shape
    code = _dtype_code(x)
    assert _dtype_code(dy) == code and _dtype_code(w) == code and dy.shape == x.shape and w.size == N
    dx = np.empty((M, N), np.float64)
    dw = np.empty(N, np.float64)
    lib().oracle_rms_bwd(_ptr(dy), _ptr(x), _ptr(w), code, M, N, float(eps), _ptr(dx), _ptr(dw))
    return dx, dw


def welford_update(s: Welford, x: float) -> Welford:
    r = Welford(s.n, s.mean, s.m2)
    lib().oracle_welford_update(ctypes.byref(r), float(x))
    return r


def chan_combine(a: Welford, b: Welford) -> Welford:
    out = Welford()
    lib().oracle_chan_combine(ctypes.byref(a), ctypes.byref(b), ctypes.byref(out))
    return out
