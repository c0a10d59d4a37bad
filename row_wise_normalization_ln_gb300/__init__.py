"""GB300-native row-wise LayerNorm / RMSNorm forward: Python binding of the
libnorm C ABI (include/libnorm.h).

The binding only marshals arguments: it reshapes ``[..., N]`` inputs to
``[M, N]`` rows (the T3 drill's host wrapper, §④), allocates outputs with
torch, and passes raw device pointers and the current CUDA stream to the
C library. Every step of the computation runs in the library's CUDA
kernels; there is no fallback. If ``libnorm.so`` has not been built the
first call raises ``LibraryNotBuilt``.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

__all__ = [
    "ln_fwd", "rms_fwd", "ln_fwd_add", "rms_fwd_add", "ln_fwd_fp8", "rms_fwd_fp8", "ln_bwd", "rms_bwd",
    "make_plan", "make_bwd_plan", "NormPlan", "NormError", "LibraryNotBuilt", "library", "host_rows_pipeline",
    "host_rows_wait",
    "NORM_F32", "NORM_BF16", "NORM_F16", "NORM_MAP_GROUP", "NORM_MAP_CTA",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnorm.so")

NORM_F32, NORM_BF16, NORM_F16 = 0, 1, 2
NORM_OK, NORM_ERR_ARG, NORM_ERR_DTYPE, NORM_ERR_CUDA, NORM_ERR_PLAN, NORM_ERR_TIMEOUT = 0, -1, -2, -3, -4, -5
NORM_MAP_GROUP, NORM_MAP_CTA = 0, 1


class NormPlan(ctypes.Structure):
    """Mirror of ``norm_plan`` in include/libnorm.h."""
    _fields_ = [
        ("mapping", ctypes.c_int32),
        ("vec_elems", ctypes.c_int32),
        ("per_thread", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("threads", ctypes.c_int32),
        ("cluster", ctypes.c_int32),
        ("rounds", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("grid", ctypes.c_int64),
    ]

    def as_dict(self) -> dict:
        return {k: getattr(self, k) for k, _ in self._fields_}

    @classmethod
    def from_dict(cls, d: dict) -> "NormPlan":
        p = cls()
        for k, v in d.items():
            setattr(p, k, int(v))
        return p


class NormError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = library().norm_status_string(status).decode()
        if status == NORM_ERR_CUDA:
            msg += f" (cudaError {library().norm_last_cuda_error()})"
        super().__init__(f"{what}: {msg} [status {status}]")


class LibraryNotBuilt(ImportError):
    pass


_lib = None


def library() -> ctypes.CDLL:
    """The loaded libnorm.so with its C signatures declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise LibraryNotBuilt(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, f32, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    L.ln_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, f32, i32, vp]
    L.rms_fwd.argtypes = [vp, vp, vp, i64, i64, f32, i32, vp]
    L.ln_fwd_planned.argtypes = L.ln_fwd.argtypes + [ctypes.POINTER(NormPlan)]
    L.rms_fwd_planned.argtypes = L.rms_fwd.argtypes + [ctypes.POINTER(NormPlan)]
    L.ln_fwd_add.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, f32, i32, vp]
    L.rms_fwd_add.argtypes = [vp, vp, vp, vp, vp, i64, i64, f32, i32, vp]
    L.ln_fwd_add_planned.argtypes = L.ln_fwd_add.argtypes + [ctypes.POINTER(NormPlan)]
    L.rms_fwd_add_planned.argtypes = L.rms_fwd_add.argtypes + [ctypes.POINTER(NormPlan)]
    L.norm_make_plan.argtypes = [i64, i64, i32, i32, i32, ctypes.POINTER(NormPlan)]
    L.norm_make_plan_add.argtypes = L.norm_make_plan.argtypes
    sz = ctypes.c_size_t
    L.ln_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i64, i64, i32, vp]
    L.rms_bwd.argtypes = [vp, vp, vp, vp, vp, vp, sz, i64, i64, f32, i32, vp]
    L.ln_bwd_planned.argtypes = L.ln_bwd.argtypes + [ctypes.POINTER(NormPlan)]
    L.rms_bwd_planned.argtypes = L.rms_bwd.argtypes + [ctypes.POINTER(NormPlan)]
    L.norm_bwd_make_plan.argtypes = [i64, i64, i32, i32, i32, i32, ctypes.POINTER(NormPlan)]
    L.norm_bwd_workspace_bytes.argtypes = [ctypes.POINTER(NormPlan), i64, i32, ctypes.POINTER(sz)]
    L.ln_fwd_strided.argtypes = [vp, i64, vp, vp, vp, i64, vp, vp, i64, i64, f32, i32, vp, ctypes.POINTER(NormPlan)]
    L.rms_fwd_strided.argtypes = [vp, i64, vp, vp, i64, i64, i64, f32, i32, vp, ctypes.POINTER(NormPlan)]
    L.ln_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, f32, i32, vp]
    L.rms_fwd_fp8.argtypes = [vp, vp, vp, vp, i64, i64, f32, i32, vp]
    L.ln_fwd_add_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, f32, i32, vp]
    L.rms_fwd_add_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, f32, i32, vp]
    L.ln_fwd_fp8_planned.argtypes = L.ln_fwd_add_fp8.argtypes + [ctypes.POINTER(NormPlan)]
    L.rms_fwd_fp8_planned.argtypes = L.rms_fwd_add_fp8.argtypes + [ctypes.POINTER(NormPlan)]
    for f in ("ln_fwd", "rms_fwd", "ln_fwd_planned", "rms_fwd_planned", "ln_fwd_add", "rms_fwd_add",
              "ln_fwd_add_planned", "rms_fwd_add_planned", "norm_make_plan", "norm_make_plan_add",
              "ln_bwd", "rms_bwd", "ln_bwd_planned", "rms_bwd_planned", "norm_bwd_make_plan",
              "norm_bwd_workspace_bytes", "ln_fwd_fp8", "rms_fwd_fp8", "ln_fwd_add_fp8", "rms_fwd_add_fp8",
              "ln_fwd_fp8_planned", "rms_fwd_fp8_planned", "ln_fwd_strided", "rms_fwd_strided",
              "norm_last_cuda_error", "norm_abi_version", "norm_wait_timeouts", "norm_synchronize",
              "norm_set_wait_limit", "norm_wait_limit"):
        getattr(L, f).restype = ctypes.c_int
    L.norm_wait_timeouts.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.norm_synchronize.argtypes = []
    L.norm_set_wait_limit.argtypes = [ctypes.c_uint64]
    L.norm_wait_limit.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
    L.norm_status_string.argtypes = [ctypes.c_int]
    L.norm_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def wait_timeouts() -> int:
    """Waits of the ring kernels (plans with stages >= 2) that ran out of
    time on the current device since the last call; resets the count.
    Synchronises the device."""
    n = ctypes.c_uint32(0)
    st = library().norm_wait_timeouts(ctypes.byref(n))
    if st != NORM_OK:
        raise NormError(st, "norm_wait_timeouts")
    return n.value


def synchronize() -> None:
    """Synchronise the current device and raise NormError (status
    NORM_ERR_TIMEOUT) if a ring kernel's wait for a bulk copy ran out since
    the last check; the count is reset either way."""
    st = library().norm_synchronize()
    if st != NORM_OK:
        raise NormError(st, "norm_synchronize")


def set_wait_limit(ns: int) -> None:
    """Time limit, in nanoseconds, of the ring kernels' per-row waits on the
    current device (default 2e9; 0 tests each copy once and gives up if it
    has not landed; at most 6e10). Applies to kernels launched afterwards."""
    st = library().norm_set_wait_limit(int(ns))
    if st != NORM_OK:
        raise NormError(st, "norm_set_wait_limit")


def wait_limit() -> int:
    """The current device's per-row wait limit in nanoseconds."""
    v = ctypes.c_uint64(0)
    st = library().norm_wait_limit(ctypes.byref(v))
    if st != NORM_OK:
        raise NormError(st, "norm_wait_limit")
    return v.value


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return NORM_F32
    if t == torch.bfloat16:
        return NORM_BF16
    if t == torch.float16:
        return NORM_F16
    raise TypeError(f"libnorm supports float32, bfloat16 and float16, got {t}")


def make_plan(M: int, N: int, dtype: torch.dtype, aligned: bool = True, num_sms: int = 152,
              add: bool = False) -> dict:
    """The launch plan the library would choose (host-only, no CUDA call);
    ``add`` for the fused residual-add calls."""
    p = NormPlan()
    fn = library().norm_make_plan_add if add else library().norm_make_plan
    st = fn(M, N, _dtype_code(dtype), int(aligned), num_sms, ctypes.byref(p))
    if st != NORM_OK:
        raise NormError(st, "norm_make_plan")
    return p.as_dict()


def make_bwd_plan(M: int, N: int, dtype: torch.dtype, layer_norm: bool, aligned: bool = True,
                  num_sms: int = 152) -> dict:
    """The backward plan ln_bwd / rms_bwd would choose (host-only)."""
    p = NormPlan()
    st = library().norm_bwd_make_plan(M, N, _dtype_code(dtype), int(layer_norm), int(aligned), num_sms,
                                      ctypes.byref(p))
    if st != NORM_OK:
        raise NormError(st, "norm_bwd_make_plan")
    return p.as_dict()


def bwd_workspace_bytes(plan, N: int, layer_norm: bool) -> int:
    n = ctypes.c_size_t()
    p = plan if isinstance(plan, NormPlan) else NormPlan.from_dict(plan)
    st = library().norm_bwd_workspace_bytes(ctypes.byref(p), N, int(layer_norm), ctypes.byref(n))
    if st != NORM_OK:
        raise NormError(st, "norm_bwd_workspace_bytes")
    return n.value


def _rows(x: torch.Tensor) -> torch.Tensor:
    if x.dim() == 0:
        raise ValueError("input must have at least one dimension")
    x2 = x.reshape(-1, x.shape[-1])
    return x2 if x2.is_contiguous() else x2.contiguous()


def _strided_rows(x: torch.Tensor) -> torch.Tensor:
    """[M, N] rows of x without a copy when its rows are evenly strided with
    unit inner stride (the T3 drill's host wrapper, §④); else a contiguous
    copy."""
    if x.dim() == 0:
        raise ValueError("input must have at least one dimension")
    x2 = x.reshape(-1, x.shape[-1])
    if x2.stride(-1) == 1 and (x2.shape[0] <= 1 or x2.stride(0) >= x2.shape[1]):
        return x2
    return x2.contiguous()


def _pitch(t: torch.Tensor) -> int:
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


def _param(p: torch.Tensor, x: torch.Tensor, name: str) -> torch.Tensor:
    if p.device != x.device or p.dtype != x.dtype:
        raise ValueError(f"{name} must be on {x.device} with dtype {x.dtype}")
    if p.numel() != x.shape[-1]:
        raise ValueError(f"{name} must have {x.shape[-1]} elements, got {p.numel()}")
    return p.reshape(-1).contiguous()


def _out(t: Optional[torch.Tensor], x: torch.Tensor, x2: torch.Tensor, name: str) -> torch.Tensor:
    y = t if t is not None else torch.empty_like(x2)
    if y.shape != x.shape and y.shape != x2.shape or not y.is_contiguous() or y.dtype != x.dtype \
            or y.device != x.device:
        raise ValueError(f"{name} must be a contiguous tensor of x's shape, dtype and device")
    return y


def _strided_out(out: Optional[torch.Tensor], x: torch.Tensor, x2: torch.Tensor) -> torch.Tensor:
    """The output rows: a new contiguous tensor, or `out` (of x's shape and
    dtype) as strided rows when its rows are evenly strided."""
    if out is None:
        return torch.empty(x2.shape, dtype=x.dtype, device=x.device)
    if out.shape != x.shape and out.shape != x2.shape or out.dtype != x.dtype or out.device != x.device:
        raise ValueError("out must have x's shape, dtype and device")
    y = out.reshape(-1, x2.shape[1])   # a view when the leading dims collapse into one row stride
    if y.data_ptr() != out.data_ptr() or y.stride(-1) != 1 or (y.shape[0] > 1 and y.stride(0) < y.shape[1]):
        raise ValueError("out must have evenly strided rows with unit inner stride")
    return y


def _shaped(y: torch.Tensor, x: torch.Tensor, out: Optional[torch.Tensor]) -> torch.Tensor:
    return out if out is not None else y.view(x.shape)


def _residual(r: torch.Tensor, x: torch.Tensor) -> torch.Tensor:
    if r.shape != x.shape or r.dtype != x.dtype or r.device != x.device:
        raise ValueError("residual must have x's shape, dtype and device")
    return _rows(r)


def _stats(M: int, x: torch.Tensor, mean, rstd, stats: bool):
    if not stats:
        return None, None
    mean = mean if mean is not None else torch.empty(M, device=x.device, dtype=torch.float32)
    rstd = rstd if rstd is not None else torch.empty(M, device=x.device, dtype=torch.float32)
    for t, n in ((mean, "mean"), (rstd, "rstd")):
        if t.dtype != torch.float32 or t.numel() != M or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous fp32 tensor of {M} elements")
    return mean, rstd


def _ptr(t: Optional[torch.Tensor]):
    return t.data_ptr() if t is not None else None


def _stream_handle(stream: Optional[torch.cuda.Stream], device: torch.device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _plan_ptr(plan):
    if plan is None:
        return None
    p = plan if isinstance(plan, NormPlan) else NormPlan.from_dict(plan)
    return ctypes.byref(p)


def ln_fwd(x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, eps: float = 1e-5, *,
           out: Optional[torch.Tensor] = None, mean: Optional[torch.Tensor] = None,
           rstd: Optional[torch.Tensor] = None, stats: bool = True,
           stream: Optional[torch.cuda.Stream] = None, plan=None):
    """LayerNorm forward over the last dimension of a CUDA tensor.

    Returns ``(y, mean, rstd)``; mean and rstd are fp32 ``[M]`` (None when
    ``stats=False``). ``out`` may be ``x`` itself (in place)."""
    if not x.is_cuda:
        raise ValueError("ln_fwd needs a CUDA tensor")
    code = _dtype_code(x.dtype)
    x2 = _strided_rows(x)
    M, N = x2.shape
    g = _param(gamma, x, "gamma")
    b = _param(beta, x, "beta")
    y = _strided_out(out, x, x2)
    mean, rstd = _stats(M, x, mean, rstd, stats)
    L = library()
    with torch.cuda.device(x.device):
        h = _stream_handle(stream, x.device)
        if x2.is_contiguous() and y.is_contiguous():
            args = (x2.data_ptr(), g.data_ptr(), b.data_ptr(), y.data_ptr(), _ptr(mean), _ptr(rstd),
                    M, N, float(eps), code)
            st = (L.ln_fwd(*args, h) if plan is None else L.ln_fwd_planned(*args, h, _plan_ptr(plan)))
        else:
            st = L.ln_fwd_strided(x2.data_ptr(), _pitch(x2), g.data_ptr(), b.data_ptr(), y.data_ptr(), _pitch(y),
                                  _ptr(mean), _ptr(rstd), M, N, float(eps), code, h, _plan_ptr(plan))
    if st != NORM_OK:
        raise NormError(st, "ln_fwd")
    return _shaped(y, x, out), mean, rstd


def rms_fwd(x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, *, out: Optional[torch.Tensor] = None,
            stream: Optional[torch.cuda.Stream] = None, plan=None) -> torch.Tensor:
    """RMSNorm forward over the last dimension of a CUDA tensor."""
    if not x.is_cuda:
        raise ValueError("rms_fwd needs a CUDA tensor")
    code = _dtype_code(x.dtype)
    x2 = _strided_rows(x)
    M, N = x2.shape
    wv = _param(w, x, "w")
    y = _strided_out(out, x, x2)
    L = library()
    with torch.cuda.device(x.device):
        h = _stream_handle(stream, x.device)
        if x2.is_contiguous() and y.is_contiguous():
            args = (x2.data_ptr(), wv.data_ptr(), y.data_ptr(), M, N, float(eps), code)
            st = (L.rms_fwd(*args, h) if plan is None else L.rms_fwd_planned(*args, h, _plan_ptr(plan)))
        else:
            st = L.rms_fwd_strided(x2.data_ptr(), _pitch(x2), wv.data_ptr(), y.data_ptr(), _pitch(y), M, N,
                                   float(eps), code, h, _plan_ptr(plan))
    if st != NORM_OK:
        raise NormError(st, "rms_fwd")
    return _shaped(y, x, out)


def ln_fwd_add(x: torch.Tensor, residual: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor,
               eps: float = 1e-5, *, h_out: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
               mean: Optional[torch.Tensor] = None, rstd: Optional[torch.Tensor] = None, stats: bool = True,
               stream: Optional[torch.cuda.Stream] = None, plan=None):
    """Fused residual add + LayerNorm: ``h = x + residual`` (rounded to x's
    dtype), ``y = LayerNorm(h)``. Returns ``(h, y, mean, rstd)``. ``h_out``
    may be ``residual`` or ``x`` (in-place residual update) and so may
    ``out``; the two must differ."""
    if not x.is_cuda:
        raise ValueError("ln_fwd_add needs a CUDA tensor")
    code = _dtype_code(x.dtype)
    x2 = _rows(x)
    r2 = _residual(residual, x)
    M, N = x2.shape
    g = _param(gamma, x, "gamma")
    b = _param(beta, x, "beta")
    hh = _out(h_out, x, x2, "h_out")
    y = _out(out, x, x2, "out")
    mean, rstd = _stats(M, x, mean, rstd, stats)
    L = library()
    args = (x2.data_ptr(), r2.data_ptr(), g.data_ptr(), b.data_ptr(), hh.data_ptr(), y.data_ptr(),
            _ptr(mean), _ptr(rstd), M, N, float(eps), code)
    with torch.cuda.device(x.device):
        s = _stream_handle(stream, x.device)
        st = (L.ln_fwd_add(*args, s) if plan is None else L.ln_fwd_add_planned(*args, s, _plan_ptr(plan)))
    if st != NORM_OK:
        raise NormError(st, "ln_fwd_add")
    return hh.view(x.shape), y.view(x.shape), mean, rstd


def rms_fwd_add(x: torch.Tensor, residual: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, *,
                h_out: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None, plan=None):
    """Fused residual add + RMSNorm: ``h = x + residual``, ``y = RMSNorm(h)``.
    Returns ``(h, y)``; aliasing as for ``ln_fwd_add``."""
    if not x.is_cuda:
        raise ValueError("rms_fwd_add needs a CUDA tensor")
    code = _dtype_code(x.dtype)
    x2 = _rows(x)
    r2 = _residual(residual, x)
    M, N = x2.shape
    wv = _param(w, x, "w")
    hh = _out(h_out, x, x2, "h_out")
    y = _out(out, x, x2, "out")
    L = library()
    args = (x2.data_ptr(), r2.data_ptr(), wv.data_ptr(), hh.data_ptr(), y.data_ptr(), M, N, float(eps), code)
    with torch.cuda.device(x.device):
        s = _stream_handle(stream, x.device)
        st = (L.rms_fwd_add(*args, s) if plan is None else L.rms_fwd_add_planned(*args, s, _plan_ptr(plan)))
    if st != NORM_OK:
        raise NormError(st, "rms_fwd_add")
    return hh.view(x.shape), y.view(x.shape)


def _aligned16(*ts) -> bool:
    return all(t.data_ptr() % 16 == 0 for t in ts)


def _bwd_common(dy, x, w, layer_norm, dx, workspace, plan):
    if not x.is_cuda:
        raise ValueError("the backward needs CUDA tensors")
    code = _dtype_code(x.dtype)
    if dy.shape != x.shape or dy.dtype != x.dtype or dy.device != x.device:
        raise ValueError("dy must have x's shape, dtype and device")
    x2, dy2 = _rows(x), _rows(dy)
    M, N = x2.shape
    wv = _param(w, x, "gamma" if layer_norm else "w")
    dxt = _out(dx, x, x2, "dx")
    if plan is None:
        sms = torch.cuda.get_device_properties(x.device).multi_processor_count
        pl = make_bwd_plan(M, N, x.dtype, layer_norm, _aligned16(x2, dy2, wv, dxt), sms)
    else:
        pl = dict(plan)
    need = bwd_workspace_bytes(pl, N, layer_norm)
    if workspace is None:
        workspace = torch.empty(max(need, 16) // 4 + 4, dtype=torch.float32, device=x.device)
    nbytes = workspace.numel() * workspace.element_size()
    return code, x2, dy2, M, N, wv, dxt, workspace, nbytes


def ln_bwd(dy: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor, mean: torch.Tensor, rstd: torch.Tensor, *,
           dx: Optional[torch.Tensor] = None, dgamma: Optional[torch.Tensor] = None,
           dbeta: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
           stream: Optional[torch.cuda.Stream] = None, plan=None):
    """LayerNorm backward: returns ``(dx, dgamma, dbeta)``; dgamma and dbeta
    are fp32 ``[N]``. ``mean``/``rstd`` are ln_fwd's fp32 statistics.
    ``workspace`` (a CUDA tensor, any dtype) is allocated when not given."""
    code, x2, dy2, M, N, g, dxt, ws, nbytes = _bwd_common(dy, x, gamma, True, dx, workspace, plan)
    for t, n in ((mean, "mean"), (rstd, "rstd")):
        if t.dtype != torch.float32 or t.numel() != M or not t.is_contiguous() or t.device != x.device:
            raise ValueError(f"{n} must be a contiguous fp32 CUDA tensor of {M} elements")
    dg = dgamma if dgamma is not None else torch.empty(N, dtype=torch.float32, device=x.device)
    db = dbeta if dbeta is not None else torch.empty(N, dtype=torch.float32, device=x.device)
    for t, n in ((dg, "dgamma"), (db, "dbeta")):
        if t.dtype != torch.float32 or t.numel() != N or not t.is_contiguous() or t.device != x.device:
            raise ValueError(f"{n} must be a contiguous fp32 CUDA tensor of {N} elements")
    L = library()
    args = (dy2.data_ptr(), x2.data_ptr(), g.data_ptr(), mean.data_ptr(), rstd.data_ptr(), dxt.data_ptr(),
            dg.data_ptr(), db.data_ptr(), ws.data_ptr(), nbytes, M, N, code)
    with torch.cuda.device(x.device):
        s = _stream_handle(stream, x.device)
        st = L.ln_bwd(*args, s) if plan is None else L.ln_bwd_planned(*args, s, _plan_ptr(plan))
    if st != NORM_OK:
        raise NormError(st, "ln_bwd")
    return dxt.view(x.shape), dg, db


def rms_bwd(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, eps: float = 1e-6, *,
            dx: Optional[torch.Tensor] = None, dw: Optional[torch.Tensor] = None,
            workspace: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None, plan=None):
    """RMSNorm backward: returns ``(dx, dw)``, dw fp32 ``[N]``; rstd is
    recomputed from x with ``eps`` (the forward's)."""
    code, x2, dy2, M, N, wv, dxt, ws, nbytes = _bwd_common(dy, x, w, False, dx, workspace, plan)
    dwt = dw if dw is not None else torch.empty(N, dtype=torch.float32, device=x.device)
    if dwt.dtype != torch.float32 or dwt.numel() != N or not dwt.is_contiguous() or dwt.device != x.device:
        raise ValueError(f"dw must be a contiguous fp32 CUDA tensor of {N} elements")
    L = library()
    args = (dy2.data_ptr(), x2.data_ptr(), wv.data_ptr(), dxt.data_ptr(), dwt.data_ptr(), ws.data_ptr(), nbytes,
            M, N, float(eps), code)
    with torch.cuda.device(x.device):
        s = _stream_handle(stream, x.device)
        st = L.rms_bwd(*args, s) if plan is None else L.rms_bwd_planned(*args, s, _plan_ptr(plan))
    if st != NORM_OK:
        raise NormError(st, "rms_bwd")
    return dxt.view(x.shape), dwt


def _scale_tensor(scale, device) -> torch.Tensor:
    if isinstance(scale, torch.Tensor):
        if scale.dtype != torch.float32 or scale.numel() != 1 or scale.device != device:
            raise ValueError("scale must be one fp32 value on the input's device")
        return scale.reshape(1)
    return torch.tensor([float(scale)], dtype=torch.float32, device=device)


def _fp8_out(out, x, x2) -> torch.Tensor:
    y8 = out if out is not None else torch.empty(x2.shape, dtype=torch.uint8, device=x.device)
    if y8.numel() != x2.numel() or not y8.is_contiguous() or y8.element_size() != 1 or y8.device != x.device:
        raise ValueError("out must be a contiguous one-byte tensor of x's shape on its device")
    return y8


def ln_fwd_fp8(x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, scale, eps: float = 1e-5, *,
               residual: Optional[torch.Tensor] = None, h_out: Optional[torch.Tensor] = None,
               out: Optional[torch.Tensor] = None, mean: Optional[torch.Tensor] = None,
               rstd: Optional[torch.Tensor] = None, stats: bool = True,
               stream: Optional[torch.cuda.Stream] = None, plan=None):
    """LayerNorm forward with an FP8 E4M3 output, ``y8 = E4M3(y / scale)``
    (uint8 codes; ``.view(torch.float8_e4m3fn)`` reads them as fp8).
    ``scale``: a float or one fp32 CUDA value. Returns ``(y8, mean, rstd)``,
    or ``(h, y8, mean, rstd)`` with ``residual`` (fused add, h = x + r)."""
    if not x.is_cuda:
        raise ValueError("ln_fwd_fp8 needs a CUDA tensor")
    code = _dtype_code(x.dtype)
    x2 = _rows(x)
    M, N = x2.shape
    g = _param(gamma, x, "gamma")
    b = _param(beta, x, "beta")
    sc = _scale_tensor(scale, x.device)
    y8 = _fp8_out(out, x, x2)
    r2 = _residual(residual, x) if residual is not None else None
    hh = _out(h_out, x, x2, "h_out") if residual is not None else None
    mean, rstd = _stats(M, x, mean, rstd, stats)
    L = library()
    with torch.cuda.device(x.device):
        s = _stream_handle(stream, x.device)
        if plan is not None:
            st = L.ln_fwd_fp8_planned(x2.data_ptr(), _ptr(r2), g.data_ptr(), b.data_ptr(), sc.data_ptr(), _ptr(hh),
                                      y8.data_ptr(), _ptr(mean), _ptr(rstd), M, N, float(eps), code, s,
                                      _plan_ptr(plan))
        elif residual is not None:
            st = L.ln_fwd_add_fp8(x2.data_ptr(), r2.data_ptr(), g.data_ptr(), b.data_ptr(), sc.data_ptr(),
                                  hh.data_ptr(), y8.data_ptr(), _ptr(mean), _ptr(rstd), M, N, float(eps), code, s)
        else:
            st = L.ln_fwd_fp8(x2.data_ptr(), g.data_ptr(), b.data_ptr(), sc.data_ptr(), y8.data_ptr(), _ptr(mean),
                              _ptr(rstd), M, N, float(eps), code, s)
    if st != NORM_OK:
        raise NormError(st, "ln_fwd_fp8")
    y8 = y8.view(x.shape)
    if residual is not None:
        return hh.view(x.shape), y8, mean, rstd
    return y8, mean, rstd


def rms_fwd_fp8(x: torch.Tensor, w: torch.Tensor, scale, eps: float = 1e-6, *,
                residual: Optional[torch.Tensor] = None, h_out: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None, plan=None):
    """RMSNorm forward with an FP8 E4M3 output; returns ``y8``, or
    ``(h, y8)`` with ``residual``."""
    if not x.is_cuda:
        raise ValueError("rms_fwd_fp8 needs a CUDA tensor")
    code = _dtype_code(x.dtype)
    x2 = _rows(x)
    M, N = x2.shape
    wv = _param(w, x, "w")
    sc = _scale_tensor(scale, x.device)
    y8 = _fp8_out(out, x, x2)
    r2 = _residual(residual, x) if residual is not None else None
    hh = _out(h_out, x, x2, "h_out") if residual is not None else None
    L = library()
    with torch.cuda.device(x.device):
        s = _stream_handle(stream, x.device)
        if plan is not None:
            st = L.rms_fwd_fp8_planned(x2.data_ptr(), _ptr(r2), wv.data_ptr(), sc.data_ptr(), _ptr(hh),
                                       y8.data_ptr(), M, N, float(eps), code, s, _plan_ptr(plan))
        elif residual is not None:
            st = L.rms_fwd_add_fp8(x2.data_ptr(), r2.data_ptr(), wv.data_ptr(), sc.data_ptr(), hh.data_ptr(),
                                   y8.data_ptr(), M, N, float(eps), code, s)
        else:
            st = L.rms_fwd_fp8(x2.data_ptr(), wv.data_ptr(), sc.data_ptr(), y8.data_ptr(), M, N, float(eps), code, s)
    if st != NORM_OK:
        raise NormError(st, "rms_fwd_fp8")
    y8 = y8.view(x.shape)
    if residual is not None:
        return hh.view(x.shape), y8
    return y8


# ------------------------------------------------------------ host buffers
_PIPELINES = {}
_PIPELINES_LOCK = threading.Lock()


def _pipeline_streams(dev: torch.device):
    """The copy-in and copy-back streams, the per-buffer events and a lock of
    host_rows_pipeline on `dev`, made once. Events are reused: each wait is
    queued after the record it refers to, which the lock keeps true when
    several host threads call at once."""
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    with _PIPELINES_LOCK:
        p = _PIPELINES.get(key)
        if p is None:
            p = (torch.cuda.Stream(dev), torch.cuda.Stream(dev), [torch.cuda.Event() for _ in range(2)],
                 [torch.cuda.Event() for _ in range(2)],  # the kernels of the buffer's last chunk
                 [torch.cuda.Event() for _ in range(2)],  # the copy back of the buffer's last chunk
                 threading.Lock())
            _PIPELINES[key] = p
    return p


def host_rows_pipeline(inputs, outputs, call, *, chunk_rows: Optional[int] = None,
                       device: Optional[torch.device] = None, wait: bool = True):
    """Run a row-wise library call over pinned host tensors, overlapping the
    copies in both directions with the kernels.

    ``inputs`` and ``outputs`` are lists of pinned CPU tensors whose first
    dimension is the row count M (an FP8 output is a uint8 tensor; per-row
    statistics are ``[M]`` fp32 tensors). The rows are taken in chunks of
    ``chunk_rows`` (default: M/4, at least 256 rows): chunk c+1 is copied to
    the device on one stream while chunk c runs on the current stream and
    chunk c-1 is copied back on a third, through two device staging buffers
    per tensor (allocated with torch). ``call(ins, outs)`` receives device
    tensors holding one chunk's rows and launches the library call for them
    on the current stream, e.g. ``lambda i, o: rms_fwd(i[0], w, eps,
    out=o[0])`` with ``w`` already on the device. Returns when all work is
    queued; the current stream waits for the last copy back, so a
    ``torch.cuda.synchronize()`` (or an event on the current stream) makes
    the host outputs readable. With ``wait=False`` it does not: the copies
    back of this call may then still run while the next call's rows are
    copied in and normalised (a stream of batches keeps both copy
    directions busy), and ``host_rows_wait()`` (or a device
    synchronisation) orders them before later work on the current stream.
    Not for calls that reduce over rows (the backward's column
    gradients)."""
    if not inputs or not outputs:
        raise ValueError("inputs and outputs must be non-empty lists of pinned host tensors")
    M = inputs[0].shape[0]
    for t in list(inputs) + list(outputs):
        if t.device.type != "cpu" or t.shape[0] != M or not t.is_contiguous():
            raise ValueError("host tensors must be contiguous CPU tensors with the same number of rows")
    if M == 0:
        return  # nothing to copy (an empty tensor has no storage to pin)
    for t in list(inputs) + list(outputs):
        if not t.is_pinned():
            raise ValueError("host tensors must be pinned (tensor.pin_memory())")
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    chunk = chunk_rows if chunk_rows is not None else max(256, -(-M // 4))
    chunk = max(1, min(chunk, M))
    comp = torch.cuda.current_stream(dev)
    s_in, s_out, in_ready, done, copied, lock = _pipeline_streams(dev)
    with lock:
        _enqueue_pipeline(inputs, outputs, call, M, chunk, dev, comp, s_in, s_out, in_ready, done, copied, wait)


def host_rows_wait(device: Optional[torch.device] = None) -> None:
    """Make the current stream wait for every copy back that
    ``host_rows_pipeline`` has queued on ``device`` (for calls made with
    ``wait=False``)."""
    dev = device if device is not None else torch.device("cuda", torch.cuda.current_device())
    s_in, s_out, _, _, _, lock = _pipeline_streams(dev)
    with lock:
        torch.cuda.current_stream(dev).wait_stream(s_out)


def _enqueue_pipeline(inputs, outputs, call, M, chunk, dev, comp, s_in, s_out, in_ready, done, copied, wait):
    d_in = [[torch.empty((chunk,) + tuple(t.shape[1:]), dtype=t.dtype, device=dev) for t in inputs] for _ in range(2)]
    d_out = [[torch.empty((chunk,) + tuple(t.shape[1:]), dtype=t.dtype, device=dev) for t in outputs] for _ in range(2)]
    s_in.wait_stream(comp)                            # staging memory and inputs as of now
    s_out.wait_stream(comp)                           # (a call without wait: not its copies back)
    for c, r0 in enumerate(range(0, M, chunk)):
        b = c % 2
        n = min(M, r0 + chunk) - r0
        if c >= 2:
            s_in.wait_event(done[b])                  # the kernels reading d_in[b] have run
        with torch.cuda.stream(s_in):
            for d, h in zip(d_in[b], inputs):
                d[:n].copy_(h[r0:r0 + n], non_blocking=True)
            in_ready[b].record(s_in)
        comp.wait_event(in_ready[b])
        if c >= 2:
            comp.wait_event(copied[b])                # d_out[b] has been copied back
        call([d[:n] for d in d_in[b]], [d[:n] for d in d_out[b]])
        done[b].record(comp)
        s_out.wait_event(done[b])
        with torch.cuda.stream(s_out):
            for h, d in zip(outputs, d_out[b]):
                h[r0:r0 + n].copy_(d[:n], non_blocking=True)
            copied[b].record(s_out)
    if wait:
        comp.wait_stream(s_out)
    comp.wait_stream(s_in)
    # keep the staging buffers alive until the queued work has used them
    for bufs in d_in + d_out:
        for t in bufs:
            t.record_stream(s_in)
            t.record_stream(s_out)
