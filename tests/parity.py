"""Comparison of CUDA results with the fp64 oracle, with the tolerances the
parity tests use.

fp32 outputs: max |y - y_ref| <= 1e-4; rstd relative error <= 1e-5; mean
within 1e-5 of the row's scale, max(|mean_ref|, sigma_ref) (a purely relative
bound is ill-posed for means near zero).

bf16 outputs: y within one bf16 ulp of the oracle's value rounded to bf16.
Near y = 0 a bf16 ulp is smaller than the fp32 error of any fp32
evaluation, so each row also gets an absolute floor from the fp32 error
budget of y = (x - mean) * rstd * gamma + beta:
    2^-21 * ((|mean| * rstd + max|x_hat|) * max|gamma| + max|beta|)
(eight fp32 ulps of every term that enters y, including the rounding of the
fp32 mean itself). For RMSNorm the floor is 2^-21 * max|x| * rstd * max|w|.

Fused residual add: h = x + r must match the oracle's correctly rounded sum
bit for bit (one IEEE addition in either dtype); y and the statistics are
then held to the bars above against the oracle's norm of that h.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

FP32_Y_ABS = 1e-4
STAT_REL = 1e-5


def np_of(t: torch.Tensor) -> np.ndarray:
    """CPU numpy view: fp32 as float32, bf16 as raw uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def as_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -126), -126)
    return np.exp2(e - 7)


def check_y(y_gpu: np.ndarray, y_ref: np.ndarray, floor_rows: np.ndarray | None = None) -> dict:
    """Compare one block of rows; returns error statistics, asserts the bar."""
    if y_gpu.dtype == np.float32:
        err = np.abs(y_gpu.astype(np.float64) - y_ref)
        worst = float(err.max()) if err.size else 0.0
        assert np.all(np.isfinite(y_gpu)), "non-finite output"
        assert worst <= FP32_Y_ABS, f"max |dy| = {worst:.3e} > {FP32_Y_ABS}"
        return {"max_abs": worst}
    ref_b = as_f64(oracle.round_bf16(y_ref))
    got = as_f64(y_gpu)
    diff = np.abs(got - ref_b)
    ulp = ulp_bf16(ref_b)
    tol = ulp if floor_rows is None else np.maximum(ulp, floor_rows[:, None])
    bad = diff > tol
    assert not bad.any(), (
        f"{int(bad.sum())} bf16 outputs off by more than 1 ulp (worst {float((diff / ulp).max()):.2f} ulp)")
    return {"exact": int((diff == 0).sum()), "one_ulp": int(((diff > 0) & (diff <= ulp)).sum()),
            "floor_only": int(((diff > ulp) & ~bad).sum()), "n": int(diff.size)}


def check_stats(mean_gpu, rstd_gpu, mean_ref, rstd_ref, eps: float) -> dict:
    out = {}
    if rstd_gpu is not None:
        rel = np.abs(rstd_gpu.astype(np.float64) - rstd_ref) / rstd_ref
        out["rstd_rel"] = float(rel.max()) if rel.size else 0.0
        assert out["rstd_rel"] <= STAT_REL, f"rstd rel err {out['rstd_rel']:.3e}"
    if mean_gpu is not None:
        sigma = np.sqrt(np.maximum(1.0 / rstd_ref ** 2 - eps, 0.0))
        scale = np.maximum(np.abs(mean_ref), sigma)
        err = np.abs(mean_gpu.astype(np.float64) - mean_ref)
        ok = err <= STAT_REL * scale
        out["mean_scaled"] = float((err / np.where(scale > 0, scale, 1)).max()) if err.size else 0.0
        assert ok.all(), f"mean err {out['mean_scaled']:.3e} of the row scale"
    return out


def ln_floor(x64, g64, b64, mean, rstd):
    xhat = np.abs(x64 - mean[:, None]) * rstd[:, None]
    return 2.0 ** -21 * ((np.abs(mean) * rstd + xhat.max(axis=1)) * np.abs(g64).max() + np.abs(b64).max())


def rms_floor(x64, w64, rstd):
    return 2.0 ** -21 * np.abs(x64).max(axis=1) * rstd * np.abs(w64).max()


def check_ln(x, gamma, beta, eps, y, mean=None, rstd=None, rows=None) -> dict:
    """x, gamma, beta: CPU tensors given to the kernel; y, mean, rstd: its
    outputs (any device). `rows` restricts the comparison to those rows."""
    xn, gn, bn = np_of(x), np_of(gamma), np_of(beta)
    yn = np_of(y)
    mn = np_of(mean) if mean is not None else None
    rn_ = np_of(rstd) if rstd is not None else None
    if rows is not None:
        xn, yn = xn[rows], yn[rows]
        mn = mn[rows] if mn is not None else None
        rn_ = rn_[rows] if rn_ is not None else None
    e = oracle.eps_as_f32(eps)
    y_ref, m_ref, r_ref = oracle.ln_fwd(xn, gn, bn, e)
    floor = ln_floor(as_f64(xn), as_f64(gn), as_f64(bn), m_ref, r_ref) if yn.dtype == np.uint16 else None
    res = check_y(yn, y_ref, floor)
    res.update(check_stats(mn, rn_, m_ref, r_ref, e))
    return res


def check_rms(x, w, eps, y, rows=None) -> dict:
    xn, wn, yn = np_of(x), np_of(w), np_of(y)
    if rows is not None:
        xn, yn = xn[rows], yn[rows]
    e = oracle.eps_as_f32(eps)
    y_ref, r_ref = oracle.rms_fwd(xn, wn, e)
    floor = rms_floor(as_f64(xn), as_f64(wn), r_ref) if yn.dtype == np.uint16 else None
    return check_y(yn, y_ref, floor)


def torch_of(a: np.ndarray) -> torch.Tensor:
    """Inverse of np_of: CPU tensor from float32 or raw bf16 (uint16) bits."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))


def check_h(x, r, h, rows=None) -> torch.Tensor:
    """h of the fused add against the oracle's rounded sum, bit for bit;
    returns the oracle's h (CPU tensor, the selected rows)."""
    xn, rn_, hn = np_of(x), np_of(r), np_of(h)
    if rows is not None:
        xn, rn_, hn = xn[rows], rn_[rows], hn[rows]
    h_ref = oracle.add_round(xn, rn_)
    bits = np.uint16 if h_ref.dtype == np.uint16 else np.uint32
    bad = hn.view(bits) != h_ref.view(bits)
    assert not bad.any(), f"{int(bad.sum())} elements of h differ from the rounded sum"
    return torch_of(h_ref)


def check_ln_add(x, r, gamma, beta, eps, h, y, mean=None, rstd=None, rows=None) -> dict:
    h_ref = check_h(x, r, h, rows)
    if rows is not None:
        y = np_of(y)[rows]
        mean = np_of(mean)[rows] if mean is not None else None
        rstd = np_of(rstd)[rows] if rstd is not None else None
    return check_ln(h_ref, gamma, beta, eps, _t(y), _t(mean), _t(rstd))


def check_rms_add(x, r, w, eps, h, y, rows=None) -> dict:
    h_ref = check_h(x, r, h, rows)
    if rows is not None:
        y = np_of(y)[rows]
    return check_rms(h_ref, w, eps, _t(y))


def _t(a):
    return torch_of(a) if isinstance(a, np.ndarray) else a


def sample_rows(M: int, k: int = 48, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(M, size=min(k, M), replace=False).tolist()) | {0, M - 1}
    return np.array(sorted(pick))
