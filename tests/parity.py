"""Comparison of CUDA results with the fp64 oracle, with the tolerances the
parity tests use.

fp32 outputs: max |y - y_ref| <= 1e-4; rstd relative error <= 1e-5; mean
within 1e-5 of the row's scale, max(|mean_ref|, sigma_ref) (a purely relative
bound is ill-posed for means near zero).

bf16 and fp16 outputs: y within one ulp of the oracle's value rounded to
that type. Near y = 0 an ulp is smaller than the fp32 error of any fp32
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


def ulp_f16(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -14), -14)
    return np.exp2(e - 10)


def round16(y_ref: np.ndarray, like: np.ndarray):
    """The oracle's values rounded to the 16-bit type of `like` (raw bf16
    bits or float16), widened back, with that type's ulp."""
    if like.dtype == np.float16:
        r = oracle.round_f16(y_ref).astype(np.float64)
        return r, ulp_f16(r)
    r = as_f64(oracle.round_bf16(y_ref))
    return r, ulp_bf16(r)


def check_y(y_gpu: np.ndarray, y_ref: np.ndarray, floor_rows: np.ndarray | None = None) -> dict:
    """Compare one block of rows; returns error statistics, asserts the bar."""
    if y_gpu.dtype == np.float32:
        err = np.abs(y_gpu.astype(np.float64) - y_ref)
        worst = float(err.max()) if err.size else 0.0
        assert np.all(np.isfinite(y_gpu)), "non-finite output"
        assert worst <= FP32_Y_ABS, f"max |dy| = {worst:.3e} > {FP32_Y_ABS}"
        return {"max_abs": worst}
    ref_b, ulp = round16(y_ref, y_gpu)
    got = as_f64(y_gpu)
    diff = np.abs(got - ref_b)
    tol = ulp if floor_rows is None else np.maximum(ulp, floor_rows[:, None])
    bad = diff > tol
    assert not bad.any(), (
        f"{int(bad.sum())} 16-bit outputs off by more than 1 ulp (worst {float((diff / ulp).max()):.2f} ulp)")
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
    floor = ln_floor(as_f64(xn), as_f64(gn), as_f64(bn), m_ref, r_ref) if yn.dtype != np.float32 else None
    res = check_y(yn, y_ref, floor)
    res.update(check_stats(mn, rn_, m_ref, r_ref, e))
    return res


def check_rms(x, w, eps, y, rows=None) -> dict:
    xn, wn, yn = np_of(x), np_of(w), np_of(y)
    if rows is not None:
        xn, yn = xn[rows], yn[rows]
    e = oracle.eps_as_f32(eps)
    y_ref, r_ref = oracle.rms_fwd(xn, wn, e)
    floor = rms_floor(as_f64(xn), as_f64(wn), r_ref) if yn.dtype != np.float32 else None
    return check_y(yn, y_ref, floor)


def torch_of(a: np.ndarray) -> torch.Tensor:
    """Inverse of np_of: CPU tensor from float32, float16 or raw bf16
    (uint16) bits."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
    if a.dtype == np.float16:
        return torch.from_numpy(a.copy())
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))


def check_h(x, r, h, rows=None) -> torch.Tensor:
    """h of the fused add against the oracle's rounded sum, bit for bit;
    returns the oracle's h (CPU tensor, the selected rows)."""
    xn, rn_, hn = np_of(x), np_of(r), np_of(h)
    if rows is not None:
        xn, rn_, hn = xn[rows], rn_[rows], hn[rows]
    h_ref = oracle.add_round(xn, rn_)
    bits = np.uint16 if h_ref.dtype.itemsize == 2 else np.uint32
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


# ---------------------------------------------------------------- backward
#
# dx (per row, u = 2^-24). The kernel forms the two row sums in fp32 with
# at most 64 sequential additions on any path (per-thread runs of <= 32
# elements, then <= 12 tree levels), so each sum is off by <= 64u of the sum
# of its absolute terms; xhat is formed from the fp32 mean and rstd, off by
# <= 2u (|xhat| + |mean| rstd). Propagating through
# dx = rstd (g - gbar - xhat * gxbar), with G = max|g|, X = max|xhat| +
# |mean| rstd, bounds the error by about u rstd G (67 + 68 X^2); the tests
# allow twice that: 2^-17 rstd G (1 + X^2).
# RMSNorm: dx = r w dy - x r^3 S / N with r from a sum of squares (<= 36u
# relative after rsqrt) and S off by <= 64u sum|g x|: <= 36u r G + 166u
# max|x| r^3 mean|g x|; allowed 2^-17 r G + 2^-15 max|x| r^3 mean|g x|.
# bf16 dx: one bf16 ulp of the rounded oracle value, or the fp32 bound.
# Column gradients: a sum over rows in fp32 along a chain of at most
# rows-per-CTA + 8 + partial-rows <= 2M + 8 additions: allowed
# 2^-24 (2M + 64) sum|terms| (+ the xhat error of each term for dgamma, and
# the rstd error for dw).

def _dx_check(dx_gpu: np.ndarray, dx_ref: np.ndarray, tol_rows: np.ndarray) -> dict:
    if dx_gpu.dtype == np.float32:
        err = np.abs(dx_gpu.astype(np.float64) - dx_ref)
        assert np.all(np.isfinite(dx_gpu)), "non-finite dx"
        ratio = err / tol_rows[:, None]
        assert (ratio <= 1).all(), f"dx off by {float(ratio.max()):.2f} x the bound"
        return {"dx_worst_of_bound": float(ratio.max()) if ratio.size else 0.0}
    ref_b, ulp = round16(dx_ref, dx_gpu)
    diff = np.abs(as_f64(dx_gpu) - ref_b)
    bad = diff > np.maximum(ulp, tol_rows[:, None])
    assert not bad.any(), f"{int(bad.sum())} 16-bit dx off by more than 1 ulp and the fp32 bound"
    return {"dx_exact": int((diff == 0).sum()), "dx_n": int(diff.size)}


def _col_check(got: np.ndarray, ref: np.ndarray, tol: np.ndarray, name: str) -> float:
    err = np.abs(got.astype(np.float64) - ref)
    ratio = err / np.where(tol > 0, tol, 1e-300)
    assert (err <= tol).all(), f"{name} off by {float(ratio.max()):.2f} x the bound"
    return float(ratio.max()) if ratio.size else 0.0


def check_ln_bwd(dy, x, gamma, eps, dx, dgamma, dbeta, rows=None) -> dict:
    """dy, x, gamma: CPU tensors given to the kernel (with the forward's
    statistics for `eps`); dx, dgamma, dbeta: its outputs. The column
    gradients are checked over all rows; `rows` restricts the dx check."""
    dyn, xn, gn = np_of(dy), np_of(x), np_of(gamma)
    M, N = xn.shape
    e = oracle.eps_as_f32(eps)
    dx_ref, dg_ref, db_ref = oracle.ln_bwd(dyn, xn, gn, e)
    _, mean, rstd = oracle.ln_fwd(xn, gn, gn, e)
    x64, dy64, g64 = as_f64(xn), as_f64(dyn), as_f64(gn)
    xh = (x64 - mean[:, None]) * rstd[:, None]
    X = np.abs(xh).max(axis=1) + np.abs(mean) * rstd
    G = np.abs(dy64 * g64[None, :]).max(axis=1)
    tol_rows = 2.0 ** -17 * rstd * G * (1 + X * X)
    dxn = np_of(dx)
    if rows is not None:
        dxn, dx_ref, tol_rows = dxn[rows], dx_ref[rows], tol_rows[rows]
    res = _dx_check(dxn, dx_ref, tol_rows)
    u = 2.0 ** -24
    tol_g = u * ((2 * M + 64) * np.abs(dy64 * xh).sum(axis=0) + 4 * (np.abs(dy64) * X[:, None]).sum(axis=0))
    tol_b = u * (2 * M + 64) * np.abs(dy64).sum(axis=0)
    res["dgamma_worst_of_bound"] = _col_check(np_of(dgamma), dg_ref, tol_g, "dgamma")
    res["dbeta_worst_of_bound"] = _col_check(np_of(dbeta), db_ref, tol_b, "dbeta")
    return res


def ln_stats_f32(x, gamma, eps):
    """The oracle's mean and rstd of each row, rounded to fp32 (CPU tensors),
    as inputs for the backward."""
    _, mean, rstd = oracle.ln_fwd(np_of(x), np_of(gamma), np_of(gamma), oracle.eps_as_f32(eps))
    return torch.from_numpy(oracle.round_f32(mean)), torch.from_numpy(oracle.round_f32(rstd))


def check_rms_bwd(dy, x, w, eps, dx, dw, rows=None) -> dict:
    dyn, xn, wn = np_of(dy), np_of(x), np_of(w)
    M, N = xn.shape
    e = oracle.eps_as_f32(eps)
    dx_ref, dw_ref = oracle.rms_bwd(dyn, xn, wn, e)
    _, r = oracle.rms_fwd(xn, wn, e)
    x64, dy64, w64 = as_f64(xn), as_f64(dyn), as_f64(wn)
    g = dy64 * w64[None, :]
    G = np.abs(g).max(axis=1)
    tol_rows = 2.0 ** -17 * r * G + 2.0 ** -15 * np.abs(x64).max(axis=1) * r ** 3 * np.abs(g * x64).mean(axis=1)
    dxn = np_of(dx)
    if rows is not None:
        dxn, dx_ref, tol_rows = dxn[rows], dx_ref[rows], tol_rows[rows]
    res = _dx_check(dxn, dx_ref, tol_rows)
    tol_w = 2.0 ** -24 * (2 * M + 128) * np.abs(dy64 * x64 * r[:, None]).sum(axis=0)
    res["dw_worst_of_bound"] = _col_check(np_of(dw), dw_ref, tol_w, "dw")
    return res


# ---------------------------------------------------------------- FP8 output
#
# The kernel forms y in fp32 and quantises y * (1/scale); the oracle
# quantises the exact y / scale. An integer code is decided by floating
# point, so the codes agree except where the exact value lies within the
# kernel's fp32 error of a rounding boundary. The bar: the decoded code is
# within half an E4M3 ulp of v = y / scale plus that slack (the fp32 floor
# of y above, over the scale, plus 2^-21 |v| for the inverse scale and the
# product), and magnitudes beyond 448 + slack give exactly +-448.

E4M3_MAX = 448.0


def ulp_e4m3(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.where(a > 0, np.maximum(e, -6), -6)
    return np.exp2(e - 3)


def check_fp8(q_gpu: np.ndarray, y_ref: np.ndarray, scale: float, floor_rows: np.ndarray) -> dict:
    v = y_ref / scale
    d = oracle.e4m3_values(q_gpu)
    assert not np.isnan(d).any(), "NaN code"
    slack = floor_rows[:, None] / scale + 2.0 ** -21 * np.abs(v)
    sat = np.abs(v) >= E4M3_MAX + slack
    assert np.all(d[sat] == np.sign(v[sat]) * E4M3_MAX), "saturated values must give +-448"
    err = np.abs(d - v)
    bound = 0.5 * ulp_e4m3(np.minimum(np.abs(v), E4M3_MAX)) + slack
    bad = ~sat & (err > bound)
    assert not bad.any(), f"{int(bad.sum())} FP8 codes farther than half an ulp (+ slack) from y / scale"
    q_ref = oracle.quant_e4m3(y_ref, scale)
    return {"codes_equal": int((q_gpu == q_ref).sum()), "n": int(q_gpu.size), "saturated": int(sat.sum())}


def check_ln_fp8(x, gamma, beta, eps, scale, y8, mean=None, rstd=None, rows=None) -> dict:
    xn, gn, bn = np_of(x), np_of(gamma), np_of(beta)
    qn = y8.detach().cpu().contiguous().numpy().view(np.uint8)
    mn = np_of(mean) if mean is not None else None
    rn_ = np_of(rstd) if rstd is not None else None
    if rows is not None:
        xn, qn = xn[rows], qn[rows]
        mn = mn[rows] if mn is not None else None
        rn_ = rn_[rows] if rn_ is not None else None
    e = oracle.eps_as_f32(eps)
    y_ref, m_ref, r_ref = oracle.ln_fwd(xn, gn, bn, e)
    floor = ln_floor(as_f64(xn), as_f64(gn), as_f64(bn), m_ref, r_ref)
    res = check_fp8(qn, y_ref, scale, floor)
    res.update(check_stats(mn, rn_, m_ref, r_ref, e))
    return res


def check_rms_fp8(x, w, eps, scale, y8, rows=None) -> dict:
    xn, wn = np_of(x), np_of(w)
    qn = y8.detach().cpu().contiguous().numpy().view(np.uint8)
    if rows is not None:
        xn, qn = xn[rows], qn[rows]
    e = oracle.eps_as_f32(eps)
    y_ref, r_ref = oracle.rms_fwd(xn, wn, e)
    return check_fp8(qn, y_ref, scale, rms_floor(as_f64(xn), as_f64(wn), r_ref))
