"""ln_bwd_noalloc, the LayerNorm backward that allocates nothing (its
scratch is a fixed static device array), called through the C ABI and
checked against the existing ln_bwd on two calls in a row, within the
backward tolerances the other tests use. Collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import row_wise_normalization_ln_gb300 as rn

from parity import as_f64, check_ln_bwd, ln_stats_f32, np_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from row_wise_normalization_ln_gb300 import _build
    _build.build()
    L = rn.library()
    vp = ctypes.c_void_p
    L.ln_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, vp]
    L.ln_bwd_noalloc.restype = ctypes.c_int
    return L


def _column_bounds(dy, x, gamma, eps):
    """The column-gradient bounds of tests/parity.py for these inputs."""
    dyn, xn, gn = np_of(dy), np_of(x), np_of(gamma)
    M = xn.shape[0]
    _, mean, rstd = oracle.ln_fwd(xn, gn, gn, oracle.eps_as_f32(eps))
    x64, dy64 = as_f64(xn), as_f64(dyn)
    xh = (x64 - mean[:, None]) * rstd[:, None]
    X = np.abs(xh).max(axis=1) + np.abs(mean) * rstd
    u = 2.0 ** -24
    tol_g = u * ((2 * M + 64) * np.abs(dy64 * xh).sum(axis=0) + 4 * (np.abs(dy64) * X[:, None]).sum(axis=0))
    tol_b = u * (2 * M + 64) * np.abs(dy64).sum(axis=0)
    return tol_g, tol_b


def _case(M, N, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(M, N, generator=g) * 2 + 1).to(dtype)
    dy = torch.randn(M, N, generator=g).to(dtype)
    gamma = (torch.rand(N, generator=g) + 0.5).to(dtype)
    return x, dy, gamma


def test_no_alloc_backward_matches_ln_bwd_twice(lib):
    """Two calls in a row (different shapes and data, so that stale scratch
    from the first would show in the second): dx equal to ln_bwd's, the
    column gradients within the backward bound of ln_bwd's and of the
    oracle. In the first case one partial row per CTA would not fit the
    scratch, so its CTAs add their columns in reduction clusters of 8
    first; the second spans 8-CTA clusters and its grid is capped to the
    scratch."""
    for (M, N, dtype, seed) in ((4096, 8192, torch.bfloat16, 1), (256, 65536, torch.float32, 2)):
        x, dy, gamma = _case(M, N, dtype, seed)
        mean, rstd = ln_stats_f32(x, gamma, 1e-5)
        xd, dyd, gd, md, rd = x.cuda(), dy.cuda(), gamma.cuda(), mean.cuda(), rstd.cuda()
        dx = torch.empty_like(xd)
        dg = torch.full((N,), float("nan"), device="cuda")
        db = torch.full((N,), float("nan"), device="cuda")
        code = rn.NORM_F32 if dtype == torch.float32 else rn.NORM_BF16
        st = lib.ln_bwd_noalloc(dyd.data_ptr(), xd.data_ptr(), gd.data_ptr(), md.data_ptr(), rd.data_ptr(),
                                dx.data_ptr(), dg.data_ptr(), db.data_ptr(), M, N, code,
                                torch.cuda.current_stream().cuda_stream)
        assert st == rn.NORM_OK, lib.norm_status_string(st)
        dx_ref, dg_ref, db_ref = rn.ln_bwd(dyd, xd, gd, md, rd)
        torch.cuda.synchronize()
        assert torch.equal(dx, dx_ref)        # dx does not depend on the grid
        tol_g, tol_b = _column_bounds(dy, x, gamma, 1e-5)
        assert np.all(np.abs(np_of(dg).astype(np.float64) - np_of(dg_ref)) <= tol_g)
        assert np.all(np.abs(np_of(db).astype(np.float64) - np_of(db_ref)) <= tol_b)
        check_ln_bwd(dy, x, gamma, 1e-5, dx, dg, db)


def test_no_alloc_rejects_sizes_beyond_the_limit(lib):
    p = ctypes.c_void_p(0x1000)
    # rows beyond the backward's one-pass limit: refused before any launch
    assert lib.ln_bwd_noalloc(p, p, p, p, p, p, p, p, 4, 65540, rn.NORM_F32, None) == rn.NORM_ERR_ARG
