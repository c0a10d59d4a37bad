"""GPU parity of fp16 rows on every path (forward, fused residual add,
backward), through the C ABI (via the Python binding), against the fp64
oracle: 16-bit outputs within one fp16 ulp of the oracle rounded to fp16
(with the fp32 floor of tests/parity.py), h of the fused add bit for bit."""
import numpy as np
import pytest
import torch

import row_wise_normalization_ln_gb300 as rn
from row_wise_normalization_ln_gb300 import workloads as wl

from parity import (check_ln, check_ln_add, check_ln_bwd, check_rms, check_rms_add, check_rms_bwd, ln_stats_f32,
                    sample_rows)

pytestmark = pytest.mark.gpu
F16 = torch.float16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from row_wise_normalization_ln_gb300 import _build
    _build.build()
    rn.library()


def _rand(M, N, seed, loc=0.0, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(M, N, generator=g) * scale + loc).to(F16)
    r = torch.randn(M, N, generator=g).to(F16)
    gamma = (torch.rand(N, generator=g) + 0.5).to(F16)
    beta = (torch.rand(N, generator=g) * 0.2 - 0.1).to(F16)
    return x, r, gamma, beta


def _all_paths(x, r, g, b, plan=None, plan_add=None, plan_bwd_ln=None, plan_bwd_rms=None):
    xd, rd, gd, bd = x.cuda(), r.cuda(), g.cuda(), b.cuda()
    y, mean, rstd = rn.ln_fwd(xd, gd, bd, 1e-5, plan=plan)
    torch.cuda.synchronize()
    check_ln(x, g, b, 1e-5, y, mean, rstd)
    y = rn.rms_fwd(xd, gd, 1e-6, plan=plan)
    torch.cuda.synchronize()
    check_rms(x, g, 1e-6, y)
    h, y, mean, rstd = rn.ln_fwd_add(xd, rd, gd, bd, 1e-5, plan=plan_add)
    torch.cuda.synchronize()
    check_ln_add(x, r, g, b, 1e-5, h, y, mean, rstd)
    h, y = rn.rms_fwd_add(xd, rd, gd, 1e-6, plan=plan_add)
    torch.cuda.synchronize()
    check_rms_add(x, r, g, 1e-6, h, y)
    if x.shape[1] <= 65536:
        m32, r32 = ln_stats_f32(x, g, 1e-5)
        dx, dg, db = rn.ln_bwd(rd, xd, gd, m32.cuda(), r32.cuda(), plan=plan_bwd_ln)
        torch.cuda.synchronize()
        check_ln_bwd(r, x, g, 1e-5, dx, dg, db)
        dx, dw = rn.rms_bwd(rd, xd, gd, 1e-6, plan=plan_bwd_rms)
        torch.cuda.synchronize()
        check_rms_bwd(r, x, g, 1e-6, dx, dw)


EDGE_N = [1, 2, 3, 5, 7, 8, 9, 31, 33, 63, 64, 65, 127, 129, 255, 257, 1000, 1023, 1025, 4095, 4096, 5000, 8191,
          8192, 16385, 32768, 65536, 100003]


@pytest.mark.parametrize("N", EDGE_N)
def test_edge_widths(N):
    x, r, g, b = _rand(5 if N < 60000 else 2, N, seed=N, loc=2.0, scale=3.0)
    _all_paths(x, r, g, b)


@pytest.mark.parametrize("M", [1, 3, 33, 257, 1000])
def test_ragged_row_counts(M):
    for N in (64, 2048, 1000):
        x, r, g, b = _rand(M, N, seed=M + N)
        _all_paths(x, r, g, b)


def _fwd_variants():
    out = []
    for v in (True, False):
        ve = 8 if v else 1
        for G in (1, 4, 32):
            for per in (1, 8):
                out.append(dict(mapping=rn.NORM_MAP_GROUP, vec_elems=ve, per_thread=per, group=G,
                                threads=256 if G < 32 else 128, cluster=1, grid=3))
        for C in (1, 2, 8):
            for T in (32, 256):
                for per in (1, 2, 4, 8):
                    out.append(dict(mapping=rn.NORM_MAP_CTA, vec_elems=ve, per_thread=per, group=0, threads=T,
                                    cluster=C, grid=C * 3))
    return out


FWD = _fwd_variants()


@pytest.mark.parametrize("plan", FWD, ids=[f"m{p['mapping']}-v{p['vec_elems']}-p{p['per_thread']}-g{p['group']}"
                                           f"-t{p['threads']}-c{p['cluster']}" for p in FWD])
def test_forward_variants(plan):
    """Explicit forward plans (plain and fused add; the fused CTAs are at
    most 512 threads): an exact and a ragged row, and three rounds."""
    if plan["mapping"] == rn.NORM_MAP_GROUP:
        cap = plan["group"] * plan["per_thread"] * plan["vec_elems"]
        sizes = sorted({cap, max(plan["vec_elems"], cap - plan["vec_elems"])})
    else:
        cap = plan["cluster"] * plan["threads"] * plan["per_thread"] * plan["vec_elems"]
        sizes = sorted({cap, max(plan["vec_elems"], cap - 3 * plan["vec_elems"]), 2 * cap + 5 * plan["vec_elems"]})
    for N in sizes:
        x, r, g, b = _rand(7, N, seed=N, loc=-1.0, scale=2.0)
        xd, rd, gd, bd = x.cuda(), r.cuda(), g.cuda(), b.cuda()
        y, mean, rstd = rn.ln_fwd(xd, gd, bd, 1e-5, plan=plan)
        torch.cuda.synchronize()
        check_ln(x, g, b, 1e-5, y, mean, rstd)
        y = rn.rms_fwd(xd, gd, 1e-6, plan=plan)
        torch.cuda.synchronize()
        check_rms(x, g, 1e-6, y)
        h, y = rn.rms_fwd_add(xd, rd, gd, 1e-6, plan=plan)
        torch.cuda.synchronize()
        check_rms_add(x, r, g, 1e-6, h, y)


def _bwd_variants():
    out = []
    for ve in (8, 1):
        for ln in (True, False):
            vmax = 8 if ve == 1 else (2 if ln else 4)
            for per in (1, 2, 4, 8):
                if per > vmax:
                    continue
                for T, C, Q in ((32, 1, 1), (96, 1, 2), (512, 1, 8), (96, 2, 2), (512, 8, 8)):
                    out.append((ln, dict(mapping=rn.NORM_MAP_CTA, vec_elems=ve, per_thread=per, group=Q, threads=T,
                                         cluster=C, grid=2 * Q)))
    return out


BWD = _bwd_variants()


@pytest.mark.parametrize("ln,plan", BWD, ids=[f"{'ln' if ln else 'rms'}-v{p['vec_elems']}-p{p['per_thread']}"
                                              f"-t{p['threads']}-c{p['cluster']}-q{p['group']}" for ln, p in BWD])
def test_backward_variants(ln, plan):
    cap = plan["cluster"] * plan["threads"] * plan["per_thread"] * plan["vec_elems"]
    for N in sorted({cap, max(plan["vec_elems"], cap - 3 * plan["vec_elems"])}):
        x, dy, g, _ = _rand(11, N, seed=N + 1, loc=1.0, scale=2.0)
        if ln:
            m32, r32 = ln_stats_f32(x, g, 1e-5)
            dx, dg, db = rn.ln_bwd(dy.cuda(), x.cuda(), g.cuda(), m32.cuda(), r32.cuda(), plan=plan)
            torch.cuda.synchronize()
            check_ln_bwd(dy, x, g, 1e-5, dx, dg, db)
        else:
            dx, dw = rn.rms_bwd(dy.cuda(), x.cuda(), g.cuda(), 1e-6, plan=plan)
            torch.cuda.synchronize()
            check_rms_bwd(dy, x, g, 1e-6, dx, dw)


def test_workload_full_size():
    """The fp16 benchmark workload at full size, as benchmarked: sampled rows
    element by element, every row's statistics."""
    w = wl.WORKLOADS["ln_f16_4096x8192"]
    inp = wl.generate(w, seed=0)
    y, mean, rstd = rn.ln_fwd(inp["x"].cuda(), inp["gamma"].cuda(), inp["beta"].cuda(), w.eps)
    torch.cuda.synchronize()
    rows = sample_rows(w.M, 40)
    check_ln(inp["x"], inp["gamma"], inp["beta"], w.eps, y, mean, rstd, rows=rows)


def test_in_place_and_unaligned():
    x, r, g, b = _rand(9, 4096, seed=3, loc=1.0)
    xd, rd = x.cuda(), r.cuda()
    h, y, mean, rstd = rn.ln_fwd_add(xd, rd, g.cuda(), b.cuda(), 1e-5, h_out=rd, out=xd)
    torch.cuda.synchronize()
    check_ln_add(x, r, g, b, 1e-5, h, y, mean, rstd)
    base = torch.randn(2 * 40 * 1000 + 3, device="cuda").to(F16)
    xu = base[1:1 + 40 * 1000].view(40, 1000)           # 2-byte offset: element accesses
    gu = (torch.rand(1001, device="cuda") + 0.5).to(F16)[1:]
    bu = torch.zeros(1001, device="cuda", dtype=F16)[1:]
    y, mean, rstd = rn.ln_fwd(xu, gu, bu, 1e-5)
    torch.cuda.synchronize()
    check_ln(xu.cpu(), gu.cpu(), bu.cpu(), 1e-5, y, mean, rstd)


def test_constant_rows_are_exact():
    for N in (5, 4096, 5000):
        x = torch.full((3, N), 812.5, dtype=F16)
        g = (torch.rand(N, generator=torch.Generator().manual_seed(N)) + 0.5).to(F16)
        b = (torch.rand(N, generator=torch.Generator().manual_seed(N + 1)) - 0.5).to(F16)
        y, mean, rstd = rn.ln_fwd(x.cuda(), g.cuda(), b.cuda(), 1e-5)
        torch.cuda.synchronize()
        assert torch.equal(y.cpu(), b.expand(3, N))
        assert torch.equal(mean.cpu(), torch.full((3,), 812.5))


def test_matches_torch_layer_norm():
    """Cross-check with torch's own fp16 layer_norm on the GPU."""
    x, _, g, b = _rand(256, 3072, seed=5, loc=1.0)
    y, _, _ = rn.ln_fwd(x.cuda(), g.cuda(), b.cuda(), 1e-5)
    ref = torch.nn.functional.layer_norm(x.cuda(), (3072,), g.cuda(), b.cuda(), 1e-5)
    assert (y.float() - ref.float()).abs().max().item() <= 2 * 2.0 ** -10 * max(1.0, ref.float().abs().max().item())
