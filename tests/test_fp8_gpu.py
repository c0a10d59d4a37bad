"""GPU parity of the FP8 (E4M3) output of the norm ("第 7 章 LayerNorm 与
RMSNorm" §7.9: the norm writes the next GEMM's quantised input, as vLLM's
static-scale fused kernels do), plain and with the fused residual add, on
fp32, bf16 and fp16 rows, through the C ABI (via the Python binding),
against the fp64 oracle (the bar in tests/parity.py), and bit for bit
against torch's quantisation of the library's own fp32 output."""
import numpy as np
import pytest
import torch

import row_wise_normalization_ln_gb300 as rn
from row_wise_normalization_ln_gb300 import workloads as wl

from parity import check_h, check_ln_fp8, check_rms_fp8, sample_rows

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from row_wise_normalization_ln_gb300 import _build
    _build.build()
    rn.library()


def _rand(M, N, dtype, seed, loc=0.0, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(M, N, generator=g) * scale + loc).to(dtype)
    r = torch.randn(M, N, generator=g).to(dtype)
    gamma = (torch.rand(N, generator=g) + 0.5).to(dtype)
    beta = (torch.rand(N, generator=g) * 0.2 - 0.1).to(dtype)
    return x, r, gamma, beta


def _both(x, g, b, scale, plan=None):
    xd, gd, bd = x.cuda(), g.cuda(), b.cuda()
    y8, mean, rstd = rn.ln_fwd_fp8(xd, gd, bd, scale, 1e-5, plan=plan)
    torch.cuda.synchronize()
    r1 = check_ln_fp8(x, g, b, 1e-5, scale, y8, mean, rstd)
    y8 = rn.rms_fwd_fp8(xd, gd, scale, 1e-6, plan=plan)
    torch.cuda.synchronize()
    r2 = check_rms_fp8(x, g, 1e-6, scale, y8)
    return r1, r2


# ------------------------------------------------------------ the workloads

FP8 = [n for n, w in wl.WORKLOADS.items() if w.fp8]


@pytest.mark.parametrize("name", FP8)
def test_workload_full_size(name):
    """The full-size launch as benchmarked: sampled rows code by code (and h
    of the fused add everywhere)."""
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, seed=0)
    rows = sample_rows(w.M, 40)
    x = inp["x"].cuda()
    if w.op == "ln":
        y8, mean, rstd = rn.ln_fwd_fp8(x, inp["gamma"].cuda(), inp["beta"].cuda(), w.qscale, w.eps)
        torch.cuda.synchronize()
        res = check_ln_fp8(inp["x"], inp["gamma"], inp["beta"], w.eps, w.qscale, y8, mean, rstd, rows=rows)
    elif w.add:
        h, y8 = rn.rms_fwd_fp8(x, inp["w"].cuda(), w.qscale, w.eps, residual=inp["r"].cuda())
        torch.cuda.synchronize()
        hr = check_h(inp["x"], inp["r"], h)
        res = check_rms_fp8(hr, inp["w"], w.eps, w.qscale, y8, rows=rows)
    else:
        y8 = rn.rms_fwd_fp8(x, inp["w"].cuda(), w.qscale, w.eps)
        torch.cuda.synchronize()
        res = check_rms_fp8(inp["x"], inp["w"], w.eps, w.qscale, y8, rows=rows)
    assert res["codes_equal"] >= 0.999 * res["n"], res


# ------------------------------------------------------------ shapes and variants

EDGE_N = [1, 2, 3, 5, 8, 31, 33, 127, 129, 257, 1000, 1024, 4096, 5000, 8193, 65536, 100003]


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", EDGE_N)
def test_edge_widths(dtype, N):
    x, _, g, b = _rand(4 if N < 60000 else 2, N, DT[dtype], seed=N, loc=1.0, scale=2.0)
    _both(x, g, b, 4.0 / 448)


def _variants():
    out = []
    for dtype, vec in (("f32", 4), ("bf16", 8)):
        for ve in (vec, 1):
            for G, per in ((1, 1), (4, 2), (32, 8)):
                out.append((dtype, dict(mapping=rn.NORM_MAP_GROUP, vec_elems=ve, per_thread=per, group=G,
                                        threads=256 if G < 32 else 128, cluster=1, grid=3)))
            for C in (1, 2, 8):
                for T in (32, 256):
                    for per in (1, 4, 8):
                        out.append((dtype, dict(mapping=rn.NORM_MAP_CTA, vec_elems=ve, per_thread=per, group=0,
                                                threads=T, cluster=C, grid=C * 3)))
    return out


VARIANTS = _variants()


@pytest.mark.parametrize("dtype,plan", VARIANTS, ids=[f"{d}-m{p['mapping']}-v{p['vec_elems']}-p{p['per_thread']}"
                                                      f"-g{p['group']}-t{p['threads']}-c{p['cluster']}"
                                                      for d, p in VARIANTS])
def test_every_variant(dtype, plan):
    """Explicit plans, an exact row and, for the CTA mapping, three rounds;
    also the fused add under the same plan."""
    ve = plan["vec_elems"]
    if plan["mapping"] == rn.NORM_MAP_GROUP:
        sizes = [plan["group"] * plan["per_thread"] * ve]
    else:
        cap = plan["cluster"] * plan["threads"] * plan["per_thread"] * ve
        sizes = [cap, 2 * cap + 3 * ve]
    for N in sizes:
        x, r, g, b = _rand(7, N, DT[dtype], seed=N, loc=-1.0, scale=3.0)
        _both(x, g, b, 8.0 / 448, plan=plan)
        h, y8 = rn.rms_fwd_fp8(x.cuda(), g.cuda(), 8.0 / 448, 1e-6, residual=r.cuda(), plan=plan)
        torch.cuda.synchronize()
        check_rms_fp8(check_h(x, r, h), g, 1e-6, 8.0 / 448, y8)


def test_saturation():
    """A scale so small that most values pass 448: those give exactly +-448."""
    x, _, g, b = _rand(16, 4096, torch.bfloat16, seed=7, scale=3.0)
    r1, r2 = _both(x, g, b, 1.0 / 448)
    assert r1["saturated"] > 0 and r2["saturated"] > 0


def test_scale_on_the_device_and_fused_add_in_place():
    x, r, g, b = _rand(33, 4096, torch.float16, seed=9, loc=0.5)
    sc = torch.tensor([3.0 / 448], device="cuda")
    xd, rd = x.cuda(), r.cuda()
    h, y8, mean, rstd = rn.ln_fwd_fp8(xd, g.cuda(), b.cuda(), sc, 1e-5, residual=rd, h_out=rd)
    torch.cuda.synchronize()
    assert h.data_ptr() == rd.data_ptr()
    check_ln_fp8(check_h(x, r, h), g, b, 1e-5, 3.0 / 448, y8, mean, rstd)


@pytest.mark.parametrize("op", ["ln", "rms"])
def test_equals_quantising_the_fp32_output(op):
    """fp32 rows: the FP8 output is exactly torch's E4M3 cast of the
    library's own fp32 output times the fp32 inverse scale, clamped to 448
    (the same fp32 value through the same nearest-even rounding)."""
    x, _, g, b = _rand(257, 5000, torch.float32, seed=11, loc=2.0, scale=2.0)
    scale = 5.0 / 448
    xd, gd, bd = x.cuda(), g.cuda(), b.cuda()
    if op == "ln":
        y, _, _ = rn.ln_fwd(xd, gd, bd, 1e-5)
        y8, _, _ = rn.ln_fwd_fp8(xd, gd, bd, scale, 1e-5)
    else:
        y = rn.rms_fwd(xd, gd, 1e-6)
        y8 = rn.rms_fwd_fp8(xd, gd, scale, 1e-6)
    inv = torch.tensor(1.0, device="cuda") / torch.tensor(scale, dtype=torch.float32, device="cuda")
    ref = (y * inv).clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(y8, ref)
