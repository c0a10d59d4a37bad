"""GPU parity of the backward (ln_bwd, rms_bwd), called through the C ABI
(via the Python binding), against the fp64 oracle ("第 7 章 LayerNorm 与
RMSNorm" §7.7): dx element by element, and the fp32 column gradients, with
the error bounds of tests/parity.py. LayerNorm is given the oracle's mean
and rstd rounded to fp32 (what ln_fwd saves), except where a test chains
the GPU forward into the backward."""
import ctypes

import numpy as np
import pytest
import torch

import row_wise_normalization_ln_gb300 as rn
from row_wise_normalization_ln_gb300 import workloads as wl

from parity import check_ln_bwd, check_rms_bwd, ln_stats_f32, sample_rows

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
    x = torch.randn(M, N, generator=g) * scale + loc
    dy = torch.randn(M, N, generator=g)
    gamma = torch.rand(N, generator=g) + 0.5
    return x.to(dtype), dy.to(dtype), gamma.to(dtype)


def run_ln_bwd(dy, x, gamma, eps, plan=None):
    mean, rstd = ln_stats_f32(x, gamma, eps)
    dx, dg, db = rn.ln_bwd(dy.cuda(), x.cuda(), gamma.cuda(), mean.cuda(), rstd.cuda(), plan=plan)
    torch.cuda.synchronize()
    return dx, dg, db


def run_rms_bwd(dy, x, w, eps, plan=None):
    dx, dw = rn.rms_bwd(dy.cuda(), x.cuda(), w.cuda(), eps, plan=plan)
    torch.cuda.synchronize()
    return dx, dw


def _check_both(x, dy, g, plan_ln=None, plan_rms=None):
    dx, dg, db = run_ln_bwd(dy, x, g, 1e-5, plan=plan_ln)
    check_ln_bwd(dy, x, g, 1e-5, dx, dg, db)
    dx, dw = run_rms_bwd(dy, x, g, 1e-6, plan=plan_rms)
    check_rms_bwd(dy, x, g, 1e-6, dx, dw)


# ------------------------------------------------------------ the workloads

BWD = [n for n, w in wl.WORKLOADS.items() if w.bwd]
SMALL_M = {"bwd_rms_f32_8192x4096": 96, "bwd_ln_bf16_4096x8192_outliers": 64, "bwd_rms_bf16_65536x2048": 517,
           "bwd_ln_f32_8192x5000": 77, "bwd_ln_f32_2048x65536": 11}


def _run_workload(w, inp, plan=None):
    if w.op == "ln":
        dx, dg, db = run_ln_bwd(inp["dy"], inp["x"], inp["gamma"], w.eps, plan=plan)
        return dx, (dg, db)
    dx, dw = run_rms_bwd(inp["dy"], inp["x"], inp["w"], w.eps, plan=plan)
    return dx, (dw,)


@pytest.mark.parametrize("name", BWD)
def test_workload_rows_with_full_size_plan(name):
    """A few rows (same N, same recipe) under the full-size launch's kernel
    variant, with a grid small enough that every CTA walks several rows."""
    w = wl.WORKLOADS[name]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = rn.make_bwd_plan(w.M, w.N, w.torch_dtype, w.op == "ln", True, sms)
    ws = w.scaled(M=SMALL_M[name])
    inp = wl.generate(ws, seed=0)
    plan["grid"] = plan["group"] * max(1, min(plan["grid"] // plan["group"], 3))
    dx, cols = _run_workload(w, inp, plan)
    if w.op == "ln":
        check_ln_bwd(inp["dy"], inp["x"], inp["gamma"], w.eps, dx, *cols)
    else:
        check_rms_bwd(inp["dy"], inp["x"], inp["w"], w.eps, dx, *cols)


@pytest.mark.parametrize("name", BWD)
def test_workload_full_size(name):
    """The full-size launch (default plan, as benchmarked): the column
    gradients over all rows, dx on sampled rows."""
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, seed=0)
    dx, cols = _run_workload(w, inp)
    rows = sample_rows(w.M, 40)
    if w.op == "ln":
        check_ln_bwd(inp["dy"], inp["x"], inp["gamma"], w.eps, dx, *cols, rows=rows)
    else:
        check_rms_bwd(inp["dy"], inp["x"], inp["w"], w.eps, dx, *cols, rows=rows)
    assert torch.isfinite(dx.float()).all()


# ------------------------------------------------------------ shapes

EDGE_N = [1, 2, 3, 5, 8, 31, 33, 127, 128, 129, 257, 1000, 1023, 1025, 4095, 4097, 5000, 8193, 16384, 32768,
          65536]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", EDGE_N)
def test_edge_widths(dtype, N):
    M = 6 if N < 30000 else 3
    x, dy, g = _rand(M, N, DT[dtype], seed=N, loc=1.0, scale=2.0)
    _check_both(x, dy, g)


@pytest.mark.parametrize("M", [1, 2, 7, 8, 9, 100, 1000, 4099])
def test_ragged_row_counts(M):
    """Row counts that leave CTAs of a reduction cluster without rows, and
    grids that walk several rows per CTA."""
    for N, dtype in ((64, torch.float32), (2048, torch.bfloat16), (1000, torch.float32)):
        x, dy, g = _rand(M, N, dtype, seed=M)
        _check_both(x, dy, g)


def test_zero_rows_give_zero_column_gradients():
    x = torch.empty(0, 64, device="cuda")
    g = torch.ones(64, device="cuda")
    e = torch.empty(0, device="cuda")
    dg = torch.full((64,), 7.0, device="cuda")
    db = torch.full((64,), 7.0, device="cuda")
    dx, dg, db = rn.ln_bwd(x, x, g, e, e, dgamma=dg, dbeta=db)
    torch.cuda.synchronize()
    assert dx.shape == (0, 64) and not dg.any() and not db.any()
    dw = torch.full((64,), 7.0, device="cuda")
    _, dw = rn.rms_bwd(x, x, g, dw=dw)
    torch.cuda.synchronize()
    assert not dw.any()


# ------------------------------------------------------------ every variant

def _variants():
    out = []
    for dtype, vec in (("f32", 4), ("bf16", 8)):
        for v in (True, False):
            ve = vec if v else 1
            for ln in (True, False):
                vmax = 8 if ve == 1 else (2 if (ln and dtype == "bf16") else 4)
                for per in (1, 2, 4, 8):
                    if per > vmax:
                        continue
                    for T in (32, 96, 512):
                        for C in (1, 2, 4, 8):
                            cap = C * T * per * ve
                            if cap > 140000:
                                continue
                            groups = (C,) if C > 1 else (1, 2, 8)
                            for Q in groups:
                                for N in sorted({cap, max(ve, cap - 3 * ve)}):
                                    out.append((dtype, ln, dict(mapping=rn.NORM_MAP_CTA, vec_elems=ve, per_thread=per,
                                                                group=Q, threads=T, cluster=C, grid=2 * Q), N))
    return out


VARIANTS = _variants()


@pytest.mark.parametrize("dtype,ln,plan,N", VARIANTS,
                         ids=[f"{d}-{'ln' if ln else 'rms'}-v{p['vec_elems']}-p{p['per_thread']}-t{p['threads']}"
                              f"-c{p['cluster']}-q{p['group']}-N{n}" for d, ln, p, n in VARIANTS])
def test_every_variant(dtype, ln, plan, N):
    """Explicit plans: every (width, accesses per thread, CTA size, row
    cluster, reduction cluster) variant, an exact and a ragged row, with a
    grid of two clusters walking 11 rows."""
    x, dy, g = _rand(11, N, DT[dtype], seed=N + plan["threads"], loc=-1.0, scale=2.0)
    if ln:
        dx, dg, db = run_ln_bwd(dy, x, g, 1e-5, plan=plan)
        check_ln_bwd(dy, x, g, 1e-5, dx, dg, db)
    else:
        dx, dw = run_rms_bwd(dy, x, g, 1e-6, plan=plan)
        check_rms_bwd(dy, x, g, 1e-6, dx, dw)


def _pipe_variants():
    out = []
    for dtype, vec in (("f32", 4), ("bf16", 8), ("f16", 8)):
        for ve in (vec, 1):
            for ln in (True, False):
                vmax = 8 if ve == 1 else (2 if (ln and dtype != "f32") else 4)
                for per in (1, 2, 4, 8):
                    if per > vmax or (dtype == "f16" and ve == 1 and per not in (1, 8)):
                        continue
                    for T in (32, 96, 512):
                        cap = T * per * ve
                        for Q in (1, 2, 8):
                            for N in sorted({cap, max(ve, cap - 3 * ve)}):
                                out.append((dtype, ln, dict(mapping=rn.NORM_MAP_CTA, vec_elems=ve, per_thread=per,
                                                            group=Q, threads=T, cluster=1, stages=1, grid=2 * Q), N))
    return out


PIPE = _pipe_variants()


@pytest.mark.parametrize("dtype,ln,plan,N", PIPE,
                         ids=[f"{d}-{'ln' if ln else 'rms'}-v{p['vec_elems']}-p{p['per_thread']}-t{p['threads']}"
                              f"-q{p['group']}-N{n}" for d, ln, p, n in PIPE])
def test_pipe_variants(dtype, ln, plan, N):
    """The register pipeline (stages 1: a CTA per row, the next row's loads
    in flight while the current one is reduced): every width, accesses per
    thread, CTA size and reduction cluster, exact and ragged rows, and
    grids whose CTAs walk an odd and an even number of rows."""
    x, dy, g = _rand(11, N, DT[dtype], seed=N + plan["threads"] + 1, loc=0.5, scale=2.0)
    if ln:
        dx, dg, db = run_ln_bwd(dy, x, g, 1e-5, plan=plan)
        check_ln_bwd(dy, x, g, 1e-5, dx, dg, db)
    else:
        dx, dw = run_rms_bwd(dy, x, g, 1e-6, plan=plan)
        check_rms_bwd(dy, x, g, 1e-6, dx, dw)
    assert rn.wait_timeouts() == 0


@pytest.mark.parametrize("M", [1, 2, 3, 152, 153, 3001])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_pipe_many_rows(M, dtype):
    """The register pipeline on a persistent grid over up to 3001 rows (each
    row-parity slot and barrier phase reused many times), against the
    backward without the pipeline on the same inputs: dx bit for bit (the
    arithmetic is the same), the column gradients against the oracle."""
    N = 8192 if dtype != "f32" else 4096
    x, dy, g = _rand(M, N, DT[dtype], seed=M, loc=2.0, scale=1.5)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for ln in (True, False):
        base = rn.make_bwd_plan(M, N, DT[dtype], ln, True, sms)
        if base["cluster"] != 1:
            continue
        pipe = dict(base, stages=1)
        plain = dict(base, stages=0)
        if ln:
            dx1, dg, db = run_ln_bwd(dy, x, g, 1e-5, plan=pipe)
            dx0, _, _ = run_ln_bwd(dy, x, g, 1e-5, plan=plain)
            check_ln_bwd(dy, x, g, 1e-5, dx1, dg, db, rows=sample_rows(M, 24))
        else:
            dx1, dw = run_rms_bwd(dy, x, g, 1e-6, plan=pipe)
            dx0, _ = run_rms_bwd(dy, x, g, 1e-6, plan=plain)
            check_rms_bwd(dy, x, g, 1e-6, dx1, dw, rows=sample_rows(M, 24))
        assert torch.equal(dx1.cpu(), dx0.cpu())
    assert rn.wait_timeouts() == 0


# ------------------------------------------------------------ layouts and errors

def _ring_variants():
    out = []
    for dtype, vec in (("f32", 4), ("bf16", 8), ("f16", 8)):
        for ln in (True, False):
            vmax = 2 if (ln and dtype != "f32") else 4
            for per in (1, 2, 4):
                if per > vmax:
                    continue
                for T in (32, 512):
                    for C in (1, 2, 8):
                        cap = C * T * per * vec
                        if cap > 140000:
                            continue
                        Q = C if C > 1 else 2
                        for S in (2, 3):
                            smem = (2 if ln else 1) * T * per * vec * 4 + S * (2 * T * per * 16 + 8)
                            if smem > 225 * 1024:
                                continue
                            for N in sorted({cap, max(vec, cap - 3 * vec)}):
                                out.append((dtype, ln, dict(mapping=rn.NORM_MAP_CTA, vec_elems=vec, per_thread=per,
                                                            group=Q, threads=T, cluster=C, stages=S, grid=2 * Q), N))
    return out


RING = _ring_variants()


@pytest.mark.parametrize("dtype,ln,plan,N", RING,
                         ids=[f"{d}-{'ln' if ln else 'rms'}-p{p['per_thread']}-t{p['threads']}-c{p['cluster']}"
                              f"-s{p['stages']}-N{n}" for d, ln, p, n in RING])
def test_ring_variants(dtype, ln, plan, N):
    """Plans with a shared-memory ring of upcoming rows (bulk copies): an
    exact and a ragged row, two clusters walking 37 rows, so every stage is
    refilled several times. No wait may run out."""
    x, dy, g = _rand(37, N, DT[dtype], seed=N + 3 * plan["threads"] + plan["stages"], loc=0.5, scale=2.0)
    if ln:
        dx, dg, db = run_ln_bwd(dy, x, g, 1e-5, plan=plan)
        check_ln_bwd(dy, x, g, 1e-5, dx, dg, db)
    else:
        dx, dw = run_rms_bwd(dy, x, g, 1e-6, plan=plan)
        check_rms_bwd(dy, x, g, 1e-6, dx, dw)
    assert rn.wait_timeouts() == 0


def test_unaligned_pointers_take_the_element_path():
    N, M = 1000, 37
    base = torch.randn(2 * M * N + 3, device="cuda")
    x = base[1:1 + M * N].view(M, N)
    dy = base[2 + M * N:2 + 2 * M * N].view(M, N)
    g = (torch.rand(N + 1, device="cuda") + 0.5)[1:]
    mean, rstd = ln_stats_f32(x.cpu(), g.cpu(), 1e-5)
    dxb = torch.empty(M * N + 1, device="cuda")[1:].view(M, N)
    dx, dg, db = rn.ln_bwd(dy, x, g, mean.cuda(), rstd.cuda(), dx=dxb)
    torch.cuda.synchronize()
    check_ln_bwd(dy.cpu(), x.cpu(), g.cpu(), 1e-5, dx, dg, db)
    dx, dw = rn.rms_bwd(dy, x, g, 1e-6, dx=dxb)
    torch.cuda.synchronize()
    check_rms_bwd(dy.cpu(), x.cpu(), g.cpu(), 1e-6, dx, dw)


@pytest.mark.parametrize("N", [1000, 4096, 65536])
def test_in_place(N):
    """dx written over dy, and over x (including an 8-CTA cluster row)."""
    x, dy, g = _rand(9, N, torch.float32, seed=N)
    mean, rstd = ln_stats_f32(x, g, 1e-5)
    for over in ("dy", "x"):
        xd, dyd = x.cuda(), dy.cuda()
        target = dyd if over == "dy" else xd
        dx, dg, db = rn.ln_bwd(dyd, xd, g.cuda(), mean.cuda(), rstd.cuda(), dx=target)
        torch.cuda.synchronize()
        assert dx.data_ptr() == target.data_ptr()
        check_ln_bwd(dy, x, g, 1e-5, dx, dg, db)
        xd, dyd = x.cuda(), dy.cuda()
        target = dyd if over == "dy" else xd
        dx, dw = rn.rms_bwd(dyd, xd, g.cuda(), 1e-6, dx=target)
        torch.cuda.synchronize()
        check_rms_bwd(dy, x, g, 1e-6, dx, dw)


def test_smem_limit_survives_smaller_configurations():
    """One kernel (LayerNorm fp32, 4 accesses per thread, ring) launched with
    192 KB of shared memory, then for the first time with 144 KB, then with
    192 KB again: a configuration first seen later must not lower the
    kernel's shared-memory limit below what an earlier one needs."""
    big = dict(mapping=rn.NORM_MAP_CTA, vec_elems=4, per_thread=4, group=8, threads=512, cluster=8, stages=2, grid=16)
    small = dict(mapping=rn.NORM_MAP_CTA, vec_elems=4, per_thread=4, group=2, threads=384, cluster=1, stages=2, grid=4)
    for N, plan in ((65536, big), (6144, small), (65536, big)):
        x, dy, g = _rand(5, N, torch.float32, seed=N)
        dx, dg, db = run_ln_bwd(dy, x, g, 1e-5, plan=plan)
        check_ln_bwd(dy, x, g, 1e-5, dx, dg, db)


def test_deterministic():
    x, dy, g = _rand(3000, 5000, torch.float32, seed=9, loc=3.0)
    mean, rstd = ln_stats_f32(x, g, 1e-5)
    args = (dy.cuda(), x.cuda(), g.cuda(), mean.cuda(), rstd.cuda())
    r1 = rn.ln_bwd(*args)
    r2 = rn.ln_bwd(*args)
    for a, c in zip(r1, r2):
        assert torch.equal(a, c)


def test_host_errors():
    x = torch.randn(4, 64, device="cuda")
    g = torch.ones(64, device="cuda")
    st = torch.ones(4, device="cuda")
    small = torch.empty(1, device="cuda")      # 4 bytes: smaller than any plan's workspace
    with pytest.raises(rn.NormError):
        rn.ln_bwd(x, x, g, st, st, workspace=small)
    with pytest.raises(rn.NormError):
        rn.rms_bwd(torch.randn(2, 140000, device="cuda"), torch.randn(2, 140000, device="cuda"),
                   torch.ones(140000, device="cuda"))   # beyond one pass of an 8-CTA cluster


def test_column_sums_exact_for_constant_dy():
    """dy = 0.5 everywhere: dbeta = 0.5 M exactly (sums of 0.5 are exact in
    fp32), and with gamma = 1 the bracket vanishes: dx within the bound."""
    M, N = 3000, 1024
    x = torch.randn(M, N, generator=torch.Generator().manual_seed(4))
    dy = torch.full((M, N), 0.5)
    g = torch.ones(N)
    dx, dg, db = run_ln_bwd(dy, x, g, 1e-5)
    assert torch.equal(db.cpu(), torch.full((N,), 0.5 * M))
    check_ln_bwd(dy, x, g, 1e-5, dx, dg, db)


# ------------------------------------------------------------ ordering

def test_forward_then_backward_in_a_cuda_graph():
    """ln_fwd's saved statistics feed ln_bwd inside one captured graph (the
    backward may start before the forward ends and must still see them)."""
    M, N = 1024, 4096
    x, dy, g = _rand(M, N, torch.bfloat16, seed=41, loc=2.0)
    xd, dyd, gd = x.cuda(), dy.cuda(), g.cuda()
    b = torch.zeros_like(gd)
    y = torch.empty_like(xd)
    mean = torch.empty(M, device="cuda")
    rstd = torch.empty(M, device="cuda")
    dx = torch.empty_like(xd)
    dg = torch.empty(N, device="cuda")
    db = torch.empty(N, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = rn.make_bwd_plan(M, N, torch.bfloat16, True, True, sms)
    ws = torch.empty(rn.bwd_workspace_bytes(plan, N, True) // 4, device="cuda")
    rn.ln_fwd(xd, gd, b, 1e-5, out=y, mean=mean, rstd=rstd)
    rn.ln_bwd(dyd, xd, gd, mean, rstd, dx=dx, dgamma=dg, dbeta=db, workspace=ws)
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            rn.ln_fwd(xd, gd, b, 1e-5, out=y, mean=mean, rstd=rstd)
            rn.ln_bwd(dyd, xd, gd, mean, rstd, dx=dx, dgamma=dg, dbeta=db, workspace=ws)
    for _ in range(2):
        for t in (mean, rstd, dx, dg, db):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        check_ln_bwd(dy, x, g, 1e-5, dx, dg, db)


def test_matches_torch_autograd_on_the_gpu():
    """Cross-check with torch's own CUDA backward (fp32): both within the
    bound of the oracle, and close to each other."""
    x, dy, g = _rand(512, 3072, torch.float32, seed=43, loc=1.0)
    xt = x.cuda().requires_grad_()
    gt = g.cuda().requires_grad_()
    bt = torch.zeros(3072, device="cuda", requires_grad=True)
    torch.nn.functional.layer_norm(xt, (3072,), gt, bt, 1e-5).backward(dy.cuda())
    dx, dg, db = run_ln_bwd(dy, x, g, 1e-5)
    assert torch.allclose(dx, xt.grad, rtol=1e-4, atol=1e-5)
    assert torch.allclose(dg, gt.grad, rtol=1e-4, atol=1e-3)
    assert torch.allclose(db, bt.grad, rtol=1e-5, atol=1e-4)
