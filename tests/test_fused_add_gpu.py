"""GPU parity of the fused residual add + norm (ln_fwd_add, rms_fwd_add),
called through the C ABI (via the Python binding), against the fp64 oracle:
h = x + r bit for bit, y and the statistics against the oracle's norm of h.

The fusion is the add + norm of a transformer's residual stream ("第 7 章
LayerNorm 与 RMSNorm" §7.9-7.10; "T3 讲解" §⑤, vLLM's fused_add_rms_norm)."""
import numpy as np
import pytest
import torch

import row_wise_normalization_ln_gb300 as rn
from row_wise_normalization_ln_gb300 import workloads as wl

from parity import check_h, check_ln_add, check_rms_add, np_of, sample_rows

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


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
    r = torch.randn(M, N, generator=g) * scale - 0.5 * loc
    gamma = torch.rand(N, generator=g) + 0.5
    beta = torch.rand(N, generator=g) * 0.2 - 0.1
    return x.to(dtype), r.to(dtype), gamma.to(dtype), beta.to(dtype)


def run_ln_add(x, r, gamma, beta, eps, plan=None, stats=True):
    h, y, mean, rstd = rn.ln_fwd_add(x.cuda(), r.cuda(), gamma.cuda(), beta.cuda(), eps, plan=plan, stats=stats)
    torch.cuda.synchronize()
    return h, y, mean, rstd


def run_rms_add(x, r, w, eps, plan=None):
    h, y = rn.rms_fwd_add(x.cuda(), r.cuda(), w.cuda(), eps, plan=plan)
    torch.cuda.synchronize()
    return h, y


def _check_both(x, r, g, b, plan=None):
    h, y, mean, rstd = run_ln_add(x, r, g, b, 1e-5, plan=plan)
    check_ln_add(x, r, g, b, 1e-5, h, y, mean, rstd)
    h, y = run_rms_add(x, r, g, 1e-6, plan=plan)
    check_rms_add(x, r, g, 1e-6, h, y)


# ------------------------------------------------------------ the workloads

FUSED = [n for n, w in wl.WORKLOADS.items() if w.add and not w.fp8]   # the FP8 one: test_fp8_gpu.py
SMALL_M = {"add_rms_f32_8192x4096": 96, "add_rms_bf16_65536x2048": 517, "add_ln_bf16_4096x8192_outliers": 64,
           "add_ln_f32_2048x65536": 6}


@pytest.mark.parametrize("name", FUSED)
def test_workload_rows_with_full_size_plan(name):
    """Scaled-down rows (same N, same recipe) under the plan of the full-size
    launch, whole outputs compared."""
    w = wl.WORKLOADS[name]
    plan = rn.make_plan(w.M, w.N, w.torch_dtype, True, torch.cuda.get_device_properties(0).multi_processor_count,
                        add=True)
    ws = w.scaled(M=SMALL_M[name])
    inp = wl.generate(ws, seed=0)
    if plan["mapping"] == rn.NORM_MAP_GROUP:
        plan["grid"] = -(-ws.M // (plan["threads"] // plan["group"]))
    else:
        plan["grid"] = ws.M * plan["cluster"]
    if w.op == "ln":
        h, y, mean, rstd = run_ln_add(inp["x"], inp["r"], inp["gamma"], inp["beta"], w.eps, plan=plan)
        check_ln_add(inp["x"], inp["r"], inp["gamma"], inp["beta"], w.eps, h, y, mean, rstd)
    else:
        h, y = run_rms_add(inp["x"], inp["r"], inp["w"], w.eps, plan=plan)
        check_rms_add(inp["x"], inp["r"], inp["w"], w.eps, h, y)


@pytest.mark.parametrize("name", FUSED)
def test_workload_full_size(name):
    """The full-size launch (default plan, as benchmarked): h of every
    element bit for bit; y and the statistics on sampled rows."""
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, seed=0)
    rows = sample_rows(w.M, 40)
    if w.op == "ln":
        h, y, mean, rstd = run_ln_add(inp["x"], inp["r"], inp["gamma"], inp["beta"], w.eps)
        check_h(inp["x"], inp["r"], h)
        check_ln_add(inp["x"], inp["r"], inp["gamma"], inp["beta"], w.eps, h, y, mean, rstd, rows=rows)
    else:
        h, y = run_rms_add(inp["x"], inp["r"], inp["w"], w.eps)
        check_h(inp["x"], inp["r"], h)
        check_rms_add(inp["x"], inp["r"], inp["w"], w.eps, h, y, rows=rows)
    assert torch.isfinite(y.float()).all()


# ------------------------------------------------------------ shapes

EDGE_N = [1, 2, 3, 5, 8, 31, 33, 127, 128, 129, 257, 1000, 1023, 1025, 4095, 4097, 5000, 8193, 32769,
          65537, 100003]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", EDGE_N)
def test_edge_widths(dtype, N):
    x, r, g, b = _rand(5 if N < 100000 else 2, N, DT[dtype], seed=N, loc=2.0, scale=3.0)
    _check_both(x, r, g, b)


@pytest.mark.parametrize("M", [1, 3, 33, 257, 1000])
def test_ragged_row_counts(M):
    for N, dtype in ((64, torch.float32), (2048, torch.bfloat16), (1024, torch.float32)):
        x, r, g, b = _rand(M, N, dtype, seed=M)
        _check_both(x, r, g, b)


def test_zero_rows():
    x = torch.empty(0, 64, device="cuda")
    h, y, mean, rstd = rn.ln_fwd_add(x, x, torch.ones(64, device="cuda"), torch.zeros(64, device="cuda"))
    assert h.shape == (0, 64) and y.shape == (0, 64) and mean.shape == (0,)
    h, y = rn.rms_fwd_add(x, x, torch.ones(64, device="cuda"))
    assert h.shape == (0, 64)


# ------------------------------------------------------------ every variant

def _variants():
    out = []
    for dtype, vec in (("f32", 4), ("bf16", 8)):
        for v in (True, False):
            ve = vec if v else 1
            for G in (1, 2, 4, 8, 16, 32):
                for per in (1, 2, 4, 8):
                    cap = G * per * ve
                    for N in sorted({cap, max(ve, cap - ve * (G // 2 + 1))}):
                        out.append((dtype, dict(mapping=rn.NORM_MAP_GROUP, vec_elems=ve, per_thread=per, group=G,
                                                threads=256 if G < 32 else 128, cluster=1, grid=3), N))
            for C in (1, 2, 4, 8):
                for T in (32, 96, 512):
                    for per in (1, 2, 4, 8):
                        cap = C * T * per * ve
                        # one exact round, one ragged round, and three rounds
                        for N in sorted({cap, max(ve, cap - 3 * ve), 2 * cap + 7 * ve}):
                            if N > 300000:
                                continue
                            out.append((dtype, dict(mapping=rn.NORM_MAP_CTA, vec_elems=ve, per_thread=per,
                                                    group=0, threads=T, cluster=C, grid=C * 3), N))
    return out


VARIANTS = _variants()


@pytest.mark.parametrize("dtype,plan,N", VARIANTS,
                         ids=[f"{d}-m{p['mapping']}-v{p['vec_elems']}-p{p['per_thread']}-g{p['group']}"
                              f"-t{p['threads']}-c{p['cluster']}-grid{p['grid']}-N{n}" for d, p, n in VARIANTS])
def test_every_variant(dtype, plan, N):
    """Explicit plans: every fused (mapping, width, registers, group, CTA
    size, cluster size, rounds) variant, with a grid smaller than the row
    count so that the grid-stride loop takes several turns."""
    x, r, g, b = _rand(7, N, DT[dtype], seed=N + plan["threads"], loc=-1.5, scale=2.0)
    _check_both(x, r, g, b, plan=plan)


# ------------------------------------------------------------ layouts

def test_unaligned_pointers_take_the_element_path():
    N, M = 1024, 40
    base = torch.randn(3 * M * N + 3, device="cuda")
    x = base[1:1 + M * N].view(M, N)                  # 4-byte offset: not 16-byte aligned
    r = base[2 + M * N:2 + 2 * M * N].view(M, N)
    g = (torch.rand(N + 1, device="cuda") + 0.5)[1:]
    b = (torch.rand(N + 1, device="cuda") - 0.5)[1:]
    hb = torch.empty(M * N + 1, device="cuda")[1:].view(M, N)
    yb = torch.empty(M * N + 1, device="cuda")[1:].view(M, N)
    h, y, mean, rstd = rn.ln_fwd_add(x, r, g, b, 1e-5, h_out=hb, out=yb)
    torch.cuda.synchronize()
    check_ln_add(x.cpu(), r.cpu(), g.cpu(), b.cpu(), 1e-5, h, y, mean, rstd)
    h, y = rn.rms_fwd_add(x, r, g, 1e-6, h_out=hb, out=yb)
    torch.cuda.synchronize()
    check_rms_add(x.cpu(), r.cpu(), g.cpu(), 1e-6, h, y)


def _cluster_plan(dtype, per, threads, cluster, M):
    return dict(mapping=rn.NORM_MAP_CTA, vec_elems=4 if dtype == torch.float32 else 8, per_thread=per, group=0,
                threads=threads, cluster=cluster, grid=M * cluster)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N,cluster_rounds", [(200, False), (1000, False), (4096, False), (65536, False),
                                              (65536, True), (100003, False)])
def test_in_place_residual_update(dtype, N, cluster_rounds):
    """The residual stream updated in place (h written over r, y over x) and
    the swapped form (h over x, y over r): group rows, CTA rows, and a
    cluster of 8 CTAs walking the row in rounds, whose output pass reads x
    and r again while other CTAs of the cluster are already writing."""
    M = 9
    x, r, g, b = _rand(M, N, dtype, seed=N)
    gd, bd = g.cuda(), b.cuda()
    plan = None
    if cluster_rounds:
        per = 8 if dtype == torch.float32 else 4
        plan = _cluster_plan(dtype, per, 128, 8, M)   # 8 * 128 * per * vec < N: two rounds
    for swap in (False, True):
        xd, rd = x.cuda(), r.cuda()
        hb, yb = (xd, rd) if swap else (rd, xd)
        h, y, mean, rstd = rn.ln_fwd_add(xd, rd, gd, bd, 1e-5, h_out=hb, out=yb, plan=plan)
        torch.cuda.synchronize()
        assert h.data_ptr() == hb.data_ptr() and y.data_ptr() == yb.data_ptr()
        check_ln_add(x, r, g, b, 1e-5, h, y, mean, rstd)
        xd, rd = x.cuda(), r.cuda()
        hb, yb = (xd, rd) if swap else (rd, xd)
        h, y = rn.rms_fwd_add(xd, rd, gd, 1e-6, h_out=hb, out=yb, plan=plan)
        torch.cuda.synchronize()
        check_rms_add(x, r, g, 1e-6, h, y)


def test_same_tensor_as_both_inputs():
    """x and r the same buffer: h = 2x, written over it."""
    x, _, g, b = _rand(17, 5000, torch.float32, seed=3, loc=1.0)
    xd = x.cuda()
    h, y, mean, rstd = rn.ln_fwd_add(xd, xd, g.cuda(), b.cuda(), 1e-5, h_out=xd)
    torch.cuda.synchronize()
    check_ln_add(x, x, g, b, 1e-5, h, y, mean, rstd)
    assert torch.equal(h.cpu(), 2 * x)


def test_h_equal_y_refused():
    x = torch.randn(4, 64, device="cuda")
    with pytest.raises(rn.NormError):
        rn.ln_fwd_add(x, x, torch.ones(64, device="cuda"), torch.zeros(64, device="cuda"), h_out=x, out=x)


def test_stats_optional_and_batched_shape_on_a_side_stream():
    x = torch.randn(4, 16, 768, device="cuda") * 3 + 1
    r = torch.randn(4, 16, 768, device="cuda")
    g = torch.rand(768, device="cuda") + 0.5
    b = torch.rand(768, device="cuda") - 0.5
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        h, y, mean, rstd = rn.ln_fwd_add(x, r, g, b, 1e-5, stats=False)
    s.synchronize()
    assert h.shape == x.shape and y.shape == x.shape and mean is None and rstd is None
    check_ln_add(x.reshape(64, 768).cpu(), r.reshape(64, 768).cpu(), g.cpu(), b.cpu(), 1e-5,
                 h.reshape(64, 768), y.reshape(64, 768))


def test_deterministic():
    x, r, g, b = _rand(300, 5000, torch.float32, seed=9, loc=3.0)
    xd, rd, gd, bd = x.cuda(), r.cuda(), g.cuda(), b.cuda()
    r1 = rn.ln_fwd_add(xd, rd, gd, bd)
    r2 = rn.ln_fwd_add(xd, rd, gd, bd)
    for a, c in zip(r1, r2):
        assert torch.equal(a, c)


# ------------------------------------------------------------ numerics

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_sum_to_a_constant_row(dtype):
    """x + r = c exactly in every element (small integers): the row of h is
    constant, so var = 0, mean = c and y = beta bit for bit."""
    for N in (5, 1024, 5000, 65536):
        g0 = torch.Generator().manual_seed(N)
        x = torch.randint(-60, 60, (3, N), generator=g0).to(dtype)
        r = (37.0 - x.float()).to(dtype)
        g = (torch.rand(N, generator=g0) + 0.5).to(dtype)
        b = (torch.rand(N, generator=g0) - 0.5).to(dtype)
        h, y, mean, rstd = run_ln_add(x, r, g, b, 1e-5)
        assert torch.equal(h.cpu(), torch.full((3, N), 37.0, dtype=dtype))
        assert torch.equal(y.cpu(), b.expand(3, N))
        assert torch.equal(mean.cpu(), torch.full((3,), 37.0))
        check_ln_add(x, r, g, b, 1e-5, h, y, mean, rstd)


def test_rounding_of_the_sum_bf16():
    """bf16 sums that are ties or near-ties of the bf16 grid: h must be the
    round-to-nearest-even of the exact sum (what a separate add stores)."""
    M, N = 16, 4096
    g0 = torch.Generator().manual_seed(11)
    big = (torch.rand(M, N, generator=g0) * 64 + 64).to(torch.bfloat16)   # ulp 0.5 in [64, 128)
    small = (torch.randint(0, 4, (M, N), generator=g0).float() * 0.125 - 0.25).to(torch.bfloat16)
    gam = torch.ones(N, dtype=torch.bfloat16)
    bet = torch.zeros(N, dtype=torch.bfloat16)
    h, y, mean, rstd = run_ln_add(big, small, gam, bet, 1e-5)
    check_ln_add(big, small, gam, bet, 1e-5, h, y, mean, rstd)
    assert not torch.equal(h.cpu().float(), big.float() + small.float())   # some sums did round


# ------------------------------------------------------------ ordering

def test_chained_residual_stream_in_a_cuda_graph():
    """A residual stream of several add + norm layers captured in one CUDA
    graph (launches may start before their predecessor ends): each link is
    checked against the oracle on the previous link's GPU results."""
    N, M = 4096, 1024
    x, r, g, b = _rand(M, N, torch.bfloat16, seed=23, loc=1.0)
    xd, rd, gd, bd = x.cuda(), r.cuda(), g.cuda(), b.cuda()
    hs = [torch.empty_like(xd) for _ in range(4)]
    ys = [torch.empty_like(xd) for _ in range(4)]
    rn.rms_fwd_add(xd, rd, gd, 1e-6, h_out=hs[0], out=ys[0])   # warm-up outside capture
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            rn.rms_fwd_add(xd, rd, gd, 1e-6, h_out=hs[0], out=ys[0])
            for i in range(3):
                # the next layer's input is this layer's normalised output
                rn.ln_fwd_add(ys[i], hs[i], gd, bd, 1e-5, h_out=hs[i + 1], out=ys[i + 1], stats=False)
    for _ in range(2):
        for t in hs + ys:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        check_rms_add(x, r, g, 1e-6, hs[0], ys[0])
        for i in range(3):
            check_ln_add(ys[i].cpu(), hs[i].cpu(), g, b, 1e-5, hs[i + 1], ys[i + 1])


def test_matches_the_unfused_calls():
    """rms_fwd_add equals a torch add followed by rms_fwd, bit for bit (the
    same kernel arithmetic on the same h, under the same plan)."""
    plan = rn.make_plan(2048, 8192, torch.bfloat16)   # one plan (one round) for both calls
    x, r, g, _ = _rand(2048, 8192, torch.bfloat16, seed=31)
    xd, rd, gd = x.cuda(), r.cuda(), g.cuda()
    h, y = rn.rms_fwd_add(xd, rd, gd, 1e-6, plan=plan)
    hh = xd + rd
    assert torch.equal(h, hh)
    assert torch.equal(y, rn.rms_fwd(hh, gd, 1e-6, plan=plan))
    assert np.array_equal(np_of(h), np_of(hh))
