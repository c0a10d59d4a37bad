"""GPU parity: every kernel variant of libnorm, called through the C ABI (via
the Python binding), against the fp64 oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import row_wise_normalization_ln_gb300 as rn
from row_wise_normalization_ln_gb300 import workloads as wl

from parity import check_ln, check_rms, np_of, sample_rows

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
    gamma = torch.rand(N, generator=g) + 0.5
    beta = torch.rand(N, generator=g) * 0.2 - 0.1
    return x.to(dtype), gamma.to(dtype), beta.to(dtype)


def run_ln(x, gamma, beta, eps, plan=None, stats=True):
    y, mean, rstd = rn.ln_fwd(x.cuda(), gamma.cuda(), beta.cuda(), eps, plan=plan, stats=stats)
    torch.cuda.synchronize()
    return y, mean, rstd


def run_rms(x, w, eps, plan=None):
    y = rn.rms_fwd(x.cuda(), w.cuda(), eps, plan=plan)
    torch.cuda.synchronize()
    return y


# ------------------------------------------------------------ the workloads

# Scaled-down rows of every workload (same N, same value recipe): whole
# outputs compared element by element, with the plan the full-size launch
# uses (so the benchmarked kernel variant is the one checked).
PLAIN = [n for n, w in wl.WORKLOADS.items() if not (w.add or w.bwd or w.fp8)]   # the others: their own files
SMALL_M = {"ln_f32_128x1024": 128, "rms_f32_8192x4096": 96, "ln_bf16_4096x8192_outliers": 64,
           "rms_bf16_65536x2048": 517, "ln_f32_2048x65536": 6, "ln_f32_8192x5000": 77,
           "ln_f16_4096x8192": 64, "ln_f32_8192x5001": 77}


@pytest.mark.parametrize("name", PLAIN)
def test_workload_rows_with_full_size_plan(name):
    w = wl.WORKLOADS[name]
    plan = rn.make_plan(w.M, w.N, w.torch_dtype, True, torch.cuda.get_device_properties(0).multi_processor_count)
    ws = w.scaled(M=SMALL_M[name])
    inp = wl.generate(ws, seed=0)
    if plan["mapping"] == rn.NORM_MAP_GROUP:
        plan["grid"] = -(-ws.M // (plan["threads"] // plan["group"]))
    elif plan["stages"]:
        plan["grid"] = plan["cluster"] * 4  # few persistent CTAs: every ring stage is reused
    else:
        plan["grid"] = ws.M * plan["cluster"]
    if w.op == "ln":
        y, mean, rstd = run_ln(inp["x"], inp["gamma"], inp["beta"], w.eps, plan=plan)
        check_ln(inp["x"], inp["gamma"], inp["beta"], w.eps, y, mean, rstd)
    else:
        y = run_rms(inp["x"], inp["w"], w.eps, plan=plan)
        check_rms(inp["x"], inp["w"], w.eps, y)


@pytest.mark.parametrize("name", PLAIN)
def test_workload_full_size_sampled(name):
    """The full-size launch (default plan, as benchmarked): sampled rows
    element by element; statistics of every row (LayerNorm)."""
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, seed=0)
    rows = sample_rows(w.M, 40)
    if w.op == "ln":
        y, mean, rstd = run_ln(inp["x"], inp["gamma"], inp["beta"], w.eps)
        check_ln(inp["x"], inp["gamma"], inp["beta"], w.eps, y, mean, rstd, rows=rows)
        # every row's statistics against the oracle's moments
        import oracle
        xn = np_of(inp["x"])
        e = oracle.eps_as_f32(w.eps)
        mref = np.empty(w.M)
        vref = np.empty(w.M)
        for r in range(w.M):
            mref[r], vref[r] = oracle.row_moments(xn[r])
        rref = 1.0 / np.sqrt(vref + e)
        from parity import check_stats
        check_stats(np_of(mean), np_of(rstd), mref, rref, e)
    else:
        y = run_rms(inp["x"], inp["w"], w.eps)
        check_rms(inp["x"], inp["w"], w.eps, y, rows=rows)
    assert torch.isfinite(y.float()).all()


# ------------------------------------------------------------ edge shapes

EDGE_N = [1, 2, 3, 4, 5, 7, 8, 9, 31, 32, 33, 63, 127, 128, 129, 255, 256, 257, 1000, 1023, 1025,
          2047, 2049, 4095, 4097, 4999, 5000, 8191, 8193, 16385, 32769, 65535, 65537, 100003, 262147]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("N", EDGE_N)
def test_edge_widths(dtype, N):
    M = 5 if N < 100000 else 2
    x, g, b = _rand(M, N, DT[dtype], seed=N, loc=2.0, scale=3.0)
    y, mean, rstd = run_ln(x, g, b, 1e-5)
    check_ln(x, g, b, 1e-5, y, mean, rstd)
    y = run_rms(x, g, 1e-6)
    check_rms(x, g, 1e-6, y)


@pytest.mark.parametrize("M", [1, 2, 31, 33, 255, 257, 1000, 4099])
def test_ragged_row_counts(M):
    """Row counts that leave the last CTA's row groups partly empty."""
    for N, dtype in ((64, torch.float32), (2048, torch.bfloat16), (1024, torch.float32)):
        x, g, b = _rand(M, N, dtype, seed=M)
        y, mean, rstd = run_ln(x, g, b, 1e-5)
        check_ln(x, g, b, 1e-5, y, mean, rstd)
        y = run_rms(x, g, 1e-6)
        check_rms(x, g, 1e-6, y)


def test_zero_rows():
    x = torch.empty(0, 64, device="cuda")
    y, mean, rstd = rn.ln_fwd(x, torch.ones(64, device="cuda"), torch.zeros(64, device="cuda"))
    assert y.shape == (0, 64) and mean.shape == (0,)
    assert rn.rms_fwd(x, torch.ones(64, device="cuda")).shape == (0, 64)


# ------------------------------------------------------------ every variant

def _variants():
    out = []
    for dtype, vec in (("f32", 4), ("bf16", 8)):
        for v in (True, False):
            ve = vec if v else 1
            for G in (1, 2, 4, 8, 16, 32):
                for per in (1, 2, 4, 8):
                    cap = G * per * ve
                    threads = 256 if G < 32 else 128
                    # a row that fills the group exactly, and a ragged one
                    for N in sorted({cap, max(ve, cap - ve * (G // 2 + 1))}):
                        out.append((dtype, dict(mapping=rn.NORM_MAP_GROUP, vec_elems=ve, per_thread=per, group=G,
                                                threads=threads, cluster=1, grid=3), N))
            for C in (1, 2, 4, 8):
                for T in (32, 96, 256, 1024):
                    for per in (1, 2, 4, 8):
                        cap = C * T * per * ve
                        # one exact round, one ragged round, and three rounds
                        for N in sorted({cap, max(ve, cap - 3 * ve), 2 * cap + 7 * ve}):
                            if N > 300000:
                                continue
                            out.append((dtype, dict(mapping=rn.NORM_MAP_CTA, vec_elems=ve, per_thread=per,
                                                    group=0, threads=T, cluster=C, grid=C * 3), N))
                        # the shared-memory ring (vector rows, one round)
                        for S in (2, 3, 4):
                            if not v or T > 512 or S * (T * per * 16 + 24) > 225 * 1024 or cap > 300000:
                                continue
                            for N, grid in ((cap, C * 2), (max(ve, cap - 3 * ve), 0)):
                                out.append((dtype, dict(mapping=rn.NORM_MAP_CTA, vec_elems=ve, per_thread=per,
                                                        group=0, threads=T, cluster=C, stages=S, grid=grid), N))
    return out


VARIANTS = _variants()


@pytest.mark.parametrize("dtype,plan,N", VARIANTS,
                         ids=[f"{d}-m{p['mapping']}-v{p['vec_elems']}-p{p['per_thread']}-g{p['group']}"
                              f"-t{p['threads']}-c{p['cluster']}-s{p.get('stages', 0)}-grid{p['grid']}-N{n}"
                              for d, p, n in VARIANTS])
def test_every_variant(dtype, plan, N):
    """Explicit plans: each (mapping, width, registers, group, CTA size,
    cluster size, rounds, ring stages) variant with a grid smaller than the
    row count, so the grid-stride loop takes several turns and the ring
    wraps."""
    M = 7 if not plan.get("stages") else 11
    x, g, b = _rand(M, N, DT[dtype], seed=N + plan["threads"], loc=-1.5, scale=2.0)
    y, mean, rstd = run_ln(x, g, b, 1e-5, plan=plan)
    check_ln(x, g, b, 1e-5, y, mean, rstd)
    y = run_rms(x, g, 1e-6, plan=plan)
    check_rms(x, g, 1e-6, y)
    if plan.get("stages"):
        assert rn.wait_timeouts() == 0


RING = [(dt, T, per, C, S, N)
        for dt, vec in (("f32", 4), ("bf16", 8), ("f16", 8))
        for (T, per, C, S, N) in ((128, 8, 1, 2, 128 * 8 * vec), (256, 4, 1, 3, 256 * 4 * vec - 5 * vec),
                                  (512, 4, 8, 2, 8 * 512 * 4 * vec), (64, 2, 2, 4, 2 * 64 * 2 * vec - vec),
                                  (32, 1, 1, 4, 32 * vec))]


@pytest.mark.parametrize("dtype,T,per,C,S,N", RING, ids=[f"{r[0]}-t{r[1]}-p{r[2]}-c{r[3]}-s{r[4]}-N{r[5]}" for r in RING])
def test_ring_many_rows(dtype, T, per, C, S, N):
    """The ring kernels on a persistent grid (grid 0: as many CTAs as fit)
    over many more rows than CTAs, so every stage is refilled many times;
    also in place (y written over x). No wait may run out."""
    vec = 4 if dtype == "f32" else 8
    plan = dict(mapping=rn.NORM_MAP_CTA, vec_elems=vec, per_thread=per, group=0, threads=T, cluster=C, stages=S,
                grid=0)
    M = 3000 if N <= 8192 else 400
    x, g, b = _rand(M, N, DT[dtype], seed=N + T + S, loc=3.0, scale=1.5)
    y, mean, rstd = run_ln(x, g, b, 1e-5, plan=plan)
    check_ln(x, g, b, 1e-5, y, mean, rstd)
    y = run_rms(x, g, 1e-6, plan=plan)
    check_rms(x, g, 1e-6, y)
    xd = x.cuda()
    y2, _, _ = rn.ln_fwd(xd, g.cuda(), b.cuda(), 1e-5, out=xd, plan=plan)
    torch.cuda.synchronize()
    assert y2.data_ptr() == xd.data_ptr()
    check_ln(x, g, b, 1e-5, xd.cpu(), mean, rstd)
    assert rn.wait_timeouts() == 0


# ------------------------------------------------------------ layouts

def test_unaligned_pointers_take_the_element_path():
    N, M = 1024, 40
    base = torch.randn(M * N + 3, device="cuda")
    x = base[1:1 + M * N].view(M, N)           # 4-byte offset: not 16-byte aligned
    g = (torch.rand(N + 1, device="cuda") + 0.5)[1:]
    b = (torch.rand(N + 1, device="cuda") - 0.5)[1:]
    out = torch.empty(M * N + 1, device="cuda")[1:].view(M, N)
    y, mean, rstd = rn.ln_fwd(x, g, b, 1e-5, out=out)
    torch.cuda.synchronize()
    check_ln(x.cpu(), g.cpu(), b.cpu(), 1e-5, y, mean, rstd)
    y = rn.rms_fwd(x, g, 1e-6, out=out)
    torch.cuda.synchronize()
    check_rms(x.cpu(), g.cpu(), 1e-6, y)


def test_in_place():
    for dtype in (torch.float32, torch.bfloat16):
        for N in (1000, 4096, 65536):
            x, g, b = _rand(9, N, dtype, seed=N)
            xd = x.cuda()
            y, mean, rstd = rn.ln_fwd(xd, g.cuda(), b.cuda(), 1e-5, out=xd)
            torch.cuda.synchronize()
            assert y.data_ptr() == xd.data_ptr()
            check_ln(x, g, b, 1e-5, y, mean, rstd)
            xd = x.cuda()
            y = rn.rms_fwd(xd, g.cuda(), 1e-6, out=xd)
            torch.cuda.synchronize()
            check_rms(x, g, 1e-6, y)


def test_stats_optional():
    x, g, b = _rand(33, 4096, torch.float32, seed=5)
    y, mean, rstd = run_ln(x, g, b, 1e-5, stats=False)
    assert mean is None and rstd is None
    check_ln(x, g, b, 1e-5, y)


def test_batched_shape_and_side_stream():
    x = torch.randn(4, 16, 768, device="cuda") * 3 + 1
    g = torch.rand(768, device="cuda") + 0.5
    b = torch.rand(768, device="cuda") - 0.5
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y, mean, rstd = rn.ln_fwd(x, g, b, 1e-5)
    s.synchronize()
    assert y.shape == x.shape and mean.shape == (64,)
    check_ln(x.reshape(64, 768).cpu(), g.cpu(), b.cpu(), 1e-5, y.reshape(64, 768), mean, rstd)


def test_deterministic():
    x, g, b = _rand(300, 5000, torch.float32, seed=9, loc=3.0)
    xd, gd, bd = x.cuda(), g.cuda(), b.cuda()
    r1 = rn.ln_fwd(xd, gd, bd)
    r2 = rn.ln_fwd(xd, gd, bd)
    for a, c in zip(r1, r2):
        assert torch.equal(a, c)


# ------------------------------------------------------------ numerics

def test_constant_rows_are_exact():
    """var = 0 exactly, rstd = fp32 rsqrt(eps) within its error, y = beta
    bit for bit ('T3 讲解' §②: eps guards the all-equal row)."""
    for N in (5, 1024, 5000, 65536):
        for dtype in (torch.float32, torch.bfloat16):
            c = 812.5 if dtype == torch.float32 else 812.0
            x = torch.full((4, N), c, dtype=dtype)
            g = (torch.rand(N) + 0.5).to(dtype)
            b = (torch.rand(N) - 0.5).to(dtype)
            y, mean, rstd = run_ln(x, g, b, 1e-5)
            assert torch.all(mean.cpu() == c)
            assert torch.allclose(rstd.cpu().double(), torch.full((4,), float(np.float32(1e-5)) ** -0.5,
                                                                   dtype=torch.float64), rtol=1e-6)
            assert torch.equal(y.cpu(), b.expand(4, N))


def test_cancellation_probe():
    """Rows of the series 1000.001..1000.010 ('第 7 章' §7.3), repeated: the
    naive E[x^2]-E[x]^2 in fp32 returns a variance of 0 or 0.25 on them
    (the oracle pins show it), which would put rstd off by 35 % or more.
    The kernels meet the ordinary fp32 tolerances here."""
    base = np.array([1000.0 + (i + 1) / 1000.0 for i in range(10)], np.float32)
    for N in (10, 4000, 4090, 65520):
        row = np.resize(base, N)
        x = torch.from_numpy(np.stack([row, np.roll(row, 3), row[::-1].copy()]))
        g = torch.ones(N)
        b = torch.zeros(N)
        y, mean, rstd = run_ln(x, g, b, 1e-5)
        check_ln(x, g, b, 1e-5, y, mean, rstd)


def test_outlier_rows_bf16():
    """The cancellation-stress workload at a few rows: per-row offsets of
    100..1000 with +-300 outlier channels, bf16 in and out."""
    w = wl.WORKLOADS["ln_bf16_4096x8192_outliers"].scaled(M=48)
    inp = wl.generate(w, seed=3)
    y, mean, rstd = run_ln(inp["x"], inp["gamma"], inp["beta"], w.eps)
    res = check_ln(inp["x"], inp["gamma"], inp["beta"], w.eps, y, mean, rstd)
    assert res["exact"] > 0.99 * res["n"]


def test_largest_row():
    """N = 2^24, the largest row: a cluster walks the row in many rounds."""
    N = 1 << 24
    x = wl.lattice(2, N, row0=11)
    g = torch.rand(N, generator=torch.Generator().manual_seed(1)) + 0.5
    b = torch.rand(N, generator=torch.Generator().manual_seed(2)) - 0.5
    y, mean, rstd = run_ln(x, g, b, 1e-5)
    check_ln(x, g, b, 1e-5, y, mean, rstd)
    y = run_rms(x, g, 1e-6)
    check_rms(x, g, 1e-6, y)


def test_more_than_2_31_elements():
    """64-bit row offsets: 2^31 + 3*16384 bf16 elements, filled on the
    device with the counter-based lattice; sampled rows are checked."""
    M, N = (1 << 17) + 3, 16384
    x = torch.empty(M, N, device="cuda", dtype=torch.bfloat16)
    for r0 in range(0, M, 8192):
        k = min(8192, M - r0)
        x[r0:r0 + k] = wl.lattice(k, N, row0=r0, device="cuda", dtype=torch.bfloat16)
    g = (torch.rand(N, generator=torch.Generator().manual_seed(4)) + 0.5).to(torch.bfloat16)
    b = (torch.rand(N, generator=torch.Generator().manual_seed(5)) - 0.5).to(torch.bfloat16)
    y, mean, rstd = rn.ln_fwd(x, g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    rows = [0, 1, M // 2, M - 2, M - 1]
    idx = torch.tensor(rows, device="cuda")
    xs = torch.cat([wl.lattice(1, N, row0=r, dtype=torch.bfloat16) for r in rows])
    assert torch.equal(xs, x[idx].cpu())
    check_ln(xs, g, b, 1e-5, y[idx], mean[idx], rstd[idx])
    del x, y, mean, rstd
    torch.cuda.empty_cache()


# ------------------------------------------------------------ ordering

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_chained_calls_read_the_previous_output(dtype):
    """Calls that consume the previous call's output, back to back on one
    stream with no synchronisation (each kernel may be scheduled before its
    predecessor ends, and must still see its output): each link equals the
    oracle applied to the previous link's GPU result."""
    N, M = 4096, 2048
    x, g, b = _rand(M, N, dtype, seed=21, loc=1.0, scale=2.0)
    xd, gd, bd = x.cuda(), g.cuda(), b.cuda()
    outs = [xd]
    for i in range(6):
        y, _, _ = rn.ln_fwd(outs[-1], gd, bd, 1e-5)
        outs.append(rn.rms_fwd(y, gd, 1e-6))
    torch.cuda.synchronize()
    for i in range(6):
        y, mean, rstd = rn.ln_fwd(outs[i], gd, bd, 1e-5)   # recomputed in isolation
        check_ln(outs[i].cpu(), g, b, 1e-5, y, mean, rstd)
        check_rms(y.cpu(), g, 1e-6, outs[i + 1])


def test_chained_calls_in_a_cuda_graph():
    N, M = 8192, 512
    x, g, b = _rand(M, N, torch.float32, seed=22)
    xd, gd, bd = x.cuda(), g.cuda(), b.cuda()
    bufs = [torch.empty_like(xd) for _ in range(4)]
    rn.ln_fwd(xd, gd, bd, 1e-5, out=bufs[0], stats=False)  # warm-up outside capture
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            rn.ln_fwd(xd, gd, bd, 1e-5, out=bufs[0], stats=False)
            for i in range(3):
                rn.rms_fwd(bufs[i], gd, 1e-6, out=bufs[i + 1])
    for _ in range(3):
        for t in bufs:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        check_ln(x, g, b, 1e-5, bufs[0])
        for i in range(3):
            check_rms(bufs[i].cpu(), g, 1e-6, bufs[i + 1])
