"""host_rows_pipeline: row-wise library calls over pinned host tensors,
chunks copied in, normalised and copied back on three streams. Outputs
checked against the fp64 oracle (tests/parity.py bars): LayerNorm with its
statistics, RMSNorm, the fused residual add (h and y) and an FP8 output;
chunk sizes that divide M, leave a ragged last chunk, or exceed M."""
import pytest
import torch

import row_wise_normalization_ln_gb300 as rn

from parity import check_h, check_ln, check_ln_fp8, check_rms, check_rms_add

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from row_wise_normalization_ln_gb300 import _build
    _build.build()
    rn.library()


def _rand(M, N, dtype, seed, loc=0.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(M, N, generator=g) * 2 + loc).to(dtype)
    r = torch.randn(M, N, generator=g).to(dtype)
    gamma = (torch.rand(N, generator=g) + 0.5).to(dtype)
    beta = (torch.rand(N, generator=g) * 0.2 - 0.1).to(dtype)
    return x, r, gamma, beta


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M,chunk", [(1000, 256), (1000, 333), (64, 4096), (517, None)])
def test_layernorm_and_rmsnorm(dtype, M, chunk):
    N = 2048
    x, _, g, b = _rand(M, N, dtype, seed=M + (chunk or 0), loc=1.0)
    hx = x.pin_memory()
    gd, bd = g.cuda(), b.cuda()
    hy = torch.empty_like(hx).pin_memory()
    hm = torch.empty(M, dtype=torch.float32).pin_memory()
    hr = torch.empty(M, dtype=torch.float32).pin_memory()
    rn.host_rows_pipeline([hx], [hy, hm, hr],
                          lambda i, o: rn.ln_fwd(i[0], gd, bd, 1e-5, out=o[0], mean=o[1], rstd=o[2]),
                          chunk_rows=chunk)
    torch.cuda.synchronize()
    check_ln(x, g, b, 1e-5, hy, hm, hr)
    rn.host_rows_pipeline([hx], [hy], lambda i, o: rn.rms_fwd(i[0], gd, 1e-6, out=o[0]), chunk_rows=chunk)
    torch.cuda.synchronize()
    check_rms(x, g, 1e-6, hy)


def test_fused_add_and_fp8():
    M, N = 777, 4096
    x, r, g, b = _rand(M, N, torch.bfloat16, seed=5)
    hx, hr_ = x.pin_memory(), r.pin_memory()
    gd, bd = g.cuda(), b.cuda()
    hh = torch.empty_like(hx).pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    rn.host_rows_pipeline([hx, hr_], [hh, hy],
                          lambda i, o: rn.rms_fwd_add(i[0], i[1], gd, 1e-6, h_out=o[0], out=o[1]), chunk_rows=200)
    torch.cuda.synchronize()
    check_h(x, r, hh)
    check_rms_add(x, r, g, 1e-6, hh, hy)
    scale = 8.0 / 448
    sc = torch.tensor([scale], dtype=torch.float32, device="cuda")
    hq = torch.empty(M, N, dtype=torch.uint8).pin_memory()
    hm = torch.empty(M, dtype=torch.float32).pin_memory()
    hs = torch.empty(M, dtype=torch.float32).pin_memory()
    rn.host_rows_pipeline([hx], [hq, hm, hs],
                          lambda i, o: rn.ln_fwd_fp8(i[0], gd, bd, sc, 1e-5, out=o[0], mean=o[1], rstd=o[2]),
                          chunk_rows=256)
    torch.cuda.synchronize()
    check_ln_fp8(x, g, b, 1e-5, scale, hq, hm, hs)


def test_zero_rows_and_a_consumer_on_the_stream():
    """M = 0 queues nothing; afterwards a kernel on the current stream sees
    the copied-back rows without a host synchronisation in between."""
    e = torch.empty(0, 64, dtype=torch.float32).pin_memory()
    rn.host_rows_pipeline([e], [torch.empty_like(e).pin_memory()], lambda i, o: None)
    x, _, g, _ = _rand(300, 1024, torch.float32, seed=3)
    hx = x.pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    gd = g.cuda()
    rn.host_rows_pipeline([hx], [hy], lambda i, o: rn.rms_fwd(i[0], gd, 1e-6, out=o[0]), chunk_rows=64)
    back = hy.to("cuda", non_blocking=True)   # ordered after the pipeline on the current stream
    torch.cuda.synchronize()
    check_rms(x, g, 1e-6, back)


def test_two_host_threads_at_once():
    """Two host threads, each on its own stream, run pipelines on the same
    device at the same time; both results match the oracle."""
    import threading
    N = 2048
    cases = []
    for k in range(2):
        x, _, g, _ = _rand(600, N, torch.float32, seed=40 + k)
        cases.append((x, g, x.pin_memory(), torch.empty(600, N).pin_memory(), g.cuda()))
    errs = []

    def work(c):
        try:
            x, g, hx, hy, gd = c
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(5):
                    rn.host_rows_pipeline([hx], [hy], lambda i, o: rn.rms_fwd(i[0], gd, 1e-6, out=o[0]), chunk_rows=128)
            s.synchronize()
        except Exception as e:  # reported below
            errs.append(e)

    ts = [threading.Thread(target=work, args=(c,)) for c in cases]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errs, errs
    torch.cuda.synchronize()
    for x, g, hx, hy, gd in cases:
        check_rms(x, g, 1e-6, hy)


def test_a_stream_of_batches_without_waits():
    """Calls with wait=False: each call's copies back may overlap the next
    call's copies in; host_rows_wait then orders all of them before a
    consumer on the current stream. Three batches, three host outputs, each
    checked against the oracle."""
    N = 2048
    x_list = [_rand(700, N, torch.float32, seed=60 + k)[0] for k in range(3)]
    g = _rand(1, N, torch.float32, seed=63)[2]
    gd = g.cuda()
    hxs = [x.pin_memory() for x in x_list]
    hys = [torch.empty_like(hx).pin_memory() for hx in hxs]
    for hx, hy in zip(hxs, hys):
        rn.host_rows_pipeline([hx], [hy], lambda i, o: rn.rms_fwd(i[0], gd, 1e-6, out=o[0]), chunk_rows=160,
                              wait=False)
    rn.host_rows_wait()
    backs = [hy.to("cuda", non_blocking=True) for hy in hys]   # ordered after every copy back
    torch.cuda.synchronize()
    for x, back in zip(x_list, backs):
        check_rms(x, g, 1e-6, back)
