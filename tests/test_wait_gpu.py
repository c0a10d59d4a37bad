"""The ring kernels' bounded waits, made to run out on purpose (GPU).

The ring kernels (forward plans with `stages` >= 2, and the backward plans
the planner picks for fp32 rows) wait on an mbarrier for each bulk copy of
an upcoming row. A wait that runs out makes the whole CTA stop waiting and
copying, wait out the copies it still has in flight, count the timeout and
finish. These tests set the per-row limit to 0 (each wait tests its copy
once and gives up if it has not landed, which a copy issued moments before
never has), check that the calls return, that the timeout is reported on
the host (norm_synchronize, norm_wait_timeouts) and that the next calls, at
the default limit, are correct. Nothing here faults or hangs the GPU: every
copy is a valid copy of valid memory, and each CTA waits for its copies
before it exits."""
import pytest
import torch

import row_wise_normalization_ln_gb300 as rn

from parity import check_ln, check_ln_bwd, check_rms, check_rms_bwd, ln_stats_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from row_wise_normalization_ln_gb300 import _build
    _build.build()
    rn.library()


@pytest.fixture
def zero_limit():
    """Per-row wait limit 0 for the test body, the previous limit after."""
    old = rn.wait_limit()
    assert old == 2_000_000_000
    rn.synchronize()  # nothing pending from earlier tests
    rn.set_wait_limit(0)
    try:
        yield
    finally:
        rn.set_wait_limit(old)
        assert rn.wait_limit() == old


def _rows(M, N, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(M, N, generator=g) * 1.5 + 3.0).to(dtype)
    dy = torch.randn(M, N, generator=g).to(dtype)
    gamma = (torch.rand(N, generator=g) + 0.5).to(dtype)
    beta = (torch.rand(N, generator=g) * 0.2 - 0.1).to(dtype)
    return x, dy, gamma, beta


FWD_RING = [(torch.float32, 4, 128, 8, 1, 2), (torch.float32, 4, 128, 4, 2, 3), (torch.bfloat16, 8, 256, 2, 1, 2)]


@pytest.mark.parametrize("dtype,vec,T,per,C,S", FWD_RING, ids=[f"{d}-t{t}-p{p}-c{c}-s{s}" for d, v, t, p, c, s in FWD_RING])
def test_forward_ring_wait_runs_out(zero_limit, dtype, vec, T, per, C, S):
    N = C * T * per * vec
    plan = dict(mapping=rn.NORM_MAP_CTA, vec_elems=vec, per_thread=per, group=0, threads=T, cluster=C, stages=S,
                grid=0)
    x, _, g, b = _rows(300, N, dtype, seed=N + S)
    xd, gd, bd = x.cuda(), g.cuda(), b.cuda()
    rn.ln_fwd(xd, gd, bd, 1e-5, plan=plan)       # returns; its outputs are void
    rn.rms_fwd(xd, gd, 1e-6, plan=plan)
    with pytest.raises(rn.NormError) as e:
        rn.synchronize()
    assert e.value.status == rn.NORM_ERR_TIMEOUT
    rn.ln_fwd(xd, gd, bd, 1e-5, plan=plan)
    assert rn.wait_timeouts() > 0                 # the same report, as a count
    assert rn.wait_timeouts() == 0                # ... which the read reset


@pytest.mark.parametrize("dtype,vec,T,per,C,S", FWD_RING, ids=[f"{d}-t{t}-p{p}-c{c}-s{s}" for d, v, t, p, c, s in FWD_RING])
def test_forward_ring_correct_after_a_timeout(dtype, vec, T, per, C, S):
    N = C * T * per * vec
    plan = dict(mapping=rn.NORM_MAP_CTA, vec_elems=vec, per_thread=per, group=0, threads=T, cluster=C, stages=S,
                grid=0)
    x, _, g, b = _rows(300, N, dtype, seed=N + S)
    xd, gd, bd = x.cuda(), g.cuda(), b.cuda()
    old = rn.wait_limit()
    rn.set_wait_limit(0)
    try:
        rn.ln_fwd(xd, gd, bd, 1e-5, plan=plan)
        assert rn.wait_timeouts() > 0
    finally:
        rn.set_wait_limit(old)
    y, mean, rstd = rn.ln_fwd(xd, gd, bd, 1e-5, plan=plan)
    y2 = rn.rms_fwd(xd, gd, 1e-6, plan=plan)
    rn.synchronize()                              # no timeout at the default limit
    check_ln(x, g, b, 1e-5, y.cpu(), mean.cpu(), rstd.cpu())
    check_rms(x, g, 1e-6, y2.cpu())


@pytest.mark.parametrize("ln", [True, False], ids=["ln", "rms"])
def test_backward_ring_wait_runs_out(zero_limit, ln):
    """The backward's default plan for fp32 rows is a 2-stage ring."""
    M, N = 200, 4096
    plan = rn.make_bwd_plan(M, N, torch.float32, ln, True, torch.cuda.get_device_properties(0).multi_processor_count)
    assert plan["stages"] >= 2
    x, dy, g, _ = _rows(M, N, torch.float32, seed=11)
    mean, rstd = ln_stats_f32(x, g, 1e-5)
    if ln:
        rn.ln_bwd(dy.cuda(), x.cuda(), g.cuda(), mean.cuda(), rstd.cuda())
    else:
        rn.rms_bwd(dy.cuda(), x.cuda(), g.cuda(), 1e-6)
    with pytest.raises(rn.NormError) as e:
        rn.synchronize()
    assert e.value.status == rn.NORM_ERR_TIMEOUT


@pytest.mark.parametrize("ln", [True, False], ids=["ln", "rms"])
def test_backward_ring_correct_after_a_timeout(ln):
    M, N = 200, 4096
    x, dy, g, _ = _rows(M, N, torch.float32, seed=12)
    mean, rstd = ln_stats_f32(x, g, 1e-5)
    args = (dy.cuda(), x.cuda(), g.cuda())
    old = rn.wait_limit()
    rn.set_wait_limit(0)
    try:
        if ln:
            rn.ln_bwd(*args, mean.cuda(), rstd.cuda())
        else:
            rn.rms_bwd(*args, 1e-6)
        assert rn.wait_timeouts() > 0
    finally:
        rn.set_wait_limit(old)
    if ln:
        dx, dg, db = rn.ln_bwd(*args, mean.cuda(), rstd.cuda())
        rn.synchronize()
        check_ln_bwd(dy, x, g, 1e-5, dx.cpu(), dg.cpu(), db.cpu())
    else:
        dx, dw = rn.rms_bwd(*args, 1e-6)
        rn.synchronize()
        check_rms_bwd(dy, x, g, 1e-6, dx.cpu(), dw.cpu())

