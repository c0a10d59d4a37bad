"""Host-side checks of the libnorm C ABI that need no GPU: the library loads,
exports every entry point its header declares, rejects bad arguments before
any CUDA call, and plans every row shape consistently."""
import ctypes
import os
import re

import pytest
import torch

import row_wise_normalization_ln_gb300 as rn
from row_wise_normalization_ln_gb300 import _build
from row_wise_normalization_ln_gb300.workloads import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "libnorm.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return rn.library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:norm_status|const char\*|int)\s+(\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_abi():
    assert set(declared_functions()) == {
        "ln_fwd", "rms_fwd", "ln_fwd_planned", "rms_fwd_planned", "norm_make_plan",
        "ln_fwd_add", "rms_fwd_add", "ln_fwd_add_planned", "rms_fwd_add_planned", "norm_make_plan_add",
        "ln_bwd", "rms_bwd", "ln_bwd_planned", "rms_bwd_planned", "norm_bwd_make_plan", "norm_bwd_workspace_bytes",
        "ln_bwd_noalloc",
        "ln_fwd_fp8", "rms_fwd_fp8", "ln_fwd_add_fp8", "rms_fwd_add_fp8", "ln_fwd_fp8_planned", "rms_fwd_fp8_planned",
        "ln_fwd_strided", "rms_fwd_strided",
        "norm_status_string", "norm_last_cuda_error", "norm_abi_version", "norm_wait_timeouts",
        "norm_synchronize", "norm_set_wait_limit", "norm_wait_limit"}


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert lib.norm_abi_version() == 1


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.norm_status_string(code)
    assert lib.norm_status_string(0) == b"ok"


# Fake device addresses: every call below must fail (or no-op) on the host
# before any CUDA call could touch them.
P = ctypes.c_void_p(0x1000)


@pytest.mark.parametrize("M,N", [(-1, 8), (4, 0), (4, -3), (4, (1 << 24) + 1), (2 ** 62, 4)])
def test_bad_sizes_rejected(lib, M, N):
    assert lib.ln_fwd(P, P, P, P, None, None, M, N, 1e-5, rn.NORM_F32, None) == rn.NORM_ERR_ARG
    assert lib.rms_fwd(P, P, P, M, N, 1e-6, rn.NORM_BF16, None) == rn.NORM_ERR_ARG


def test_bad_dtype_rejected(lib):
    assert lib.ln_fwd(P, P, P, P, None, None, 4, 8, 1e-5, 7, None) == rn.NORM_ERR_DTYPE
    assert lib.rms_fwd(P, P, P, 4, 8, 1e-6, -1, None) == rn.NORM_ERR_DTYPE


@pytest.mark.parametrize("eps", [-1e-5, float("nan"), float("inf")])
def test_bad_eps_rejected(lib, eps):
    assert lib.ln_fwd(P, P, P, P, None, None, 4, 8, eps, rn.NORM_F32, None) == rn.NORM_ERR_ARG
    assert lib.rms_fwd(P, P, P, 4, 8, eps, rn.NORM_F32, None) == rn.NORM_ERR_ARG


def test_null_pointers_rejected(lib):
    for args in [(None, P, P, P), (P, None, P, P), (P, P, None, P), (P, P, P, None)]:
        assert lib.ln_fwd(*args, None, None, 4, 8, 1e-5, rn.NORM_F32, None) == rn.NORM_ERR_ARG
    for args in [(None, P, P), (P, None, P), (P, P, None)]:
        assert lib.rms_fwd(*args, 4, 8, 1e-6, rn.NORM_F32, None) == rn.NORM_ERR_ARG


def test_wait_limit_checked_on_the_host(lib):
    assert lib.norm_set_wait_limit(60_000_000_001) == rn.NORM_ERR_ARG
    assert lib.norm_set_wait_limit(2 ** 64 - 1) == rn.NORM_ERR_ARG
    assert lib.norm_wait_limit(None) == rn.NORM_ERR_ARG
    assert lib.norm_status_string(rn.NORM_ERR_TIMEOUT) != lib.norm_status_string(-99)


def test_no_alloc_null_pointers_rejected_before_any_cuda_call(lib):
    vp = ctypes.c_void_p
    f = lib.ln_bwd_noalloc
    f.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, vp]
    f.restype = ctypes.c_int
    # On a machine without a GPU any CUDA call would give NORM_ERR_CUDA
    # instead: NORM_ERR_ARG shows the check came first.
    for k in range(8):
        args = [P] * 8
        args[k] = None
        assert f(*args, 4, 1024, rn.NORM_F32, None) == rn.NORM_ERR_ARG, k
    assert f(P, P, P, P, P, P, None, P, 0, 1024, rn.NORM_F32, None) == rn.NORM_ERR_ARG   # dgamma even for M == 0
    assert f(P, P, P, P, P, P, P, P, 4, 65540, rn.NORM_F32, None) == rn.NORM_ERR_ARG     # beyond the row limit


def test_wait_timeouts_needs_a_destination(lib):
    # checked before any CUDA call
    assert lib.norm_wait_timeouts(None) == rn.NORM_ERR_ARG


def test_zero_rows_is_a_noop(lib):
    # M == 0: OK, nothing launched, pointers may be NULL
    assert lib.ln_fwd(None, None, None, None, None, None, 0, 8, 1e-5, rn.NORM_F32, None) == rn.NORM_OK
    assert lib.rms_fwd(None, None, None, 0, 8, 1e-6, rn.NORM_BF16, None) == rn.NORM_OK


Q = ctypes.c_void_p(0x2000)   # a second fake buffer


@pytest.mark.parametrize("M,N", [(-1, 8), (4, 0), (4, (1 << 24) + 1), (2 ** 62, 4)])
def test_fused_add_bad_sizes_rejected(lib, M, N):
    assert lib.ln_fwd_add(P, P, P, P, P, Q, None, None, M, N, 1e-5, rn.NORM_F32, None) == rn.NORM_ERR_ARG
    assert lib.rms_fwd_add(P, P, P, P, Q, M, N, 1e-6, rn.NORM_BF16, None) == rn.NORM_ERR_ARG


def test_fused_add_bad_dtype_and_eps_rejected(lib):
    assert lib.ln_fwd_add(P, P, P, P, P, Q, None, None, 4, 8, 1e-5, 3, None) == rn.NORM_ERR_DTYPE
    assert lib.rms_fwd_add(P, P, P, P, Q, 4, 8, float("nan"), rn.NORM_F32, None) == rn.NORM_ERR_ARG


def test_fused_add_null_pointers_rejected(lib):
    for i in range(6):
        args = [P, P, P, P, P, Q]
        args[i] = None
        assert lib.ln_fwd_add(*args, None, None, 4, 8, 1e-5, rn.NORM_F32, None) == rn.NORM_ERR_ARG
    for i in range(5):
        args = [P, P, P, P, Q]
        args[i] = None
        assert lib.rms_fwd_add(*args, 4, 8, 1e-6, rn.NORM_F32, None) == rn.NORM_ERR_ARG


def test_fused_add_h_and_y_must_differ(lib):
    # h == y: both are written, refused on the host
    assert lib.ln_fwd_add(P, Q, P, P, Q, Q, None, None, 4, 8, 1e-5, rn.NORM_F32, None) == rn.NORM_ERR_ARG
    assert lib.rms_fwd_add(P, Q, P, P, P, 4, 8, 1e-6, rn.NORM_BF16, None) == rn.NORM_ERR_ARG


def test_fused_add_zero_rows_is_a_noop(lib):
    assert lib.ln_fwd_add(None, None, None, None, None, None, None, None, 0, 8, 1e-5, rn.NORM_F32,
                          None) == rn.NORM_OK
    assert lib.rms_fwd_add(None, None, None, None, None, 0, 8, 1e-6, rn.NORM_BF16, None) == rn.NORM_OK


@pytest.mark.parametrize("kw", [
    dict(stages=3, grid=0),          # no ring kernel for the fused add
    dict(threads=544),               # above the 512-thread cap of the fused kernels
    dict(threads=1024, per_thread=1),
])
def test_fused_add_plans_rejected(lib, kw):
    p = _plan(**kw)
    assert lib.rms_fwd_add_planned(P, P, P, P, Q, 4, 1000, 1e-6, rn.NORM_F32, None,
                                   ctypes.byref(p)) == rn.NORM_ERR_PLAN
    assert lib.ln_fwd_add_planned(P, P, P, P, P, Q, None, None, 4, 1000, 1e-5, rn.NORM_F32, None,
                                  ctypes.byref(p)) == rn.NORM_ERR_PLAN


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_no_device_reports_cuda_error(lib):
    assert lib.rms_fwd(P, P, P, 4, 8, 1e-6, rn.NORM_F32, None) == rn.NORM_ERR_CUDA
    assert lib.norm_last_cuda_error() != 0


def _plan(**kw):
    base = dict(mapping=rn.NORM_MAP_CTA, vec_elems=4, per_thread=4, group=0, threads=256, cluster=1, grid=8)
    base.update(kw)
    return rn.NormPlan.from_dict(base)


@pytest.mark.parametrize("kw", [
    dict(mapping=5),
    dict(vec_elems=8),                          # fp32 vectors hold 4
    dict(vec_elems=2),
    dict(per_thread=3), dict(per_thread=16), dict(per_thread=0),
    dict(threads=48), dict(threads=0), dict(threads=2048),
    dict(cluster=3), dict(cluster=16),
    dict(cluster=4, grid=6),                    # grid not a multiple of the cluster
    dict(grid=0), dict(grid=1 << 31),
    dict(mapping=rn.NORM_MAP_GROUP, group=3),
    dict(mapping=rn.NORM_MAP_GROUP, group=64),
    dict(mapping=rn.NORM_MAP_GROUP, group=8, per_thread=2),   # 8*2*4 < N: does not cover the row
    dict(stages=1), dict(stages=5), dict(stages=-1),
    dict(stages=3, vec_elems=1),                # the ring needs 16-byte vectors
    dict(stages=3, threads=64, per_thread=1),   # 64*1*4 < N: two rounds, not allowed with a ring
    dict(stages=4, threads=1024, per_thread=8, grid=0),  # 4*1024*8*16 B of ring > 225 KB
    dict(stages=2, threads=1024, per_thread=1, grid=0),  # ring CTAs hold at most 512 threads
    dict(mapping=rn.NORM_MAP_GROUP, group=32, per_thread=8, stages=2),
    dict(grid=0),                               # grid 0 only for ring plans
    dict(mapping=3),
])
def test_bad_plans_rejected(lib, kw):
    p = _plan(**kw)
    st = lib.rms_fwd_planned(P, P, P, 4, 1000, 1e-6, rn.NORM_F32, None, ctypes.byref(p))
    assert st == rn.NORM_ERR_PLAN


def test_vector_plan_needs_alignment(lib):
    # x at 0x1004 and y at 0x1000 sit at different offsets within 16 bytes:
    # no 128-bit plan
    q = ctypes.c_void_p(0x1004)
    p = _plan()
    assert lib.rms_fwd_planned(q, P, P, 4, 1000, 1e-6, rn.NORM_F32, None, ctypes.byref(p)) == rn.NORM_ERR_PLAN
    # not even element-aligned
    assert lib.rms_fwd_planned(ctypes.c_void_p(0x1002), P, ctypes.c_void_p(0x1002), 4, 1000, 1e-6, rn.NORM_F32, None,
                               ctypes.byref(p)) == rn.NORM_ERR_PLAN
    # rows of 1001 fp32 are not whole vectors: a vector plan needs the CTA mapping and no ring
    for kw in (dict(mapping=rn.NORM_MAP_GROUP, group=32, per_thread=8, threads=128),
               dict(stages=3, grid=0, threads=256, per_thread=1)):
        pp = _plan(**kw)
        assert lib.rms_fwd_planned(P, P, P, 4, 1001, 1e-6, rn.NORM_F32, None, ctypes.byref(pp)) == rn.NORM_ERR_PLAN


@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on the fake pointers")
def test_phase_plans_pass_the_host_checks(lib):
    """x and y both at offset 4 within 16 bytes, or rows of 1001 fp32: a
    128-bit CTA plan is accepted (the call then fails at the device query)."""
    q, r = ctypes.c_void_p(0x1004), ctypes.c_void_p(0x2004)
    p = _plan()
    assert lib.rms_fwd_planned(q, P, r, 4, 1000, 1e-6, rn.NORM_F32, None, ctypes.byref(p)) == rn.NORM_ERR_CUDA
    assert lib.rms_fwd_planned(P, P, P, 4, 1001, 1e-6, rn.NORM_F32, None, ctypes.byref(p)) == rn.NORM_ERR_CUDA


@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on the fake pointers")
def test_ring_plan_accepted_before_launch(lib):
    """A valid ring plan passes the host checks; without a GPU the call then
    fails at the device query."""
    p = _plan(stages=3, grid=0)
    st = lib.rms_fwd_planned(P, P, P, 4, 1000, 1e-6, rn.NORM_F32, None, ctypes.byref(p))
    assert st == rn.NORM_ERR_CUDA


def _covers(plan, N):
    cap = plan["per_thread"] * plan["vec_elems"]
    if plan["mapping"] == rn.NORM_MAP_GROUP:
        return plan["group"] * cap >= N and plan["rounds"] == 1
    per_round = plan["cluster"] * plan["threads"] * cap
    return plan["rounds"] * per_round >= N > (plan["rounds"] - 1) * per_round


NS = [1, 2, 3, 4, 5, 7, 8, 9, 31, 32, 33, 64, 100, 255, 256, 257, 1000, 1023, 1024, 1025, 2048, 4095,
      4096, 4999, 5000, 8192, 16384, 32768, 65535, 65536, 100000, 262144, 262145, 1 << 20, (1 << 24)]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("aligned", [True, False])
@pytest.mark.parametrize("M", [1, 3, 128, 8192, 65536])
def test_plans_are_consistent(lib, dtype, aligned, M):
    s = 4 if dtype == torch.float32 else 2
    for N in NS:
        p = rn.make_plan(M, N, dtype, aligned, 152)
        if aligned and (N * s) % 16 == 0:
            vec = 16 // s                                  # every row on a 16-byte boundary
        elif aligned and -(-N // (16 // s)) >= 64:
            vec = 16 // s                                  # rows off boundaries: vector body, CTA mapping
            assert p["mapping"] == rn.NORM_MAP_CTA
        else:
            vec = 1
        assert p["vec_elems"] == vec
        assert p["per_thread"] in (1, 2, 4, 8)
        assert p["threads"] % 32 == 0 and 32 <= p["threads"] <= 1024
        assert _covers(p, N), (N, p)
        if p["mapping"] == rn.NORM_MAP_GROUP:
            assert p["group"] in (1, 2, 4, 8, 16, 32) and p["threads"] % p["group"] == 0
            rows_per_cta = p["threads"] // p["group"]
            assert p["grid"] == max(1, -(-M // rows_per_cta))
        else:
            assert p["cluster"] in (1, 2, 4, 8)
            if p["stages"]:
                assert p["grid"] == 0 and p["rounds"] == 1 and p["vec_elems"] > 1
                assert p["stages"] * (p["threads"] * p["per_thread"] * 16 + 24) <= 225 * 1024 and p["threads"] <= 512
            else:
                assert p["grid"] % p["cluster"] == 0 and p["grid"] == M * p["cluster"]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("M", [1, 3, 128, 8192])
def test_fused_add_plans_are_consistent(lib, dtype, M):
    """The fused calls' plans: CTAs of at most 512 threads, no ring, the row
    covered; short rows in lane groups as the plain calls; at most 4
    accesses per thread per round."""
    for N in NS:
        p = rn.make_plan(M, N, dtype, True, 152, add=True)
        q = rn.make_plan(M, N, dtype, True, 152)
        assert 32 <= p["threads"] <= 512 and p["stages"] == 0
        assert _covers(p, N), (N, p)
        if q["mapping"] == rn.NORM_MAP_GROUP:
            assert p == q, (N, p, q)
        else:
            assert p["mapping"] == rn.NORM_MAP_CTA and p["per_thread"] <= 4
            assert p["grid"] == M * p["cluster"]


def test_plans_for_the_workloads(lib):
    """The mapping each benchmark workload gets (152 SMs, aligned buffers)."""
    got = {name: rn.make_plan(w.M, w.N, w.torch_dtype, True, 152) for name, w in WORKLOADS.items()}
    want = {
        "ln_f32_128x1024": dict(mapping=rn.NORM_MAP_CTA, per_thread=1, threads=256, cluster=1, rounds=1),
        "rms_f32_8192x4096": dict(mapping=rn.NORM_MAP_CTA, per_thread=8, threads=128, cluster=1, rounds=1),
        "ln_bf16_4096x8192_outliers": dict(mapping=rn.NORM_MAP_CTA, per_thread=8, threads=128, cluster=1,
                                           rounds=1),
        "rms_bf16_65536x2048": dict(mapping=rn.NORM_MAP_CTA, per_thread=4, threads=64, cluster=1, rounds=1),
        "ln_f32_2048x65536": dict(mapping=rn.NORM_MAP_CTA, per_thread=8, threads=128, cluster=8, rounds=2),
        "ln_f32_8192x5000": dict(mapping=rn.NORM_MAP_CTA, per_thread=8, threads=160, cluster=1, rounds=1),
        "ln_f16_4096x8192": dict(mapping=rn.NORM_MAP_CTA, per_thread=8, threads=128, cluster=1, rounds=1),
        "ln_f32_8192x5001": dict(mapping=rn.NORM_MAP_CTA, vec_elems=4, per_thread=8, threads=160, cluster=1,
                                 rounds=1),
    }
    got.update({name: rn.make_plan(w.M, w.N, w.torch_dtype, True, 152, add=True)
                for name, w in WORKLOADS.items() if w.add})
    want.update({   # the fused add: 4 accesses per thread per round, more rounds; long rows 2 per round
        "add_rms_f32_8192x4096": dict(mapping=rn.NORM_MAP_CTA, per_thread=4, threads=128, cluster=1, rounds=2),
        "add_rms_bf16_65536x2048": dict(mapping=rn.NORM_MAP_CTA, per_thread=4, threads=64, cluster=1, rounds=1),
        "add_ln_bf16_4096x8192_outliers": dict(mapping=rn.NORM_MAP_CTA, per_thread=4, threads=128, cluster=1,
                                               rounds=2),
        "add_ln_f32_2048x65536": dict(mapping=rn.NORM_MAP_CTA, per_thread=2, threads=128, cluster=8, rounds=8),
    })
    for name, w in want.items():
        for k, v in w.items():
            assert got[name][k] == v, (name, k, got[name])


def test_make_plan_rejects_bad_arguments(lib):
    p = rn.NormPlan()
    assert lib.norm_make_plan(4, 0, 0, 1, 152, ctypes.byref(p)) == rn.NORM_ERR_ARG
    assert lib.norm_make_plan(4, 8, 0, 1, 0, ctypes.byref(p)) == rn.NORM_ERR_ARG
    assert lib.norm_make_plan(4, 8, 9, 1, 152, ctypes.byref(p)) == rn.NORM_ERR_DTYPE
    assert lib.norm_make_plan(4, 8, 0, 1, 152, None) == rn.NORM_ERR_ARG


def test_binding_rejects_cpu_tensors():
    x = torch.zeros(2, 8)
    with pytest.raises(ValueError):
        rn.ln_fwd(x, torch.ones(8), torch.zeros(8))
    with pytest.raises(ValueError):
        rn.rms_fwd(x, torch.ones(8))
    with pytest.raises(ValueError):
        rn.ln_fwd_add(x, x, torch.ones(8), torch.zeros(8))
    with pytest.raises(ValueError):
        rn.rms_fwd_add(x, x, torch.ones(8))



# ---------------------------------------------------------------- backward

W = ctypes.c_void_p(0x100000)   # a fake 16-byte aligned workspace


def _bwd_plan(**kw):
    base = dict(mapping=rn.NORM_MAP_CTA, vec_elems=4, per_thread=4, group=8, threads=256, cluster=1, grid=16)
    base.update(kw)
    return rn.NormPlan.from_dict(base)


def _ln_bwd(lib, M, N, dtype=rn.NORM_F32, ws=W, nbytes=1 << 30, plan=None, ptrs=None):
    p = ptrs or [P] * 8
    if plan is None:
        return lib.ln_bwd(*p, ws, nbytes, M, N, dtype, None)
    return lib.ln_bwd_planned(*p, ws, nbytes, M, N, dtype, None, ctypes.byref(plan))


@pytest.mark.parametrize("M,N", [(-1, 8), (4, 0), (2 ** 62, 4)])
def test_bwd_bad_sizes_rejected(lib, M, N):
    assert _ln_bwd(lib, M, N) == rn.NORM_ERR_ARG
    assert lib.rms_bwd(P, P, P, P, P, W, 1 << 30, M, N, 1e-6, rn.NORM_F32, None) == rn.NORM_ERR_ARG


def test_bwd_rows_beyond_the_limit_rejected(lib):
    """One register pass of an 8-CTA cluster: 65536 fp32 (LayerNorm and
    RMSNorm), 65536 bf16 LayerNorm, 131072 bf16 RMSNorm, 32768 with element
    accesses; refused on the host before any CUDA call."""
    assert _ln_bwd(lib, 4, 65540) == rn.NORM_ERR_ARG
    assert _ln_bwd(lib, 4, 65544, rn.NORM_BF16) == rn.NORM_ERR_ARG
    assert lib.rms_bwd(P, P, P, P, P, W, 1 << 30, 4, 131080, 1e-6, rn.NORM_BF16, None) == rn.NORM_ERR_ARG
    assert lib.rms_bwd(P, P, P, P, P, W, 1 << 30, 4, 32769, 1e-6, rn.NORM_F32, None) == rn.NORM_ERR_ARG
    q = ctypes.c_void_p(0x1004)   # unaligned: element accesses
    assert _ln_bwd(lib, 4, 32772, ptrs=[q] + [P] * 7) == rn.NORM_ERR_ARG
    for N, dt, ln in ((65536, torch.float32, True), (65536, torch.bfloat16, True), (131072, torch.bfloat16, False),
                      (65536, torch.float32, False)):
        p = rn.make_bwd_plan(8, N, dt, ln, True, 152)
        assert p["cluster"] == 8 and p["threads"] <= 512


def test_bwd_null_pointers_rejected(lib):
    for i in range(8):
        ptrs = [P] * 8
        ptrs[i] = None
        assert _ln_bwd(lib, 4, 64, ptrs=ptrs) == rn.NORM_ERR_ARG
    for i in range(5):
        ptrs = [P] * 5
        ptrs[i] = None
        assert lib.rms_bwd(*ptrs, W, 1 << 30, 4, 64, 1e-6, rn.NORM_F32, None) == rn.NORM_ERR_ARG


def test_bwd_workspace_checked_on_the_host(lib):
    p = _bwd_plan()
    need = rn.bwd_workspace_bytes(p, 1024, True)
    assert need == (16 // 8) * 2 * 1024 * 4
    assert rn.bwd_workspace_bytes(p, 1024, False) == need // 2
    assert _ln_bwd(lib, 40, 1024, nbytes=need - 1, plan=p) == rn.NORM_ERR_ARG      # too small
    assert _ln_bwd(lib, 40, 1024, ws=None, plan=p) == rn.NORM_ERR_ARG              # missing
    assert _ln_bwd(lib, 40, 1024, ws=ctypes.c_void_p(0x100004), plan=p) == rn.NORM_ERR_ARG  # misaligned


@pytest.mark.skipif(torch.cuda.is_available(), reason="would launch on the fake pointers")
@pytest.mark.parametrize("stages", [0, 1, 2, 4])
def test_bwd_valid_plan_passes_the_host_checks(lib, stages):
    p = _bwd_plan(stages=stages)
    need = rn.bwd_workspace_bytes(p, 1024, True)
    assert _ln_bwd(lib, 40, 1024, nbytes=need, plan=p) == rn.NORM_ERR_CUDA


@pytest.mark.parametrize("kw", [
    dict(mapping=rn.NORM_MAP_GROUP), dict(stages=5), dict(stages=-1),
    dict(stages=1, cluster=2, group=2, threads=64),  # the register pipeline: one CTA per row
    dict(stages=2, vec_elems=1),                # the ring moves 16-byte vectors
    dict(stages=4, threads=512, per_thread=4),  # 2*512*4*16 B per stage: the ring exceeds 225 KB
    dict(vec_elems=8), dict(per_thread=8), dict(per_thread=3),
    dict(threads=1024), dict(threads=48),
    dict(cluster=3), dict(cluster=16), dict(group=16), dict(group=3),
    dict(cluster=2, group=8),                   # a row cluster is the launched cluster
    dict(grid=12),                              # not a multiple of the cluster
    dict(threads=32, per_thread=1),             # 32*1*4 < 1024: does not cover the row in one pass
])
def test_bwd_bad_plans_rejected(lib, kw):
    assert _ln_bwd(lib, 40, 1024, plan=_bwd_plan(**kw)) == rn.NORM_ERR_PLAN


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("ln", [True, False])
@pytest.mark.parametrize("M", [0, 1, 3, 9, 4096, 65536])
def test_bwd_plans_are_consistent(lib, dtype, ln, M):
    s = 4 if dtype == torch.float32 else 2
    limit = 65536 if (s == 4 or ln) else 131072
    for N in NS + [limit]:
        if N > limit:
            continue
        vec = 16 // s if (N * s) % 16 == 0 else 1
        if vec == 1 and N > 32768:
            with pytest.raises(rn.NormError):
                rn.make_bwd_plan(M, N, dtype, ln, True, 152)
            continue
        p = rn.make_bwd_plan(M, N, dtype, ln, True, 152)
        assert p["vec_elems"] == vec and p["rounds"] == 1
        # a 2-stage ring for fp32 vector rows (it overlaps the register
        # accumulators' slots), the register pipeline for 16-bit vector rows
        # of one CTA, neither otherwise
        acc = (2 if ln else 1) * p["threads"] * p["per_thread"] * vec * 4
        ring = 2 * (2 * p["threads"] * p["per_thread"] * 16 + 8)
        if vec == 4:
            assert max(acc, ring) <= 225 * 1024 and p["stages"] == 2
        elif vec == 8 and p["cluster"] == 1:
            assert p["stages"] == 1
        else:
            assert p["stages"] == 0
        if vec > 1 and p["cluster"] == 1 and p["per_thread"] > 2:
            # fewer accesses per thread would need more than 512 threads
            assert -(-N // (vec * p["per_thread"] // 2)) > 480
        assert p["cluster"] * p["threads"] * p["per_thread"] * vec >= N
        assert p["threads"] % 32 == 0 and 32 <= p["threads"] <= 512
        assert p["cluster"] in (1, 2, 4, 8) and p["group"] in (1, 2, 4, 8)
        if p["cluster"] > 1:
            assert p["group"] == p["cluster"]
        if M == 0:
            assert p["grid"] == 0 and rn.bwd_workspace_bytes(p, N, ln) == 0
        else:
            assert p["grid"] % p["group"] == 0 and p["grid"] >= p["group"]
            assert rn.bwd_workspace_bytes(p, N, ln) == p["grid"] // p["group"] * (2 if ln else 1) * N * 4



# ---------------------------------------------------------------- FP8 output

def test_fp8_argument_checks(lib):
    S = ctypes.c_void_p(0x3000)
    # no scale, no output, h == y8, bad sizes
    assert lib.rms_fwd_fp8(P, P, None, Q, 4, 64, 1e-6, rn.NORM_F32, None) == rn.NORM_ERR_ARG
    assert lib.rms_fwd_fp8(P, P, S, None, 4, 64, 1e-6, rn.NORM_F32, None) == rn.NORM_ERR_ARG
    assert lib.rms_fwd_add_fp8(P, P, P, S, Q, Q, 4, 64, 1e-6, rn.NORM_BF16, None) == rn.NORM_ERR_ARG
    assert lib.ln_fwd_fp8(P, P, P, S, Q, None, None, 4, 0, 1e-5, rn.NORM_F32, None) == rn.NORM_ERR_ARG
    assert lib.ln_fwd_fp8(P, P, None, S, Q, None, None, 4, 64, 1e-5, rn.NORM_F32, None) == rn.NORM_ERR_ARG
    assert lib.ln_fwd_fp8(None, None, None, None, None, None, None, 0, 64, 1e-5, rn.NORM_F16, None) == rn.NORM_OK
    # no ring plans with an FP8 output
    p = _plan(stages=3, grid=0)
    assert lib.rms_fwd_fp8_planned(P, None, P, S, None, Q, 4, 1000, 1e-6, rn.NORM_F32, None,
                                   ctypes.byref(p)) == rn.NORM_ERR_PLAN



# ---------------------------------------------------------------- strided rows

def test_strided_argument_checks(lib):
    # pitches below N, overflowing extents
    assert lib.ln_fwd_strided(P, 7, P, P, Q, 8, None, None, 4, 8, 1e-5, rn.NORM_F32, None, None) == rn.NORM_ERR_ARG
    assert lib.rms_fwd_strided(P, 8, P, Q, 3, 4, 8, 1e-6, rn.NORM_F32, None, None) == rn.NORM_ERR_ARG
    assert lib.rms_fwd_strided(P, 1 << 40, P, Q, 8, 1 << 24, 8, 1e-6, rn.NORM_F32, None, None) == rn.NORM_ERR_ARG
    assert lib.rms_fwd_strided(None, 8, None, None, 8, 0, 8, 1e-6, rn.NORM_F32, None, None) == rn.NORM_OK
    # pitches that differ modulo 16 bytes: no vector plan
    p = _plan(threads=256, per_thread=1, vec_elems=4)
    assert lib.rms_fwd_strided(P, 1001, P, Q, 1002, 4, 1000, 1e-6, rn.NORM_F32, None,
                               ctypes.byref(p)) == rn.NORM_ERR_PLAN


def test_host_pipeline_refuses_unpinned_tensors():
    # checked before any device work
    x = torch.zeros(4, 8)
    with pytest.raises(ValueError):
        rn.host_rows_pipeline([x], [torch.zeros(4, 8)], lambda i, o: None)
    with pytest.raises(ValueError):
        rn.host_rows_pipeline([], [x], lambda i, o: None)
    with pytest.raises(ValueError):  # row counts differ
        rn.host_rows_pipeline([x], [torch.zeros(3, 8)], lambda i, o: None)
    with pytest.raises(ValueError):  # not contiguous
        rn.host_rows_pipeline([torch.zeros(8, 4).t()], [x], lambda i, o: None)


def test_host_pipeline_zero_rows_is_a_no_op():
    # nothing to copy: returns before any device work or pinning check
    calls = []
    assert rn.host_rows_pipeline([torch.zeros(0, 8)], [torch.zeros(0, 8)], lambda i, o: calls.append(1)) is None
    assert calls == []
