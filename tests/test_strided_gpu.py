"""GPU parity of strided rows (row pitch > N, e.g. a column block of a wider
matrix), through ln_fwd_strided / rms_fwd_strided (via the Python binding,
which keeps evenly strided views, the T3 drill's host wrapper, §④), against
the fp64 oracle on the same rows."""
import pytest
import torch

import row_wise_normalization_ln_gb300 as rn

from parity import check_ln, check_rms

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from row_wise_normalization_ln_gb300 import _build
    _build.build()
    rn.library()


def _mat(M, L, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(M, L, generator=g) * 2 + 1).to(dtype)


def _params(N, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.rand(N, generator=g) + 0.5).to(dtype), (torch.rand(N, generator=g) - 0.5).to(dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("N,pad", [(1000, 24), (1000, 3), (4096, 64), (4096, 1), (5000, 8), (64, 7), (17, 5),
                                   (65536, 16)])
def test_column_block(dtype, N, pad):
    """x = the first N columns of an [M, N + pad] matrix (the pad makes the
    pitch whole vectors, or not); y contiguous."""
    M = 9
    big = _mat(M, N + pad, DT[dtype], seed=N + pad).cuda()
    x = big[:, :N]
    assert not x.is_contiguous()
    g, b = _params(N, DT[dtype], seed=N)
    y, mean, rstd = rn.ln_fwd(x, g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    check_ln(x.cpu(), g, b, 1e-5, y, mean, rstd)
    y = rn.rms_fwd(x, g.cuda(), 1e-6)
    torch.cuda.synchronize()
    check_rms(x.cpu(), g, 1e-6, y)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_strided_output_and_in_place(dtype):
    """y written into a column block of another matrix, and over x itself."""
    M, N = 33, 2048
    big = _mat(M, N + 32, DT[dtype], seed=1).cuda()
    x = big[:, 16:16 + N]
    x_cpu = x.cpu()
    g, b = _params(N, DT[dtype], seed=2)
    out_big = torch.full((M, N + 48), 7.0, dtype=DT[dtype], device="cuda")
    out = out_big[:, 8:8 + N]
    y, mean, rstd = rn.ln_fwd(x, g.cuda(), b.cuda(), 1e-5, out=out)
    torch.cuda.synchronize()
    assert y.data_ptr() == out.data_ptr()
    check_ln(x_cpu, g, b, 1e-5, y, mean, rstd)
    assert torch.all(out_big[:, :8] == 7) and torch.all(out_big[:, 8 + N:] == 7)   # nothing outside the block
    y = rn.rms_fwd(x, g.cuda(), 1e-6, out=x)
    torch.cuda.synchronize()
    check_rms(x_cpu, g, 1e-6, y)
    assert torch.all(big[:, :16].cpu() == _mat(M, N + 32, DT[dtype], seed=1)[:, :16])


def test_three_dimensional_view():
    """[B, S, N] taken from [B, S, L]: the leading dims collapse into one row
    stride, no copy."""
    B, S, N, L = 3, 11, 768, 800
    big = _mat(B * S, L, torch.bfloat16, seed=5).cuda().view(B, S, L)
    x = big[..., :N]
    g, b = _params(N, torch.bfloat16, seed=6)
    y, mean, rstd = rn.ln_fwd(x, g.cuda(), b.cuda(), 1e-5)
    torch.cuda.synchronize()
    assert y.shape == x.shape
    check_ln(x.reshape(-1, N).cpu(), g, b, 1e-5, y.reshape(-1, N), mean, rstd)


@pytest.mark.parametrize("plan", [
    dict(mapping=rn.NORM_MAP_CTA, vec_elems=4, per_thread=8, group=0, threads=128, cluster=1, grid=5),
    dict(mapping=rn.NORM_MAP_CTA, vec_elems=4, per_thread=2, group=0, threads=64, cluster=4, grid=8),
    dict(mapping=rn.NORM_MAP_GROUP, vec_elems=4, per_thread=8, group=32, threads=128, cluster=1, grid=2),
    dict(mapping=rn.NORM_MAP_CTA, vec_elems=4, per_thread=2, group=0, threads=128, cluster=1, stages=3, grid=0),
    dict(mapping=rn.NORM_MAP_CTA, vec_elems=1, per_thread=4, group=0, threads=64, cluster=2, grid=6),
])
def test_explicit_plans(plan):
    """Group, CTA, cluster, ring and element plans on rows of pitch 1056 (whole vectors)."""
    M, N, L = 13, 1024, 1056
    big = _mat(M, L, torch.float32, seed=9).cuda()
    x = big[:, :N]
    g, b = _params(N, torch.float32, seed=10)
    y, mean, rstd = rn.ln_fwd(x, g.cuda(), b.cuda(), 1e-5, plan=plan)
    torch.cuda.synchronize()
    check_ln(x.cpu(), g, b, 1e-5, y, mean, rstd)
    y = rn.rms_fwd(x, g.cuda(), 1e-6, plan=plan)
    torch.cuda.synchronize()
    check_rms(x.cpu(), g, 1e-6, y)
