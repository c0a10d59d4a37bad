"""GPU parity of rows that do not start on 16-byte boundaries (odd widths,
tensors that start at the same misalignment): the CTA kernels take 16-byte
vectors from each row's first aligned element and the elements around them
one by one (the pages' Apex note: consume the head until aligned, then
vectors), checked element by element against the fp64 oracle."""
import pytest
import torch

import row_wise_normalization_ln_gb300 as rn

from parity import check_h, check_ln, check_ln_add, check_ln_fp8, check_rms, check_rms_add, check_rms_fp8

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from row_wise_normalization_ln_gb300 import _build
    _build.build()
    rn.library()


def _at(t: torch.Tensor, off: int) -> torch.Tensor:
    """A CUDA copy of t whose first element sits `off` elements past a
    256-byte boundary."""
    buf = torch.empty(t.numel() + off + 64, dtype=t.dtype, device="cuda")
    v = buf[off:off + t.numel()].view(t.shape)
    v.copy_(t)
    return v


def _rand(M, N, dtype, seed, loc=1.0, scale=2.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(M, N, generator=g) * scale + loc).to(dtype)
    r = torch.randn(M, N, generator=g).to(dtype)
    gamma = (torch.rand(N, generator=g) + 0.5).to(dtype)
    beta = (torch.rand(N, generator=g) * 0.2 - 0.1).to(dtype)
    return x, r, gamma, beta


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("N", [513, 1000, 1023, 4097, 5001, 8191, 8200, 65537])
@pytest.mark.parametrize("off", [0, 1, 3])
def test_shared_offset(dtype, N, off):
    """x and y start `off` elements past a 16-byte boundary; the parameters
    are aligned (off = 0: only the odd widths move the rows off boundaries)."""
    x, _, g, b = _rand(9, N, DT[dtype], seed=N + off)
    xd, gd, bd = _at(x, off), g.cuda(), b.cuda()
    yd = _at(torch.zeros_like(x), off)
    y, mean, rstd = rn.ln_fwd(xd, gd, bd, 1e-5, out=yd)
    torch.cuda.synchronize()
    check_ln(x, g, b, 1e-5, y, mean, rstd)
    y = rn.rms_fwd(xd, gd, 1e-6, out=yd)
    torch.cuda.synchronize()
    check_rms(x, g, 1e-6, y)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_offset_parameters(dtype):
    """gamma and beta off 16-byte boundaries (rows aligned): element loads of
    the parameters, vector rows."""
    x, _, g, b = _rand(7, 4096, DT[dtype], seed=3)
    y, mean, rstd = rn.ln_fwd(x.cuda(), _at(g, 1), _at(b, 2), 1e-5)
    torch.cuda.synchronize()
    check_ln(x, g, b, 1e-5, y, mean, rstd)


def test_different_offsets_take_the_element_path():
    x, _, g, b = _rand(5, 4100, torch.float32, seed=4)
    xd = _at(x, 1)
    yd = _at(torch.zeros_like(x), 2)
    y, mean, rstd = rn.ln_fwd(xd, g.cuda(), b.cuda(), 1e-5, out=yd)
    torch.cuda.synchronize()
    check_ln(x, g, b, 1e-5, y, mean, rstd)


def _variants():
    out = []
    for dtype, vec in (("f32", 4), ("bf16", 8)):
        for C in (1, 2, 8):
            for T in (32, 256):
                for per in (1, 4, 8):
                    cap = C * T * per * vec
                    for N, off in ((cap - 1, 0), (cap - vec - 3, 1), (2 * cap + 5, 3)):
                        if N >= 64 * vec:
                            out.append((dtype, dict(mapping=rn.NORM_MAP_CTA, vec_elems=vec, per_thread=per, group=0,
                                                    threads=T, cluster=C, grid=C * 3), N, off))
    return out


VARIANTS = _variants()


@pytest.mark.parametrize("dtype,plan,N,off", VARIANTS,
                         ids=[f"{d}-p{p['per_thread']}-t{p['threads']}-c{p['cluster']}-N{n}-off{o}"
                              for d, p, n, o in VARIANTS])
def test_every_variant(dtype, plan, N, off):
    """Explicit vector CTA plans on rows off 16-byte boundaries: one round
    (exact and ragged) and three rounds, plain, fused add (h bit for bit)
    and FP8 output."""
    x, r, g, b = _rand(7, N, DT[dtype], seed=N + off, loc=-1.0)
    xd, rd, gd, bd = _at(x, off), _at(r, off), g.cuda(), b.cuda()
    y, mean, rstd = rn.ln_fwd(xd, gd, bd, 1e-5, out=_at(torch.zeros_like(x), off), plan=plan)
    torch.cuda.synchronize()
    check_ln(x, g, b, 1e-5, y, mean, rstd)
    y = rn.rms_fwd(xd, gd, 1e-6, out=_at(torch.zeros_like(x), off), plan=plan)
    torch.cuda.synchronize()
    check_rms(x, g, 1e-6, y)
    if plan["threads"] <= 512:
        h, y = rn.rms_fwd_add(xd, rd, gd, 1e-6, h_out=_at(torch.zeros_like(x), off),
                              out=_at(torch.zeros_like(x), off), plan=plan)
        torch.cuda.synchronize()
        check_rms_add(x, r, g, 1e-6, h, y)
    # FP8: the byte row must start at the same phase as x's elements
    y8 = _at(torch.zeros(x.shape, dtype=torch.uint8), off)
    y8 = rn.rms_fwd_fp8(xd, gd, 8.0 / 448, 1e-6, out=y8, plan=plan)
    torch.cuda.synchronize()
    check_rms_fp8(x, g, 1e-6, 8.0 / 448, y8)


@pytest.mark.parametrize("N", [4097, 65537])
def test_fused_add_in_place_off_boundaries(N):
    """h written over the residual and y over x, all at offset 1, including
    an 8-CTA cluster row in rounds (the element 0 of such a row is held by
    one thread and written after the row's barrier)."""
    for dtype in (torch.float32, torch.bfloat16):
        x, r, g, b = _rand(5, N, dtype, seed=N)
        xd, rd = _at(x, 1), _at(r, 1)
        h, y, mean, rstd = rn.ln_fwd_add(xd, rd, g.cuda(), b.cuda(), 1e-5, h_out=rd, out=xd)
        torch.cuda.synchronize()
        check_ln_add(x, r, g, b, 1e-5, h, y, mean, rstd)


def test_fp8_ln_off_boundaries():
    x, _, g, b = _rand(11, 4099, torch.bfloat16, seed=8)
    y8, mean, rstd = rn.ln_fwd_fp8(_at(x, 3), g.cuda(), b.cuda(), 6.0 / 448, 1e-5,
                                   out=_at(torch.zeros(x.shape, dtype=torch.uint8), 3))
    torch.cuda.synchronize()
    check_ln_fp8(x, g, b, 1e-5, 6.0 / 448, y8, mean, rstd)
