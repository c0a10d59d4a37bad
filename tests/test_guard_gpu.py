"""Guard bands: every output buffer is surrounded by a canary pattern that
must survive every call (no write outside the output), on every path:
forward (aligned rows, odd widths, shifted starts), fused residual add, FP8
output, strided rows, the statistics, and the backward (dx and the column
gradients)."""
import pytest
import torch

import row_wise_normalization_ln_gb300 as rn

pytestmark = pytest.mark.gpu

G = 256  # guard elements on each side
CANARY = {torch.float32: 12345.5, torch.bfloat16: 12345.0, torch.float16: 1234.0, torch.uint8: 0x5A}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from row_wise_normalization_ln_gb300 import _build
    _build.build()
    rn.library()


class Guarded:
    """A CUDA buffer of `n` elements at element offset `off` past a 16-byte
    boundary, with G canary elements before and after."""

    def __init__(self, n, dtype, off=0):
        self.dtype, self.off, self.n = dtype, off, n
        self.buf = torch.full((2 * G + off + n,), CANARY[dtype], dtype=dtype, device="cuda")
        self.view = self.buf[G + off:G + off + n]

    def intact(self):
        head = self.buf[:G + self.off]
        tail = self.buf[G + self.off + self.n:]
        c = CANARY[self.dtype]
        return bool((head == c).all()) and bool((tail == c).all())


CASES = [(torch.float32, 8, 1024, 0), (torch.float32, 5, 5001, 0), (torch.float32, 3, 4096, 1),
         (torch.bfloat16, 7, 8191, 0), (torch.bfloat16, 4, 8192, 3), (torch.float16, 9, 700, 0),
         (torch.bfloat16, 33, 64, 0), (torch.float32, 2, 65537, 0), (torch.float32, 3, 3, 0)]


@pytest.mark.parametrize("dtype,M,N,off", CASES, ids=[f"{str(d)[6:]}-{m}x{n}-off{o}" for d, m, n, o in CASES])
def test_forward_paths_write_only_their_outputs(dtype, M, N, off):
    g = torch.Generator().manual_seed(N)
    x = Guarded(M * N, dtype, off)
    x.view.copy_((torch.randn(M * N, generator=g) + 1).to(dtype))
    r = Guarded(M * N, dtype, off)
    r.view.copy_(torch.randn(M * N, generator=g).to(dtype))
    gam = (torch.rand(N, generator=g) + 0.5).to(dtype).cuda()
    bet = torch.zeros(N, dtype=dtype, device="cuda")
    xv, rv = x.view.view(M, N), r.view.view(M, N)
    y, h = Guarded(M * N, dtype, off), Guarded(M * N, dtype, off)
    mean, rstd = Guarded(M, torch.float32), Guarded(M, torch.float32)
    rn.ln_fwd(xv, gam, bet, 1e-5, out=y.view.view(M, N), mean=mean.view, rstd=rstd.view)
    rn.rms_fwd(xv, gam, 1e-6, out=y.view.view(M, N))
    rn.ln_fwd_add(xv, rv, gam, bet, 1e-5, h_out=h.view.view(M, N), out=y.view.view(M, N), mean=mean.view,
                  rstd=rstd.view)
    q = Guarded(M * N, torch.uint8, off)
    rn.rms_fwd_fp8(xv, gam, 4.0 / 448, 1e-6, out=q.view.view(M, N))
    rn.ln_fwd_fp8(xv, gam, bet, 4.0 / 448, 1e-5, residual=rv, h_out=h.view.view(M, N), out=q.view.view(M, N),
                  mean=mean.view, rstd=rstd.view)
    torch.cuda.synchronize()
    for name, buf in (("x", x), ("r", r), ("y", y), ("h", h), ("mean", mean), ("rstd", rstd), ("y8", q)):
        assert buf.intact(), name


@pytest.mark.parametrize("dtype,M,N", [(torch.float32, 9, 1000), (torch.bfloat16, 5, 8192), (torch.float32, 3, 65536),
                                       (torch.float16, 7, 33), (torch.float32, 2, 4097)])
def test_backward_writes_only_its_outputs(dtype, M, N):
    g = torch.Generator().manual_seed(N + 1)
    x = (torch.randn(M, N, generator=g) * 2).to(dtype).cuda()
    dy = torch.randn(M, N, generator=g).to(dtype).cuda()
    gam = (torch.rand(N, generator=g) + 0.5).to(dtype).cuda()
    _, mean, rstd = rn.ln_fwd(x, gam, torch.zeros_like(gam), 1e-5)
    dx = Guarded(M * N, dtype)
    dg, db = Guarded(N, torch.float32), Guarded(N, torch.float32)
    rn.ln_bwd(dy, x, gam, mean, rstd, dx=dx.view.view(M, N), dgamma=dg.view, dbeta=db.view)
    dw = Guarded(N, torch.float32)
    rn.rms_bwd(dy, x, gam, 1e-6, dx=dx.view.view(M, N), dw=dw.view)
    torch.cuda.synchronize()
    for name, buf in (("dx", dx), ("dgamma", dg), ("dbeta", db), ("dw", dw)):
        assert buf.intact(), name


def test_strided_rows_write_only_their_block():
    M, N, L = 17, 1000, 1037
    src = torch.randn(M, L, device="cuda")
    dst = torch.full((M, L), CANARY[torch.float32], device="cuda")
    rn.ln_fwd(src[:, 5:5 + N], torch.ones(N, device="cuda"), torch.zeros(N, device="cuda"), 1e-5,
              out=dst[:, 20:20 + N])
    torch.cuda.synchronize()
    assert bool((dst[:, :20] == CANARY[torch.float32]).all()) and bool((dst[:, 20 + N:] == CANARY[torch.float32]).all())
