"""Seeded synthetic inputs for the LayerNorm / RMSNorm forward workloads.

This module only draws numbers: it holds none of the normalisation
arithmetic. Both the CUDA path (tests, benchmark) and the CPU oracle read the
very same tensors produced here, so the choice of generator does not affect
parity.

Workloads (shapes and value distributions of the source pages):
  ln_f32_128x1024          LayerNorm fp32, M=128 N=1024 (the ROCm LayerNorm
                           README's usage example); x ~ N(0,1), gamma ~ U(.5,1.5),
                           beta ~ U(-.1,.1), eps 1e-5.
  rms_f32_8192x4096        RMSNorm fp32, B=8 T=1024 C=4096 ("CUDA算子优化(2)：
                           RMSNorm" §2); x ~ U(-1,1), w ~ U(0,1), eps 1e-6.
  ln_bf16_4096x8192_outliers  LayerNorm bf16, M=4096 N=8192 (the T3 drill's
                           N); row offset ~ U(100,1000) + N(0, 0.01^2) noise,
                           1 % of channels (fixed per seed) replaced by +-300.
  rms_bf16_65536x2048      RMSNorm bf16, B=64 T=1024 C=2048 (the RMSNorm
                           post's V0/V2 sizes); x ~ U(-1,1), w ~ U(0,1), eps 1e-6.
  ln_f32_2048x65536        LayerNorm fp32 long rows; x ~ N(3,1).
  ln_f32_8192x5000         LayerNorm fp32, N not a power of two; x ~ N(3,1).
  ln_f16_4096x8192         LayerNorm fp16 rows, the T3 drill's N; x ~ N(3,1).
  ln_f32_8192x5001         LayerNorm fp32, odd N: rows off 16-byte boundaries.
  add_*                    the fused residual add + norm on the shape and
                           recipe of the workload it names: the residual r is
                           drawn from the same recipe, after the parameters.
  fp8_*                    the forward with an FP8 E4M3 output (static scale
                           `qscale`, chosen so the outputs span the format:
                           |y| <= 2 for the U(-1,1) rows, <= 16 for the
                           outlier rows) on the shape and recipe named.
  bwd_*                    the backward on the shape and recipe of the
                           workload it names: the upstream gradient
                           dy ~ N(0,1) is drawn after the parameters.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    op: str        # "ln" or "rms"
    dtype: str     # "f32", "bf16" or "f16"
    M: int
    N: int
    eps: float
    recipe: str    # key of the value distribution below
    add: bool = False  # fused residual add: h = x + r, y = norm(h)
    bwd: bool = False  # backward: dx (and the column gradients) from dy, x
    qscale: float = 0.0  # FP8 E4M3 output with this static scale (0: output in the row dtype)

    @property
    def torch_dtype(self) -> torch.dtype:
        return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[self.dtype]

    @property
    def elem_size(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def fp8(self) -> bool:
        return self.qscale > 0

    @property
    def row_tensors(self) -> int:
        """[M, N] tensors one call moves: x, y; with the fused add also r, h;
        backward: dy, x, dx."""
        return 4 if self.add else 3 if self.bwd else 2

    @property
    def row_bytes(self) -> int:
        """HBM bytes per element of the [M, N] tensors one call moves (an
        FP8 output is one byte per element)."""
        s = self.elem_size
        return self.row_tensors * s - (s - 1 if self.fp8 else 0)

    def algorithmic_bytes(self, M: int | None = None) -> int:
        """HBM bytes one call must move. Forward: read x (and r), write y
        (and h), read the per-column parameters, write 8 B of statistics per
        row (LayerNorm). Backward: read dy and x, write dx, read gamma (w)
        and, for LayerNorm, the 8 B of statistics per row; write the fp32
        column gradients (dgamma and dbeta, or dw)."""
        M = self.M if M is None else M
        s = self.elem_size
        if self.bwd:
            stats = 8 * M if self.op == "ln" else 0
            cols = (2 if self.op == "ln" else 1) * 4 * self.N
            return 3 * M * self.N * s + self.N * s + stats + cols
        params = 2 if self.op == "ln" else 1
        stats = 8 * M if self.op == "ln" else 0
        return self.row_bytes * M * self.N + params * self.N * s + stats + (4 if self.fp8 else 0)

    def scaled(self, M: int | None = None, N: int | None = None) -> "Workload":
        return Workload(self.name, self.op, self.dtype, M or self.M, N or self.N, self.eps, self.recipe, self.add,
                        self.bwd, self.qscale)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("ln_f32_128x1024", "ln", "f32", 128, 1024, 1e-5, "normal01"),
        Workload("rms_f32_8192x4096", "rms", "f32", 8192, 4096, 1e-6, "uniform_pm1"),
        Workload("ln_bf16_4096x8192_outliers", "ln", "bf16", 4096, 8192, 1e-5, "offset_outliers"),
        Workload("rms_bf16_65536x2048", "rms", "bf16", 65536, 2048, 1e-6, "uniform_pm1"),
        Workload("ln_f32_2048x65536", "ln", "f32", 2048, 65536, 1e-5, "normal31"),
        Workload("ln_f32_8192x5000", "ln", "f32", 8192, 5000, 1e-5, "normal31"),
        Workload("ln_f16_4096x8192", "ln", "f16", 4096, 8192, 1e-5, "normal31"),
        Workload("ln_f32_8192x5001", "ln", "f32", 8192, 5001, 1e-5, "normal31"),
        Workload("add_rms_f32_8192x4096", "rms", "f32", 8192, 4096, 1e-6, "uniform_pm1", True),
        Workload("add_rms_bf16_65536x2048", "rms", "bf16", 65536, 2048, 1e-6, "uniform_pm1", True),
        Workload("add_ln_bf16_4096x8192_outliers", "ln", "bf16", 4096, 8192, 1e-5, "offset_outliers", True),
        Workload("add_ln_f32_2048x65536", "ln", "f32", 2048, 65536, 1e-5, "normal31", True),
        Workload("fp8_rms_bf16_8192x4096", "rms", "bf16", 8192, 4096, 1e-6, "uniform_pm1", qscale=2 / 448),
        Workload("fp8_ln_bf16_4096x8192_outliers", "ln", "bf16", 4096, 8192, 1e-5, "offset_outliers",
                 qscale=16 / 448),
        Workload("fp8_add_rms_bf16_8192x4096", "rms", "bf16", 8192, 4096, 1e-6, "uniform_pm1", True, qscale=2 / 448),
        Workload("bwd_rms_f32_8192x4096", "rms", "f32", 8192, 4096, 1e-6, "uniform_pm1", bwd=True),
        Workload("bwd_ln_bf16_4096x8192_outliers", "ln", "bf16", 4096, 8192, 1e-5, "offset_outliers", bwd=True),
        Workload("bwd_rms_bf16_65536x2048", "rms", "bf16", 65536, 2048, 1e-6, "uniform_pm1", bwd=True),
        Workload("bwd_ln_f32_8192x5000", "ln", "f32", 8192, 5000, 1e-5, "normal31", bwd=True),
        Workload("bwd_ln_f32_2048x65536", "ln", "f32", 2048, 65536, 1e-5, "normal31", bwd=True),
    ]
}

BENCH_WORKLOAD = "rms_f32_8192x4096"

# The forward configurations the headline metric is quoted on: the ROCm
# LayerNorm README's 128 x 1024 example, the RMSNorm post's B*T x C shapes,
# the T3 drill's N = 8192 with the cancellation recipe, and the long and the
# non-power-of-two LayerNorm rows.
BASELINE_CONFIGS = ("ln_f32_128x1024", "rms_f32_8192x4096", "ln_bf16_4096x8192_outliers", "rms_bf16_65536x2048",
                    "ln_f32_2048x65536", "ln_f32_8192x5000")


def _draw(recipe: str, M: int, N: int, g: torch.Generator) -> torch.Tensor:
    if recipe == "normal01":
        return torch.randn(M, N, generator=g)
    if recipe == "normal31":
        return torch.randn(M, N, generator=g) + 3.0
    if recipe == "uniform_pm1":
        return torch.rand(M, N, generator=g) * 2.0 - 1.0
    if recipe == "offset_outliers":
        offset = torch.rand(M, 1, generator=g) * 900.0 + 100.0
        x = offset + torch.randn(M, N, generator=g) * 0.01
        n_out = max(1, round(0.01 * N))
        cols = torch.randperm(N, generator=g)[:n_out]
        signs = torch.where(torch.rand(n_out, generator=g) < 0.5, -1.0, 1.0)
        x[:, cols] = signs * 300.0
        return x
    raise KeyError(recipe)


def generate(w: Workload, seed: int = 0) -> dict[str, torch.Tensor]:
    """CPU tensors for one workload: {"x", "gamma", "beta"} (LayerNorm) or
    {"x", "w"} (RMSNorm), plus "r" for the fused add and "dy" for the
    backward, all in the workload's dtype, drawn in a fixed order from one
    seeded CPU generator."""
    g = torch.Generator().manual_seed(seed)
    M, N = w.M, w.N
    out = {"x": _draw(w.recipe, M, N, g)}
    if w.op == "ln":
        out["gamma"] = torch.rand(N, generator=g) + 0.5
        out["beta"] = torch.rand(N, generator=g) * 0.2 - 0.1
    else:
        out["w"] = torch.rand(N, generator=g)
    if w.add:
        out["r"] = _draw(w.recipe, M, N, g)
    if w.bwd:
        out["dy"] = torch.randn(M, N, generator=g)
    return {k: v.to(w.torch_dtype).contiguous() for k, v in out.items()}


def lattice(rows: int, N: int, row0: int = 0, device="cpu", dtype=torch.float32) -> torch.Tensor:
    """Deterministic counter-based pattern for inputs too large to draw on the
    host: value(r, c) = ((r*7919 + c*104729) mod 65536)/16384 + 1, in [1, 5), computed
    in exact int64 arithmetic, so the host and the device produce bit-identical
    rows. Used for sampled checks of very large launches."""
    r = torch.arange(row0, row0 + rows, device=device, dtype=torch.int64).unsqueeze(1)
    c = torch.arange(N, device=device, dtype=torch.int64).unsqueeze(0)
    v = (r * 7919 + c * 104729) % 65536
    return (v.to(torch.float32) / 16384.0 + 1.0).to(dtype)
