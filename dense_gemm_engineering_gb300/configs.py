"""The five GEMM workloads: shapes, layouts, dtypes and input recipes.

Sources of the shapes:
  * 128 x 128 x 64: "TIRx GEMM on Blackwell", V1 (one tile, one MMA, no K loop).
  * 256 x 256 x 1024: "TIRx GEMM on Blackwell", V2 (the K loop reuses the same
    barrier across 16 chunks of 64).
  * 4096^3 A.Bt FP16: "TIRx GEMM on Blackwell", The short version / V3-V9
    (the headline measurement shape).
  * 8192 x 17408 x 5120 A.B BF16: "Choosing schedules and instructions for a
    backend", section 1 (the TileFoundry H200 workload, B stored K x N).
  * 3000 x 5000 x 4000 A.Bt FP16: a ragged shape, not a multiple of any tile,
    that exercises the out-of-bounds fill on loads and the clipped stores.

FP8 workloads (E4M3 inputs, BF16 output; "TIRx: A Unified Tile Primitive ML
Compiler", kernel performance: FP8 GEMMs with M = 8192 and model-derived weight
shapes, which the page does not list): the headline square shape in FP8, and
M = N = K = 8192.  The block-scaled (MX) workloads take the same two shapes
with one UE8M0 scale per 32 K elements of each row, scale bytes uniform in
[124, 130] (scales 2^-3 .. 2^3).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class GemmConfig:
    name: str
    layout: str  # "abt": D = A.Bt, B is N x K;  "ab": D = A.B, B is K x N
    M: int
    N: int
    K: int
    dtype: str  # input type: "f16" / "bf16" (also the output), or FP8 "e4m3" / "e5m2"
    dist: str  # "uniform" U[-1,1) or "normal" N(0, 0.02^2)
    seed: int
    out_dtype: str = ""  # FP8 inputs: the 16-bit output type ("" = dtype)
    alpha: float = 1.0  # FP8 inputs: D = alpha * A.Bt
    mx: bool = False  # FP8 inputs with one UE8M0 scale per 32 K elements of each row

    @property
    def is_fp8(self) -> bool:
        return self.dtype in ("e4m3", "e5m2")

    @property
    def out(self) -> str:
        return self.out_dtype or self.dtype

    @property
    def elem_bytes(self) -> int:
        return 1 if self.is_fp8 else 2

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> int:
        scales = (self.M + self.N) * -(-self.K // 32) if self.mx else 0
        return self.elem_bytes * (self.M * self.K + self.N * self.K) + 2 * self.M * self.N + scales

    @property
    def rtol(self) -> float:
        # |got - ref| <= 1e-2 + rtol * |ref|, set by the 16-bit output type
        return 1e-3 if self.out == "f16" else 8e-3

    atol: float = 1e-2


CONFIGS = [
    GemmConfig("single_tile_128x128x64_f16_abt", "abt", 128, 128, 64, "f16", "uniform", 0),
    GemmConfig("kloop_256x256x1024_f16_abt", "abt", 256, 256, 1024, "f16", "uniform", 1),
    GemmConfig("square_4096x4096x4096_f16_abt", "abt", 4096, 4096, 4096, "f16", "uniform", 2),
    GemmConfig("rect_8192x17408x5120_bf16_ab", "ab", 8192, 17408, 5120, "bf16", "normal", 3),
    GemmConfig("ragged_3000x5000x4000_f16_abt", "abt", 3000, 5000, 4000, "f16", "uniform", 4),
]

FP8_CONFIGS = [
    GemmConfig("fp8_square_4096x4096x4096_e4m3_abt", "abt", 4096, 4096, 4096, "e4m3", "uniform",
               12, out_dtype="bf16"),
    GemmConfig("fp8_8192x8192x8192_e4m3_abt", "abt", 8192, 8192, 8192, "e4m3", "normal", 13,
               out_dtype="bf16"),
]

MX_CONFIGS = [
    GemmConfig("mx_square_4096x4096x4096_e4m3_abt", "abt", 4096, 4096, 4096, "e4m3", "uniform",
               22, out_dtype="bf16", mx=True),
    GemmConfig("mx_8192x8192x8192_e4m3_abt", "abt", 8192, 8192, 8192, "e4m3", "normal", 23,
               out_dtype="bf16", mx=True),
    # M = 8192 against a transformer MLP's weights (hidden 4096, inner 14336): the
    # widening projection (N = 14336, K = 4096) and the narrowing one (N = 4096,
    # K = 14336); the page names "model-derived weight shapes" without listing them
    GemmConfig("mx_8192x14336x4096_e4m3_abt", "abt", 8192, 14336, 4096, "e4m3", "normal", 24,
               out_dtype="bf16", mx=True),
    GemmConfig("mx_8192x4096x14336_e4m3_abt", "abt", 8192, 4096, 14336, "e4m3", "normal", 25,
               out_dtype="bf16", mx=True),
]

BY_NAME = {c.name: c for c in CONFIGS + FP8_CONFIGS + MX_CONFIGS}

# The measured workload: FP16 A.Bt at 4096^3.
HEADLINE = CONFIGS[2]
