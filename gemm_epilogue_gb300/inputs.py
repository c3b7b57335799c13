"""Seeded synthetic inputs for the fused GEMM + epilogue workloads.

This module only draws random numbers and stores them in the operand types.
It holds none of the method's arithmetic, and both the CUDA path's tests and
the oracle take their inputs from here.

Recipe (every workload): ``numpy.random.default_rng(seed)``; draws in the
order A (M x K), B (K x N), bias (N), then Y (M x N) for the gate; each draw is
float32 standard normal (or uniform for the FFN bias) times the stated scale,
then rounded once to the storage type (fp16 by numpy, bf16 by torch's CPU
conversion; both round to nearest even).  16-bit values are kept as raw
``uint16`` bit patterns so that the oracle decodes them itself.

The named workloads follow the shapes of the pages' examples: the 4096-square
layer of "Triton: Fused Matmul + Bias + ReLU (Epilogue Fusion)", the GLU block
(M = 1024, N = 21568) of "Optimizing GEMM + Activation on CDNA4 with TLX" at
K = 4096, an FFN up-projection, and decode-like skinny M.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

# element type codes (the oracle's codes)
F16, BF16, F32, E4M3 = 1, 2, 3, 4
TYPE_NAMES = {F16: "f16", BF16: "bf16", F32: "f32", E4M3: "e4m3"}
ELEM_BYTES = {F16: 2, BF16: 2, F32: 4, E4M3: 1}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    ab_type: int             # A, B (and Y) element type
    bias_type: int
    out_type: int
    epilogue: str            # "bias_relu" or "gate"
    scale: float             # A and B are N(0,1) * scale
    bias_dist: str           # "normal" or "uniform"  (uniform is U(-1, 1))
    seed: int
    y_dtype: int | None = None  # the gate's Y type when it differs from the operand type

    @property
    def y_type(self) -> int:
        return self.ab_type if self.y_dtype is None else self.y_dtype

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    def unavoidable_bytes(self) -> int:
        """A + B + bias + (Y) + out, each touched once."""
        es = ELEM_BYTES
        b = self.M * self.K * es[self.ab_type] + self.K * self.N * es[self.ab_type]
        b += self.N * es[self.bias_type] + self.M * self.N * es[self.out_type]
        if self.epilogue == "gate":
            b += self.M * self.N * es[self.y_type]
        return b


WORKLOADS = {
    "ragged_200x136x72": Workload("ragged_200x136x72", 200, 136, 72, F16, F32, F16,
                                  "bias_relu", 1.0 / math.sqrt(72.0), "normal", 0),
    "square_4096": Workload("square_4096", 4096, 4096, 4096, BF16, BF16, BF16,
                            "bias_relu", 1.0 / 64.0, "normal", 1),
    "glu_gate_1024x21568x4096": Workload("glu_gate_1024x21568x4096", 1024, 21568, 4096,
                                         F16, F16, F16, "gate", 1.0 / 64.0, "normal", 2),
    "ffn_up_8192x14336x4096": Workload("ffn_up_8192x14336x4096", 8192, 14336, 4096,
                                       BF16, BF16, BF16, "bias_relu", 1.0 / 64.0, "uniform", 3),
}
# The GLU block at the K values of the page's own measurements ("Optimizing GEMM + Activation on
# CDNA4 with TLX", "Configuration Details": M = 1024, N = 21568, fp16, K in {256, 512, 1024}).
for _k in (256, 512, 1024):
    WORKLOADS[f"glu_gate_1024x21568x{_k}"] = Workload(f"glu_gate_1024x21568x{_k}", 1024, 21568, _k,
                                                      F16, F16, F16, "gate", 1.0 / 64.0, "normal",
                                                      5)
# fp8 e4m3 operands (fp32 bias, bf16 out): the FFN up-projection and the square layer
WORKLOADS["ffn_up_fp8_8192x14336x4096"] = Workload("ffn_up_fp8_8192x14336x4096", 8192, 14336, 4096,
                                                   E4M3, F32, BF16, "bias_relu", 1.0 / 8.0,
                                                   "uniform", 6)
WORKLOADS["square_fp8_4096"] = Workload("square_fp8_4096", 4096, 4096, 4096, E4M3, F32, BF16,
                                        "bias_relu", 1.0 / 8.0, "normal", 7)
# the GLU block with the projection in fp8 and Y, out in fp16 ("Optimizing GEMM + Activation on
# CDNA4 with TLX", "Future Work": FP8 precision); fp32 bias
WORKLOADS["glu_gate_fp8_1024x21568x4096"] = Workload("glu_gate_fp8_1024x21568x4096", 1024, 21568,
                                                     4096, E4M3, F32, F16, "gate", 1.0 / 8.0,
                                                     "normal", 8, y_dtype=F16)
for _m in (1, 16, 64, 128):
    WORKLOADS[f"skinny_M{_m}_8192"] = Workload(f"skinny_M{_m}_8192", _m, 8192, 8192, BF16, BF16,
                                               BF16, "bias_relu", 1.0 / 90.0, "normal", 4)
# decode-like shapes with fp8 e4m3 operands (half the bytes of B), fp32 bias, bf16 out
for _m in (1, 16, 64, 128):
    WORKLOADS[f"skinny_fp8_M{_m}_8192"] = Workload(f"skinny_fp8_M{_m}_8192", _m, 8192, 8192, E4M3,
                                                   F32, BF16, "bias_relu", 1.0 / 8.0, "normal", 9)


def quantize(x: np.ndarray, t: int) -> np.ndarray:
    """Round float32/float64 values to storage type ``t`` once (RNE).

    Returns uint16 bit patterns for F16/BF16, uint8 for fp8 e4m3, float32 for F32.
    """
    if t == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if t == E4M3:
        import torch
        src = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
        return src.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
    if t == F16:
        return np.ascontiguousarray(x).astype(np.float16).view(np.uint16)
    if t == BF16:
        import torch
        src = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
        return src.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    raise ValueError(f"unknown type code {t}")


@dataclasses.dataclass
class Inputs:
    A: np.ndarray
    B: np.ndarray
    bias: np.ndarray
    Y: np.ndarray | None


def make(w: Workload, seed: int | None = None) -> Inputs:
    """Draw the inputs of workload ``w`` (optionally with another seed)."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    A = quantize(rng.standard_normal((w.M, w.K), dtype=np.float32) * np.float32(w.scale), w.ab_type)
    B = quantize(rng.standard_normal((w.K, w.N), dtype=np.float32) * np.float32(w.scale), w.ab_type)
    if w.bias_dist == "uniform":
        b = rng.uniform(-1.0, 1.0, w.N).astype(np.float32)
    else:
        b = rng.standard_normal(w.N, dtype=np.float32)
    bias = quantize(b, w.bias_type)
    Y = None
    if w.epilogue == "gate":
        Y = quantize(rng.standard_normal((w.M, w.N), dtype=np.float32), w.y_type)
    return Inputs(A, B, bias, Y)


def random_problem(M: int, N: int, K: int, ab_type: int, bias_type: int, seed: int,
                   scale: float | None = None, gate: bool = False,
                   y_type: int | None = None) -> Inputs:
    """Small seeded problem of any shape: A, B ~ N(0,1)/sqrt(K) (or ``scale``); Y (gate) of
    ``y_type``, by default the operand type."""
    rng = np.random.default_rng(seed)
    s = np.float32(scale if scale is not None else 1.0 / math.sqrt(max(K, 1)))
    A = quantize(rng.standard_normal((M, K), dtype=np.float32) * s, ab_type)
    B = quantize(rng.standard_normal((K, N), dtype=np.float32) * s, ab_type)
    bias = quantize(rng.standard_normal(N, dtype=np.float32), bias_type)
    yt = ab_type if y_type is None else y_type
    Y = quantize(rng.standard_normal((M, N), dtype=np.float32), yt) if gate else None
    return Inputs(A, B, bias, Y)


def integer_problem(M: int, N: int, K: int, ab_type: int, bias_type: int, seed: int,
                    lo: int = -3, hi: int = 3, gate: bool = False,
                    y_type: int | None = None) -> Inputs:
    """Small-integer inputs in [lo, hi] (exact in every type, exact sums for small K); Y (gate)
    of ``y_type``, by default the operand type."""
    rng = np.random.default_rng(seed)
    A = quantize(rng.integers(lo, hi + 1, (M, K)).astype(np.float32), ab_type)
    B = quantize(rng.integers(lo, hi + 1, (K, N)).astype(np.float32), ab_type)
    bias = quantize(rng.integers(2 * lo, 2 * hi + 1, N).astype(np.float32), bias_type)
    yt = ab_type if y_type is None else y_type
    Y = quantize(rng.integers(-2, 3, (M, N)).astype(np.float32), yt) if gate else None
    return Inputs(A, B, bias, Y)
