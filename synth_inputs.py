"""Seeded synthetic inputs for the tiled GEMM and the H-tiled convolution.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle.  It holds none of the method's arithmetic: it only draws random
numbers with numpy's PCG64 generator and rounds them to the storage dtype
(fp16 or bf16) once, on the host, so that both sides see the same quantised
values.

Workload recipes (one seed per workload, draws in row-major order, A before B,
x before w):

  gemm_512      M=N=K=512,  fp16 in, fp32 out, U[-1,1),          seed 0
  gemm_4096     M=N=K=4096, fp16 in, fp16 out, U[-1,1),          seed 1
  gemm_batched  b=16, M=N=2048, K=1024, bf16 in/out, N(0,1),      seed 2
  gemm_ragged   M=5000, N=3000, K=4096, bf16 in, fp32 out,
                N(0, 1/K) (standard deviation 1/sqrt(K)),         seed 3
  conv_htiled   x[8,64,224,224], w[128,64,3,3], stride 2, pad 1,
                dilation 1, tile_oh 16, fp16 in/out, U[-1,1),     seed 4

bf16 values are carried as their 16-bit patterns in ``numpy.uint16`` arrays,
because numpy has no bf16 type.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F16 = "f16"
BF16 = "bf16"
F32 = "f32"

DTYPE_BYTES = {F16: 2, BF16: 2, F32: 4}


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (via float32, round-to-nearest-even).

    The float64 -> float32 step rounds to nearest even (numpy's cast); the
    float32 -> bf16 step keeps the top 16 bits after adding the usual
    round-to-nearest-even bias.  Inputs are finite.
    """
    f32 = np.ascontiguousarray(x, dtype=np.float32)
    bits = f32.view(np.uint32).astype(np.uint64)
    bias = ((bits >> 16) & 1) + 0x7FFF
    return ((bits + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    u32 = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u32.view(np.float32).astype(np.float64)


def quantise(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 draws to the storage dtype (fp16 array or bf16 bits)."""
    if dtype == F16:
        return np.ascontiguousarray(x, dtype=np.float64).astype(np.float16)
    if dtype == BF16:
        return f64_to_bf16_bits(x)
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of a stored array (fp16, bf16 bits or fp32) to float64."""
    if dtype == BF16:
        return bf16_bits_to_f64(x)
    return np.asarray(x).astype(np.float64)


def draw(rng: np.random.Generator, dist: str, shape, scale: float = 1.0) -> np.ndarray:
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=shape)
    if dist == "normal":
        return rng.normal(0.0, scale, size=shape)
    raise ValueError(f"unknown distribution {dist!r}")


@dataclass(frozen=True)
class GemmWorkload:
    name: str
    b: int
    m: int
    n: int
    k: int
    in_dtype: str
    out_dtype: str
    dist: str
    seed: int
    scale: float = 1.0

    @property
    def flops(self) -> int:
        return 2 * self.b * self.m * self.n * self.k

    def a_shape(self):
        return (self.b, self.m, self.k) if self.b > 1 else (self.m, self.k)

    def b_shape(self):
        return (self.b, self.k, self.n) if self.b > 1 else (self.k, self.n)

    def c_shape(self):
        return (self.b, self.m, self.n) if self.b > 1 else (self.m, self.n)


@dataclass(frozen=True)
class ConvWorkload:
    name: str
    n: int
    c: int
    h: int
    w: int
    c_out: int
    kh: int
    kw: int
    sh: int
    sw: int
    ph: int
    pw: int
    dh: int
    dw: int
    tile_oh: int
    in_dtype: str
    out_dtype: str
    dist: str
    seed: int

    @property
    def oh(self) -> int:
        return (self.h + 2 * self.ph - (self.kh - 1) * self.dh - 1) // self.sh + 1

    @property
    def ow(self) -> int:
        return (self.w + 2 * self.pw - (self.kw - 1) * self.dw - 1) // self.sw + 1

    @property
    def flops(self) -> int:
        return 2 * self.n * self.c_out * self.oh * self.ow * self.c * self.kh * self.kw


WORKLOADS = {
    "gemm_512": GemmWorkload("gemm_512", 1, 512, 512, 512, F16, F32, "uniform", 0),
    "gemm_4096": GemmWorkload("gemm_4096", 1, 4096, 4096, 4096, F16, F16, "uniform", 1),
    "gemm_batched": GemmWorkload("gemm_batched", 16, 2048, 2048, 1024, BF16, BF16, "normal", 2),
    "gemm_ragged": GemmWorkload("gemm_ragged", 1, 5000, 3000, 4096, BF16, F32, "normal", 3,
                                scale=1.0 / 64.0),
    "conv_htiled": ConvWorkload("conv_htiled", 8, 64, 224, 224, 128, 3, 3, 2, 2, 1, 1, 1, 1, 16,
                                F16, F16, "uniform", 4),
}


def gemm_inputs(wl: GemmWorkload):
    """Quantised (A, B) for a GEMM workload, drawn A first then B."""
    rng = np.random.default_rng(wl.seed)
    a = quantise(draw(rng, wl.dist, wl.a_shape(), wl.scale), wl.in_dtype)
    b = quantise(draw(rng, wl.dist, wl.b_shape(), wl.scale), wl.in_dtype)
    return a, b


def conv_inputs(wl: ConvWorkload):
    """Quantised (x, w) for a convolution workload, NCHW and OIHW, x first."""
    rng = np.random.default_rng(wl.seed)
    x = quantise(draw(rng, wl.dist, (wl.n, wl.c, wl.h, wl.w)), wl.in_dtype)
    w = quantise(draw(rng, wl.dist, (wl.c_out, wl.c, wl.kh, wl.kw)), wl.in_dtype)
    return x, w


def random_matrix(seed: int, shape, dtype: str, dist: str = "uniform", scale: float = 1.0):
    """A quantised random array for ad-hoc test shapes."""
    rng = np.random.default_rng(seed)
    return quantise(draw(rng, dist, shape, scale), dtype)


def integer_matrix(seed: int, shape, dtype: str, lo: int = -2, hi: int = 2):
    """Integer-valued entries in [lo, hi], exact in fp16 and bf16."""
    rng = np.random.default_rng(seed)
    return quantise(rng.integers(lo, hi + 1, size=shape).astype(np.float64), dtype)
