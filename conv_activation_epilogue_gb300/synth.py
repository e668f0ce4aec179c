"""Seeded synthetic inputs and the workload table.

This module holds no arithmetic of the fused operator: it only draws the input
tensors (as 16-bit codes and fp32 biases) that both the CUDA path and the
oracle consume, and names the workloads with their sizes.  It imports nothing
but numpy, so the oracle's tests can use it without touching the product.

Random numbers: SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used counter-style: element e
of stream s is ``mix(s + (e + 1) * 0x9E3779B97F4A7C15)`` with the published
finaliser ``mix``.  Uniform doubles take the top 53 bits.  Normals use the
Box-Muller transform on consecutive pairs.  Values are then rounded to the
input dtype: float16 by numpy's round-to-nearest-even conversion, bfloat16 by
rounding to float32 and then to the upper 16 bits with round-to-nearest-even.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def splitmix64(stream: int, n: int) -> np.ndarray:
    """The first n outputs of SplitMix64 seeded with `stream` (uint64 array)."""
    out = np.empty(n, dtype=np.uint64)
    s = np.uint64(stream & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for lo in range(0, n, _CHUNK):
            hi = min(n, lo + _CHUNK)
            z = np.arange(lo + 1, hi + 1, dtype=np.uint64) * _GAMMA + s
            z = (z ^ (z >> np.uint64(30))) * _M1
            z = (z ^ (z >> np.uint64(27))) * _M2
            out[lo:hi] = z ^ (z >> np.uint64(31))
    return out


def uniform(stream: int, shape, lo: float, hi: float) -> np.ndarray:
    n = int(np.prod(shape))
    u = (splitmix64(stream, n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return (lo + (hi - lo) * u).reshape(shape)


def normal(stream: int, shape, std: float) -> np.ndarray:
    n = int(np.prod(shape))
    m = n + (n & 1)
    u = (splitmix64(stream, m) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    u1 = 1.0 - u[0::2]                      # (0, 1]
    u2 = u[1::2]
    rad = np.sqrt(-2.0 * np.log(u1))
    g = np.empty(m, dtype=np.float64)
    g[0::2] = rad * np.cos(2.0 * np.pi * u2)
    g[1::2] = rad * np.sin(2.0 * np.pi * u2)
    return (std * g[:n]).reshape(shape)


def to_codes(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float64 values to 16-bit codes of `dtype` ('f16' or 'bf16')."""
    if dtype == "f16":
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32)
        u = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
        return (u >> np.uint32(16)).astype(np.uint16)
    raise ValueError(f"unknown 16-bit dtype {dtype!r}")


def draw(stream: int, shape, dist) -> np.ndarray:
    kind = dist[0]
    if kind == "uniform":
        return uniform(stream, shape, dist[1], dist[2])
    if kind == "normal":
        return normal(stream, shape, dist[1])
    raise ValueError(kind)


def stream_id(seed: int, tensor: int) -> int:
    return seed * 0x1000 + tensor


# tensor ids inside a workload's seed
T_A, T_B, T_BIAS, T_X, T_W, T_CBIAS = 1, 2, 3, 4, 5, 6


@dataclass(frozen=True)
class GemmWorkload:
    name: str
    M: int
    N: int
    K: int
    ab_dtype: str          # 'f16' | 'bf16'
    c_dtype: str           # 'f32' | 'f16' | 'bf16'
    act: str               # 'none' | 'relu' | 'leaky_relu' | 'tanh'
    alpha: float
    seed: int
    a_dist: tuple = ("uniform", -1.0, 1.0)
    b_dist: tuple = ("uniform", -1.0, 1.0)
    bias_dist: tuple = ("uniform", -1.0, 1.0)

    kind: str = field(default="gemm", init=False)

    def inputs(self, with_bias: bool = True) -> dict:
        A = to_codes(draw(stream_id(self.seed, T_A), (self.M, self.K), self.a_dist), self.ab_dtype)
        B = to_codes(draw(stream_id(self.seed, T_B), (self.K, self.N), self.b_dist), self.ab_dtype)
        bias = (draw(stream_id(self.seed, T_BIAS), (self.N,), self.bias_dist).astype(np.float32)
                if with_bias else None)
        return {"A": A, "B": B, "bias": bias}


@dataclass(frozen=True)
class ConvWorkload:
    name: str
    N: int
    C: int
    H: int
    W: int
    Co: int
    kh: int
    kw: int
    stride: tuple
    pads: tuple            # (top, bottom, left, right)
    dilation: tuple
    dtype: str             # input dtype 'f16' | 'bf16'
    out_dtype: str
    act: str
    alpha: float
    seed: int
    x_std: float = 1.0
    bias_dist: tuple = ("uniform", -0.1, 0.1)
    x_seed: int | None = None
    w_tensor: int = T_W

    kind: str = field(default="conv", init=False)

    def inputs(self, with_bias: bool = True) -> dict:
        xs = self.seed if self.x_seed is None else self.x_seed
        x = to_codes(normal(stream_id(xs, T_X), (self.N, self.C, self.H, self.W), self.x_std), self.dtype)
        fan_in = self.C * self.kh * self.kw
        w = to_codes(normal(stream_id(self.seed, self.w_tensor), (self.Co, self.C, self.kh, self.kw),
                            (1.0 / fan_in) ** 0.5), self.dtype)
        bias = (draw(stream_id(self.seed, T_CBIAS), (self.Co,), self.bias_dist).astype(np.float32)
                if with_bias else None)
        return {"x": x, "w": w, "bias": bias}


# The eight workloads of the hot path, named by what they are.
WORKLOADS = {
    w.name: w for w in [
        GemmWorkload("matmul_leakyrelu_1024x640x256_f16", 1024, 640, 256, "f16", "f32",
                     "leaky_relu", 0.01, seed=1),
        GemmWorkload("gemm_relu_4096x4096x4096_bf16", 4096, 4096, 4096, "bf16", "bf16",
                     "relu", 0.0, seed=2),
        ConvWorkload("conv3x3_s1p1d1_tanh_8x64x56x56_f16", 8, 64, 56, 56, 128, 3, 3,
                     (1, 1), (1, 1, 1, 1), (1, 1), "f16", "f16", "tanh", 0.0, seed=3),
        ConvWorkload("conv3x3_s2p2d2_tanh_16x128x64x64_bf16", 16, 128, 64, 64, 256, 3, 3,
                     (2, 2), (2, 2, 2, 2), (2, 2), "bf16", "bf16", "tanh", 0.0, seed=4),
        ConvWorkload("conv1x1_s2_tanh_16x128x64x64_bf16", 16, 128, 64, 64, 256, 1, 1,
                     (2, 2), (0, 0, 0, 0), (1, 1), "bf16", "bf16", "tanh", 0.0, seed=4,
                     w_tensor=7),
        GemmWorkload("gemm_leakyrelu_8192x8192x8192_bf16", 8192, 8192, 8192, "bf16", "bf16",
                     "leaky_relu", 0.2, seed=5),
        GemmWorkload("gemm_leakyrelu_16384x4096x1024_bf16", 16384, 4096, 1024, "bf16", "bf16",
                     "leaky_relu", 0.2, seed=6),
        GemmWorkload("gemm_leakyrelu_128x8192x8192_bf16", 128, 8192, 8192, "bf16", "bf16",
                     "leaky_relu", 0.2, seed=7),
    ]
}

# The one the throughput metric is quoted on.
HEADLINE = "gemm_leakyrelu_8192x8192x8192_bf16"
