"""Seeded synthetic inputs shared by the oracle-side tests and the CUDA path.

This module draws the bf16 tensors that both sides consume. It holds none of the
attention arithmetic: only a counter-based uniform generator, a Gaussian transform,
the fp32 -> bf16 rounding of the drawn values, and the table of workload shapes.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; the 64-bit finaliser as published by Vigna). The n-th draw
of a stream is the finaliser applied to ``base + (n + 1) * GOLDEN`` with ``base``
derived from ``(seed, stream)``, so any element can be regenerated on its own.
Normals: Box-Muller in fp64 (Box and Muller, 1958), both the cosine and the sine
branch. Values are scaled by sigma, rounded to fp32, then rounded to bf16 with
round-to-nearest-even. The same bf16 bytes go to the GPU and to the oracle, which
widens them exactly to fp64 (the fp64-from-the-same-quantised-bytes discipline of
the Rigel paper, section 3 "Methodology", the checksum gate).
"""
from __future__ import annotations

import dataclasses
import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Per-tensor substreams.
STREAM_Q, STREAM_K, STREAM_V, STREAM_DO = 0, 1, 2, 3


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _stream_base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([np.uint64(seed) * GOLDEN + np.uint64(stream) + np.uint64(1)], dtype=np.uint64)
    return _mix(s)[0]


def uniform_u64(seed: int, stream: int, n: int, start: int = 0) -> np.ndarray:
    """Draws ``start .. start+n-1`` of the (seed, stream) sequence as uint64."""
    base = _stream_base(seed, stream)
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(base + idx * GOLDEN)


def normal_f64(seed: int, stream: int, n: int) -> np.ndarray:
    """n standard normals in fp64 via Box-Muller on pairs of 53-bit uniforms."""
    pairs = (n + 1) // 2
    u = uniform_u64(seed, stream, 2 * pairs)
    # 53-bit uniforms in (0, 1]: (x >> 11 + 1) * 2^-53
    f = ((u >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u1, u2 = f[0::2], f[1::2]
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * np.pi * u2
    out = np.empty(2 * pairs, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:n]


def f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    bias = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    with np.errstate(over="ignore"):
        return ((b + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def normal_bf16_bits(seed: int, stream: int, shape, sigma: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    x = (normal_f64(seed, stream, n) * sigma).astype(np.float32)
    return f32_to_bf16_bits(x).reshape(shape)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention workload: shapes, value distributions and seed."""
    name: str
    B: int
    H: int
    T: int
    d: int
    sigma_q: float = 1.0
    sigma_k: float = 1.0
    sigma_v: float = 1.0
    sigma_do: float = 1.0
    causal: bool = True
    seed: int = 1000

    @property
    def scale(self) -> float:
        return float(1.0 / np.sqrt(self.d))

    @property
    def shape(self):
        return (self.B, self.H, self.T, self.d)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: a tiny case, then shapes of the 12M, ~100M and 205M-parameter
# models of the Forge paper (section "Results" and RESEARCH.md section 6), and a
# long-context stress with peaked softmax (Q, K ~ N(0, 3^2)).
WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 64, 32, seed=1000),
    "gpt12m": Workload("gpt12m", 8, 6, 256, 64, seed=1001),
    "gpt100m": Workload("gpt100m", 8, 12, 1024, 64, sigma_do=0.1, seed=1002),
    "gpt205m": Workload("gpt205m", 4, 16, 2048, 64, sigma_do=0.1, seed=1003),
    "long8k": Workload("long8k", 1, 16, 8192, 128, sigma_q=3.0, sigma_k=3.0, seed=1004),
}


def make_inputs(w: Workload):
    """bf16 bit patterns (uint16, [B,H,T,d]) for q, k, v and dO."""
    return {
        "q": normal_bf16_bits(w.seed, STREAM_Q, w.shape, w.sigma_q),
        "k": normal_bf16_bits(w.seed, STREAM_K, w.shape, w.sigma_k),
        "v": normal_bf16_bits(w.seed, STREAM_V, w.shape, w.sigma_v),
        "do": normal_bf16_bits(w.seed, STREAM_DO, w.shape, w.sigma_do),
    }
