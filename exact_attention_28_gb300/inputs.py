"""Seeded synthetic inputs shared by the tests, the oracle runs and the bench.

This module holds no attention arithmetic: it only draws numbers.  Both the
CUDA path and the oracle consume the bf16 bit patterns it returns, so a parity
test compares the two on identical inputs.

Generator (counter-based, so any element can be drawn independently):

* SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): the k-th output of the stream with seed ``s`` is
  mix(s + (k+1) * 0x9E3779B97F4A7C15 mod 2^64) with the published 64-bit
  finaliser ``mix``.
* Box-Muller (G. Box, M. Muller, 1958): outputs 2i and 2i+1 give
  u1 = ((x >> 11) + 1) / 2^53 in (0, 1] and u2 = (x >> 11) / 2^53 in [0, 1),
  then z_{2i} = r cos(2 pi u2), z_{2i+1} = r sin(2 pi u2), r = sqrt(-2 ln u1).
* value = sigma * z, rounded to fp32, then to bf16 with round-to-nearest-even.

Workloads: the five attention-forward shapes this library is measured on, the
ragged-tail variant of the short-query shape (Nk = 8192 + 37), and a decoding
shape for the split-key path.  Q, K, V of workload number c use seeds
1000*c + 0, 1, 2.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, first: int, count: int) -> np.ndarray:
    """Outputs first..first+count-1 of the SplitMix64 stream with this seed."""
    k = np.arange(first + 1, first + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + k * _GAMMA)


def fp32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_fp32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, shape, sigma: float = 1.0, chunk_pairs: int = 1 << 21) -> np.ndarray:
    """Seeded N(0, sigma^2) samples as bf16 bit patterns (uint16) of `shape`."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    npairs = (n + 1) // 2
    for p0 in range(0, npairs, chunk_pairs):
        p1 = min(npairs, p0 + chunk_pairs)
        x = splitmix64(seed, 2 * p0, 2 * (p1 - p0))
        u1 = ((x[0::2] >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * 2.0 ** -53
        u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        r = np.sqrt(-2.0 * np.log(u1))
        theta = 2.0 * math.pi * u2
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(theta)
        z[1::2] = r * np.sin(theta)
        lo, hi = 2 * p0, min(n, 2 * p1)
        out[lo:hi] = fp32_to_bf16_bits((sigma * z[: hi - lo]).astype(np.float32))
    return out.reshape(shape)


@dataclass(frozen=True)
class Workload:
    name: str
    index: int          # seed base: 1000 * index
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    sigma_q: float = 1.0
    sigma_k: float = 1.0
    sigma_v: float = 1.0

    @property
    def scale(self) -> float:
        """1/sqrt(d) as the fp32 value passed to the kernel."""
        return float(np.float32(1.0 / math.sqrt(self.d)))

    @property
    def flops(self) -> int:
        """4*B*H*Nq*Nk*d, halved when causal (the convention the metric uses)."""
        f = 4 * self.B * self.H * self.Nq * self.Nk * self.d
        return f // 2 if self.causal else f

    @property
    def algorithmic_bytes(self) -> int:
        """One read of Q, K, V and one write of O (bf16) and LSE (fp32)."""
        bh = self.B * self.H
        return bh * (2 * self.Nq * self.d * 2 + 2 * self.Nk * self.d * 2 + 4 * self.Nq)

    def shapes(self):
        return ((self.B, self.H, self.Nq, self.d), (self.B, self.H, self.Nk, self.d))


WORKLOADS = {
    w.name: w
    for w in [
        Workload("single_head_n256_d64", 1, 1, 1, 256, 256, 64, False),
        Workload("causal_b4_h16_n1024_d64", 2, 4, 16, 1024, 1024, 64, True),
        Workload("b2_h16_n4096_d128", 3, 2, 16, 4096, 4096, 128, False),
        Workload("causal_h32_n16384_d128_sigma2", 4, 1, 32, 16384, 16384, 128, True,
                 sigma_q=2.0, sigma_k=2.0, sigma_v=1.0),
        Workload("b8_h32_q128_kv8192_d128", 5, 8, 32, 128, 8192, 128, False),
        Workload("b8_h32_q128_kv8229_d128", 5, 8, 32, 128, 8229, 128, False),
        # decoding: one query per head against a long key/value cache, the case
        # the split-key path exists for (32 work items without splitting)
        Workload("decode_b1_h32_q1_kv32768_d128", 6, 1, 32, 1, 32768, 128, False),
    ]
}


def make_inputs(w: Workload):
    """(Q, K, V) bf16 bit arrays for a workload, and its fp32 scale."""
    qs, ks = w.shapes()
    q = normal_bf16(1000 * w.index + 0, qs, w.sigma_q)
    k = normal_bf16(1000 * w.index + 1, ks, w.sigma_k)
    v = normal_bf16(1000 * w.index + 2, ks, w.sigma_v)
    return q, k, v, w.scale


def custom_inputs(seed: int, B: int, H: int, Nq: int, Nk: int, d: int,
                  sigma=(1.0, 1.0, 1.0)):
    """Seeded bf16 inputs of an arbitrary shape (edge-case tests)."""
    q = normal_bf16(seed + 0, (B, H, Nq, d), sigma[0])
    k = normal_bf16(seed + 1, (B, H, Nk, d), sigma[1])
    v = normal_bf16(seed + 2, (B, H, Nk, d), sigma[2])
    return q, k, v
