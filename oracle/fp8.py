"""FP8 (E4M3) quantisation and attention on the dequantised inputs: the
oracle for the FP8 forward.

TEST INFRASTRUCTURE ONLY (imported by the tests and the bench's CPU leg,
never by the product path).

Follows "9.4 FlashAttention 与 FlashMLA" section 9.4.4: FlashAttention-3 runs
attention in FP8 (E4M3 / E5M2) and, to soften the precision loss, multiplies
Q and K by a random orthogonal matrix before quantising them ("incoherent
processing"), so that quantisation error is spread evenly over the channels.
The page names the technique only; the readings taken here:

* Format: E4M3 as the OCP 8-bit floating point specification defines it --
  1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, subnormals below
  2^-6, no infinities, S.1111.111 is NaN, largest finite magnitude 448.
* Scaling: one scale per (batch, head) tensor.  x ~ code * descale, codes by
  round-to-nearest-even on the value scaled so that the largest magnitude
  maps to 448 (saturating at +-448).
* Rotation: the same M = D H / sqrt(d) for Q and K (so (QM)(KM)^T = Q K^T),
  with D a diagonal of random signs (an input: the random numbers are drawn
  by the caller) and H the Sylvester-Hadamard matrix, applied with the fast
  Walsh-Hadamard transform (radix-2 butterflies (a, b) -> (a + b, a - b) at
  strides 1, 2, 4, ...; Fino and Algazi, 1976).  The 1/sqrt(d) is folded into
  descale.  V is not rotated.
* The codes are decided in fp32, the precision the GPU decides them in:
  u = butterflies of x * sign in fp32 (exact sign flips, fp32 adds),
  amax = max |u|, inv = fp32(448 / amax), code = RNE_e4m3(fp32(u * inv)),
  descale = fp32(amax / 448) (times fp32(1/sqrt(d)) when rotated, in fp32);
  a head of zeros gets codes 0 and descale 1.
* V is stored transposed, [B*H][d][N rounded up to 16] with zero padding,
  so that the keys are the contiguous (reduction) dimension of P V.
* Attention: the exact three-pass definition in fp64 on the dequantised
  inputs code * descale.  The kernel's own approximation, P rounded to E4M3
  before P V (P in V's type, as the bf16 path casts P to bf16), is not part
  of the definition; the tolerance accounts for it.
"""
from __future__ import annotations

import math

import numpy as np

from . import attention_rows_f64


def _decode_table() -> np.ndarray:
    v = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            v[code] = np.nan
        elif e == 0:
            v[code] = sign * (m / 8.0) * 2.0 ** (1 - 7)     # subnormal
        else:
            v[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return v


E4M3 = _decode_table()          # value of every code
E4M3_MAX = 448.0


def decode_e4m3(codes) -> np.ndarray:
    """fp64 values of E4M3 codes (uint8)."""
    return E4M3[np.asarray(codes, dtype=np.uint8)]


def encode_e4m3(x, chunk: int = 1 << 15) -> np.ndarray:
    """E4M3 codes of finite values x: round to nearest, ties to the even
    code, magnitudes above 448 saturate to 448; the sign is kept (so -0 and
    negative values that round to zero give 0x80).  By exhaustive search over
    the 127 non-negative finite codes."""
    x = np.asarray(x, dtype=np.float64)
    flat = x.reshape(-1)
    out = np.empty(flat.size, dtype=np.uint8)
    mags = E4M3[:127]                                  # codes 0x00..0x7E, ascending
    even = (np.arange(127) % 2 == 0)
    for c0 in range(0, flat.size, chunk):
        a = np.minimum(np.abs(flat[c0:c0 + chunk]), E4M3_MAX)
        dist = np.abs(a[:, None] - mags[None, :])
        best = dist.min(axis=1, keepdims=True)
        cand = dist == best
        # among the nearest codes (one, or two on a tie) prefer the even one
        score = cand * (1 + even[None, :])
        code = score.argmax(axis=1).astype(np.uint8)
        neg = np.signbit(flat[c0:c0 + chunk])
        out[c0:c0 + chunk] = code | (neg.astype(np.uint8) << 7)
    return out.reshape(x.shape)


def fwht_f32(u) -> np.ndarray:
    """Unnormalised fast Walsh-Hadamard transform along the last axis, in
    fp32: log2(d) stages of butterflies (a, b) -> (a + b, a - b) at strides
    1, 2, 4, ..., each a single fp32 add or subtract."""
    u = np.asarray(u, dtype=np.float32)
    d = u.shape[-1]
    if d & (d - 1):
        raise ValueError("d must be a power of two")
    lead = u.shape[:-1]
    h = 1
    while h < d:
        v = u.reshape(*lead, d // (2 * h), 2, h)
        a, b = v[..., 0, :], v[..., 1, :]
        u = np.stack([a + b, a - b], axis=-2).reshape(*lead, d)
        h *= 2
    return u


def rotation_matrix(signs) -> np.ndarray:
    """M = D H / sqrt(d) in fp64 (for pins; quantise() uses the transform)."""
    from scipy.linalg import hadamard
    s = np.asarray(signs, dtype=np.float64)
    d = s.size
    return (s[:, None] * hadamard(d)) / math.sqrt(d)


def quantize(x_bits, signs=None, transpose: bool = False):
    """Per-(batch, head) E4M3 quantisation of bf16 inputs.

    x_bits: uint16 bf16 bits [B, H, N, d]; signs: None or d values +-1 (the
    rotation); transpose: return the codes as [B, H, d, ceil16(N)].
    Returns (codes uint8, descale float32 [B, H])."""
    from . import bf16_bits_to_f64
    x = bf16_bits_to_f64(x_bits).astype(np.float32)              # exact
    B, H, N, d = x.shape
    if signs is not None:
        s = np.asarray(signs, dtype=np.float32)
        u = fwht_f32(x * s)                                       # sign flips are exact
    else:
        u = x
    amax = np.abs(u).reshape(B, H, -1).max(axis=2).astype(np.float32)
    live = amax > 0
    inv = np.where(live, np.float32(E4M3_MAX) / np.where(live, amax, np.float32(1)), np.float32(0))
    inv = inv.astype(np.float32)
    scaled = (u * inv[:, :, None, None]).astype(np.float32)       # one fp32 rounding
    codes = encode_e4m3(scaled)
    descale = np.where(live, amax / np.float32(E4M3_MAX), np.float32(1)).astype(np.float32)
    if signs is not None:
        descale = np.where(live, descale * np.float32(1.0 / math.sqrt(d)), descale).astype(np.float32)
    if transpose:
        npad = -(-N // 16) * 16
        t = np.zeros((B, H, d, npad), dtype=np.uint8)
        t[:, :, :, :N] = codes.transpose(0, 1, 3, 2)
        codes = t
    return codes, descale


def dequantize(codes, descale, transposed: bool = False, n: int | None = None) -> np.ndarray:
    """code * descale in fp64, as [B, H, N, d] (un-transposing V)."""
    v = decode_e4m3(codes) * np.asarray(descale, dtype=np.float64)[:, :, None, None]
    if transposed:
        v = v[:, :, :, :n].transpose(0, 1, 3, 2)
    return np.ascontiguousarray(v)


def attention_fp8(q8, k8, vt8, dq, dk, dv, scale, causal, nk: int, rows=None, nthreads=None):
    """Exact attention (three-pass, fp64) on the dequantised FP8 inputs:
    q8, k8 [B, H, N, d] codes, vt8 [B, H, d, ceil16(nk)] codes, per-head
    descales; returns (O [rows, d], LSE [rows]) like attention_rows."""
    Q = dequantize(q8, dq)
    K = dequantize(k8, dk)
    V = dequantize(vt8, dv, transposed=True, n=nk)
    return attention_rows_f64(Q, K, V, float(np.float32(scale)), causal, rows=rows, nthreads=nthreads)
