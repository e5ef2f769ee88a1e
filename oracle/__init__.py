"""The oracle: plain, slow, obviously correct CPU attention in fp64.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import anything from here.  The product
package never does, and nothing here imports the product package.

Contents
--------
* ``attention`` / ``attention_rows`` -- the three-pass definition in C
  (``attention.c``), on the bf16 bits the GPU receives, widened to fp64.
* ``online`` -- the pages' online-softmax recurrences, blocked attention and the
  partial-result merge, in numpy (``online.py``).
* ``backward`` -- gradients of attention in fp64 (``backward.py``).
* ``paged`` -- attention over a paged key/value cache (``paged.py``).
* ``fp8`` -- E4M3 quantisation (with the Hadamard rotation of incoherent
  processing) and attention on the dequantised inputs (``fp8.py``).

Pinned by ``tests/test_oracle_pins.py``; every function has at least one pin
that does not re-derive it from itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import backward, online  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False, out: str | None = None, defines: tuple = ()) -> str:
    """Compile ``attention.c`` into a shared library with gcc; returns its path."""
    out = out or _LIB_PATH
    src = os.path.join(_HERE, "attention.c")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           *[f"-D{d}" for d in defines], "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def load(path: str | None = None):
    """Load (building if needed) the C oracle library."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    f = lib.oracle_attention_rows
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_float, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    g = lib.oracle_attention_rows_f64
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_double, ctypes.c_int,
                  ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    if path is None:
        _lib = lib
    return lib


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy uint16)")
    return a


def attention_rows(Q, K, V, scale, causal, rows=None, nthreads=None, lib=None):
    """Attention outputs for selected rows.

    Q: uint16 [B,H,Nq,d] (bf16 bits); K, V: uint16 [B,H,Nk,d].
    rows: flat row ids (b*H + h)*Nq + i, or None for every row.
    Returns (O [nrows, d] fp64, LSE [nrows] fp64).
    """
    Q, K, V = _u16(Q), _u16(K), _u16(V)
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    if K.shape != (B, H, Nk, d) or V.shape != (B, H, Nk, d):
        raise ValueError("shape mismatch")
    if rows is None:
        nrows = B * H * Nq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
    O = np.empty((nrows, d), dtype=np.float64)
    LSE = np.empty(nrows, dtype=np.float64)
    nthreads = nthreads or os.cpu_count() or 1
    rc = (lib or load()).oracle_attention_rows(
        Q.ctypes.data, K.ctypes.data, V.ctypes.data, B, H, Nq, Nk, d,
        ctypes.c_float(scale), int(bool(causal)),
        None if rows_arr is None else rows_arr.ctypes.data, nrows,
        O.ctypes.data, LSE.ctypes.data, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows failed with {rc}")
    return O, LSE


def attention(Q, K, V, scale, causal, nthreads=None, lib=None):
    """Full attention: O [B,H,Nq,d] fp64 and LSE [B,H,Nq] fp64."""
    B, H, Nq, d = Q.shape
    O, LSE = attention_rows(Q, K, V, scale, causal, None, nthreads, lib)
    return O.reshape(B, H, Nq, d), LSE.reshape(B, H, Nq)


def attention_rows_f64(Q, K, V, scale, causal, rows=None, nthreads=None, lib=None):
    """attention_rows on fp64 inputs (same layouts); `scale` is used as given."""
    Q, K, V = (np.ascontiguousarray(a, dtype=np.float64) for a in (Q, K, V))
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    if K.shape != (B, H, Nk, d) or V.shape != (B, H, Nk, d):
        raise ValueError("shape mismatch")
    if rows is None:
        nrows, rows_arr = B * H * Nq, None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
    O = np.empty((nrows, d), dtype=np.float64)
    LSE = np.empty(nrows, dtype=np.float64)
    rc = (lib or load()).oracle_attention_rows_f64(
        Q.ctypes.data, K.ctypes.data, V.ctypes.data, B, H, Nq, Nk, d, float(scale), int(bool(causal)),
        None if rows_arr is None else rows_arr.ctypes.data, nrows, O.ctypes.data, LSE.ctypes.data,
        int(nthreads or os.cpu_count() or 1))
    if rc != 0:
        raise RuntimeError(f"oracle_attention_rows_f64 failed with {rc}")
    return O, LSE


def bf16_bits_to_f64(a) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64 (for numpy-side oracle pieces)."""
    a = _u16(a)
    return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


from . import fp8, paged  # noqa: E402,F401  (use bf16_bits_to_f64 / attention_rows_f64 above)
