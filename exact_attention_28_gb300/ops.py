"""ctypes binding of libfa_gb300.so: the C entry points under the same names.

Argument marshalling only -- every step of the computation runs in the CUDA
library.  There is no fallback: a missing library or a failing call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from .build import LIB_PATH

(FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_MISALIGNED, FA_ERR_CUDA, FA_ERR_TIMEOUT,
 FA_ERR_TOO_LARGE) = range(7)

_lib = None


class FAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(msg)
        self.status = status


def load_library(path: str | None = None):
    """Load the compiled library (build it first with __graft_entry__.build())."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise FileNotFoundError(
            f"{path} is missing: the CUDA library has not been built (run __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_host.restype = i
    lib.fa_host_groups.argtypes = [i, i, i, i, i, i]
    lib.fa_host_groups.restype = i
    lib.fa_fwd_test_missing_load.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_test_missing_load.restype = i
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp, ctypes.c_size_t, vp]
    lib.fa_fwd_splitkv.restype = i
    lib.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_splitkv_noalloc.restype = i
    lib.fa_splitkv_workspace.argtypes = [i, i, i, i, i, i, vp, vp]
    lib.fa_splitkv_workspace.restype = i
    lib.fa_fwd_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_paged.restype = i
    lib.fa_fwd_paged_splitkv.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, vp,
                                         ctypes.c_size_t, vp]
    lib.fa_fwd_paged_splitkv.restype = i
    lib.fa_quantize_fp8.argtypes = [vp, vp, vp, i, i, i, i, vp, i, vp]
    lib.fa_quantize_fp8.restype = i
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, ctypes.c_size_t, vp]
    lib.fa_bwd.restype = i
    lib.fa_bwd_workspace.argtypes = [i, i, i, i, i, vp]
    lib.fa_bwd_workspace.restype = i
    lib.fa_check_device_status.argtypes = [vp]
    lib.fa_check_device_status.restype = i
    lib.fa_schedule.argtypes = [i, i, i, i, i, i, i, i, vp, ctypes.c_int64, vp]
    lib.fa_schedule.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    if path == LIB_PATH:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().fa_status_string(status).decode()


def _check(status: int):
    if status != FA_OK:
        raise FAError(status, status_string(status))


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(getattr(stream, "cuda_stream", stream))


def _shape(q, k):
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    return B, H, Nq, Nk, d


def fa_fwd(q, k, v, o=None, lse=None, scale=None, causal=False, stream=None):
    """O, LSE = attention(q, k, v) on the GPU through the C ABI.

    q: bf16 [B,H,Nq,d], k/v: bf16 [B,H,Nk,d], contiguous CUDA tensors.
    Returns (o, lse); o bf16 [B,H,Nq,d], lse fp32 [B,H,Nq].
    """
    for t in (q, k, v):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
            raise TypeError("q, k, v must be contiguous bf16 CUDA tensors")
    B, H, Nq, Nk, d = _shape(q, k)
    if k.shape != (B, H, Nk, d) or v.shape != (B, H, Nk, d):
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(load_library().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                 B, H, Nq, Nk, d, scale, int(bool(causal)), _stream_handle(stream)))
    return o, lse


def fa_fwd_host(hq, hk, hv, ho, hlse, dq, dk, dv, do, dlse, scale, causal=False, stream=None):
    """End-to-end call from (pinned) host tensors through caller-owned device buffers."""
    B, H, Nq, Nk, d = _shape(hq, hk)
    _check(load_library().fa_fwd_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(),
                                      hlse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                      do.data_ptr(), dlse.data_ptr(), B, H, Nq, Nk, d, scale,
                                      int(bool(causal)), _stream_handle(stream)))


def fa_fwd_test_missing_load(q, k, v, item=0, scale=None, causal=False, stream=None):
    """fa_fwd with the first K tile of work item `item` never loaded (tests the
    bounded waits); returns the launch status, and the device status word then
    reads FA_ERR_TIMEOUT."""
    B, H, Nq, Nk, d = _shape(q, k)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return int(load_library().fa_fwd_test_missing_load(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                        lse.data_ptr(), B, H, Nq, Nk, d, scale, int(bool(causal)),
                                                        item, _stream_handle(stream)))


def host_groups(B, H, Nq, Nk, d, num_sms):
    """Number of head groups fa_fwd_host pipelines for these shapes (1: none)."""
    return int(load_library().fa_host_groups(B, H, Nq, Nk, d, num_sms))


def fa_fwd_paged(q, k_cache, v_cache, block_table, seq_lens, o=None, lse=None, scale=None, causal=False,
                 stream=None, num_splits=None, workspace=None):
    """Attention over a paged cache: k_cache, v_cache [num_blocks, H, block_size, d] bf16,
    block_table int32 [B, max_blocks], seq_lens int32 [B] (all CUDA tensors).

    num_splits: None runs fa_fwd_paged; an int (0 = the library's choice)
    runs fa_fwd_paged_splitkv with that many key slices, allocating the
    workspace unless one is given."""
    B, H, Nq, d = q.shape
    num_blocks, Hc, block_size, dc = k_cache.shape
    if Hc != H or dc != d or v_cache.shape != k_cache.shape:
        raise ValueError("cache shape mismatch")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    max_blocks = block_table.shape[1]
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if num_splits is None:
        _check(load_library().fa_fwd_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                           block_table.data_ptr(), seq_lens.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                           B, H, Nq, max_blocks, num_blocks, block_size, d, scale,
                                           int(bool(causal)), _stream_handle(stream)))
        return o, lse
    splits, nbytes = splitkv_workspace(B, H, Nq, max_blocks * block_size, d, causal, num_splits)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check(load_library().fa_fwd_paged_splitkv(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                               block_table.data_ptr(), seq_lens.data_ptr(), o.data_ptr(),
                                               lse.data_ptr(), B, H, Nq, max_blocks, num_blocks, block_size, d,
                                               scale, int(bool(causal)), splits, workspace.data_ptr(),
                                               workspace.numel() * workspace.element_size(), _stream_handle(stream)))
    return o, lse


def quantize_fp8(x, signs=None, transpose=False, stream=None):
    """E4M3 codes (torch.uint8) and per-head descale (fp32 [B, H]) of a bf16
    [B, H, N, d] CUDA tensor; `signs` (fp32 [d] of +-1, CUDA) rotates rows by
    diag(signs) H / sqrt(d); transpose gives [B, H, d, ceil16(N)]."""
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()):
        raise TypeError("x must be a contiguous bf16 CUDA tensor")
    B, H, N, d = x.shape
    if transpose:
        x8 = torch.empty((B, H, d, -(-N // 16) * 16), dtype=torch.uint8, device=x.device)
    else:
        x8 = torch.empty((B, H, N, d), dtype=torch.uint8, device=x.device)
    descale = torch.empty((B, H), dtype=torch.float32, device=x.device)
    _check(load_library().fa_quantize_fp8(x.data_ptr(), x8.data_ptr(), descale.data_ptr(), B, H, N, d,
                                          None if signs is None else signs.data_ptr(), int(bool(transpose)),
                                          _stream_handle(stream)))
    return x8, descale


def fa_fwd_fp8(q8, k8, vt8, descale_q, descale_k, descale_v, o=None, lse=None, scale=None, causal=False,
               stream=None):
    """Attention on E4M3 codes: q8 [B,H,Nq,d], k8 [B,H,Nk,d], vt8 [B,H,d,ceil16(Nk)]
    (torch.uint8 CUDA tensors) with per-head descales; returns bf16 O and fp32 LSE."""
    B, H, Nq, d = q8.shape
    Nk = k8.shape[2]
    if k8.shape != (B, H, Nk, d) or vt8.shape != (B, H, d, -(-Nk // 16) * 16):
        raise ValueError("shape mismatch")
    if o is None:
        o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q8.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(load_library().fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), descale_q.data_ptr(),
                                     descale_k.data_ptr(), descale_v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     B, H, Nq, Nk, d, scale, int(bool(causal)), _stream_handle(stream)))
    return o, lse


def fa_bwd(q, k, v, o, lse, do, dq=None, dk=None, dv=None, scale=None, causal=False, workspace=None,
           stream=None):
    """dQ, dK, dV of the attention forward (o, lse from fa_fwd) for upstream gradient do."""
    B, H, Nq, Nk, d = _shape(q, k)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    nb = ctypes.c_size_t(0)
    _check(load_library().fa_bwd_workspace(B, H, Nq, Nk, d, ctypes.byref(nb)))
    if workspace is None:
        workspace = torch.empty(nb.value, dtype=torch.uint8, device=q.device)
    _check(load_library().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                 do.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d,
                                 scale, int(bool(causal)), workspace.data_ptr(), workspace.numel(),
                                 _stream_handle(stream)))
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    """Autograd wrapper: forward through fa_fwd (saving O and LSE), backward
    through fa_bwd.  Marshalling only; both directions run in the library."""

    @staticmethod
    def forward(ctx, q, k, v, scale, causal):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        o, lse = fa_fwd(q, k, v, scale=scale, causal=causal)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.scale, ctx.causal = scale, causal
        ctx.mark_non_differentiable(lse)
        return o, lse

    @staticmethod
    def backward(ctx, do, _dlse):
        q, k, v, o, lse = ctx.saved_tensors
        dq, dk, dv = fa_bwd(q, k, v, o, lse, do.contiguous(), scale=ctx.scale, causal=ctx.causal)
        return dq, dk, dv, None, None


def flash_attention(q, k, v, causal=False, scale=None, return_lse=False):
    """softmax(scale * q k^T) v for bf16 CUDA tensors [B, H, N, d] (d = 64 or
    128), differentiable with respect to q, k and v.  scale defaults to
    1/sqrt(d); causal applies the top-left mask (key j visible to query i iff
    j <= i).  Returns O, or (O, LSE) with return_lse."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    o, lse = _Attention.apply(q, k, v, float(scale), bool(causal))
    return (o, lse) if return_lse else o


def check_device_status(stream=None):
    """Synchronise and raise if a kernel of the library hit a wait limit."""
    _check(load_library().fa_check_device_status(_stream_handle(stream)))


def schedule(B, H, Nq, Nk, d, causal, num_sms, num_splits=1):
    """The kernel's work list: int32 array [n_items, 8] of (cta, round,
    batch*head, first query row, first KV tile, end KV tile of query tile 0,
    of query tile 1 (-1 if absent), key slice)."""
    import numpy as np
    lib = load_library()
    n = ctypes.c_int64(0)
    args = (B, H, Nq, Nk, d, int(bool(causal)), num_sms, num_splits)
    _check(lib.fa_schedule(*args, None, 0, ctypes.byref(n)))
    out = np.zeros((n.value, 8), dtype=np.int32)
    _check(lib.fa_schedule(*args, out.ctypes.data, n.value, ctypes.byref(n)))
    return out


def splitkv_workspace(B, H, Nq, Nk, d, causal=False, num_splits=0):
    """(num_splits, workspace bytes) for fa_fwd_splitkv; num_splits=0 lets the library choose."""
    ns = ctypes.c_int(num_splits)
    nb = ctypes.c_size_t(0)
    _check(load_library().fa_splitkv_workspace(B, H, Nq, Nk, d, int(bool(causal)), ctypes.byref(ns), ctypes.byref(nb)))
    return ns.value, nb.value


def fa_fwd_splitkv(q, k, v, o=None, lse=None, scale=None, causal=False, num_splits=0, workspace=None,
                   stream=None):
    """Split-key attention forward; `workspace` is a CUDA uint8 tensor (allocated here if None)."""
    B, H, Nq, Nk, d = _shape(q, k)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    num_splits, nbytes = splitkv_workspace(B, H, Nq, Nk, d, causal, num_splits)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _check(load_library().fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                         B, H, Nq, Nk, d, scale, int(bool(causal)), num_splits,
                                         workspace.data_ptr(), workspace.numel(), _stream_handle(stream)))
    return o, lse


def fa_fwd_splitkv_noalloc(q, k, v, o, lse, scale=None, causal=False, num_splits=0, stream=None):
    """Split-key forward whose partials live in the library's fixed scratch area
    (no allocation anywhere on this call; o and lse are caller-provided:
    o bf16 like q, lse fp32 [B, H, Nq], both contiguous on q's device)."""
    for t in (q, k, v):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
            raise TypeError("q, k, v must be contiguous bf16 CUDA tensors")
    B, H, Nq, Nk, d = _shape(q, k)
    if k.shape != (B, H, Nk, d) or v.shape != (B, H, Nk, d):
        raise ValueError(f"shape mismatch: q {tuple(q.shape)} k {tuple(k.shape)} v {tuple(v.shape)}")
    if not (isinstance(o, torch.Tensor) and o.dtype == torch.bfloat16 and o.shape == q.shape
            and o.is_contiguous() and o.device == q.device):
        raise TypeError("o must be a contiguous bf16 tensor shaped like q on q's device")
    if not (isinstance(lse, torch.Tensor) and lse.dtype == torch.float32 and lse.shape == (B, H, Nq)
            and lse.is_contiguous() and lse.device == q.device):
        raise TypeError("lse must be a contiguous fp32 tensor [B, H, Nq] on q's device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(load_library().fa_fwd_splitkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                                 lse.data_ptr(), B, H, Nq, Nk, d, scale, int(bool(causal)),
                                                 num_splits, _stream_handle(stream)))
    return o, lse


def raw_fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Nq, Nk, d, scale, causal, stream_handle=0) -> int:
    """The C call with raw integers; returns the status code (argument tests)."""
    return load_library().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Nq, Nk, d, scale,
                                 int(causal), stream_handle)
