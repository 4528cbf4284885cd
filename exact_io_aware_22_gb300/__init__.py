"""Exact IO-aware attention (FlashAttention-2 forward and backward) for GB300.

Thin ctypes binding over the C ABI in ``include/fa.h`` (``libfa_gb300.so``,
built for sm_103a by ``exact_io_aware_22_gb300.build``).  This module only
marshals arguments: it checks tensor devices, dtypes, shapes and contiguity,
then passes raw device pointers and torch's current CUDA stream to the
library.  Every step of the computation runs in the library's CUDA kernels.
There is no fallback: if the library is missing or cannot be loaded, every
call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

__all__ = ["fwd", "bwd", "bwd_workspace_size", "device_status", "set_wait_limit_ns",
           "selftest_timeout", "trace_enable", "trace_read", "FAError", "library_path", "load_library", "STATUS"]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libfa_gb300.so")

STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_VALUE", 2: "FA_ERR_UNSUPPORTED",
          3: "FA_ERR_MISALIGNED", 4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT"}
FA_FP16, FA_BF16 = 0, 1

_lib = None


class FAError(RuntimeError):
    """A non-FA_OK status from the library."""

    def __init__(self, code: int, what: str):
        self.code = code
        self.name = STATUS.get(code, str(code))
        msg = f"{what}: {self.name}"
        if code == 4 and _lib is not None:
            msg += f" (cudaError {_lib.fa_last_cuda_error()})"
        super().__init__(msg)


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None):
    """Load (once) and return the ctypes handle of the CUDA library."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"CUDA library not built: {p} is missing "
                           "(run exact_io_aware_22_gb300.build.build())")
    lib = ctypes.CDLL(p)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_bwd_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_bwd_workspace_size.restype = sz
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, vp]
    lib.fa_bwd.restype = i
    lib.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_gqa.restype = i
    lib.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, i,
                               vp]
    lib.fa_bwd_gqa.restype = i
    lib.fa_fwd_swa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_swa.restype = i
    lib.fa_bwd_swa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, i,
                               vp]
    lib.fa_bwd_swa.restype = i
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_varlen.restype = i
    lib.fa_bwd_varlen_workspace_size.argtypes = [i, i, i, i]
    lib.fa_bwd_varlen_workspace_size.restype = sz
    lib.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, i, i, i, i, i, i,
                                  i, i, f, i, vp]
    lib.fa_bwd_varlen.restype = i
    lib.fa_decode_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_decode_workspace_size.restype = sz
    lib.fa_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, i, vp]
    lib.fa_decode.restype = i
    lib.fa_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, f, f, f, i, vp]
    lib.fa_decode_fp8.restype = i
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, f, f, f, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_quantize_fp8.argtypes = [vp, vp, ctypes.c_longlong, i, i, f, i, i, vp]
    lib.fa_quantize_fp8.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_last_cuda_error.restype = i
    lib.fa_device_status.argtypes = [vp]
    lib.fa_device_status.restype = i
    lib.fa_set_wait_limit_ns.argtypes = [ctypes.c_ulonglong]
    lib.fa_set_wait_limit_ns.restype = i
    lib.fa_selftest_timeout.argtypes = [ctypes.c_ulonglong, vp]
    lib.fa_selftest_timeout.restype = i
    lib.fa_trace_enable.argtypes = [i]
    lib.fa_trace_enable.restype = i
    lib.fa_trace_kind_name.argtypes = [i]
    lib.fa_trace_kind_name.restype = ctypes.c_char_p
    lib.fa_trace_read.argtypes = [i, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_longlong)]
    lib.fa_trace_read.restype = i
    if path is None:
        _lib = lib
    return lib


def _check(code: int, what: str):
    if code != 0:
        raise FAError(code, what)


def _stream():
    import torch
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return FA_FP16
    if t.dtype == torch.bfloat16:
        return FA_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: fp16 or bf16 expected")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _need_cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous (B, H, N, d)")


def _kv_heads(q, k, v) -> int:
    """Hkv of K and V shaped (B, Hkv, N, d) beside q (B, H, N, d), H a multiple of Hkv."""
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be (B, H, N, d) and k, v one (B, Hkv, N, d) shape")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if (k.shape[0], k.shape[2], k.shape[3]) != (B, N, d) or Hkv < 1 or H % Hkv:
        raise ValueError("k, v must be (B, Hkv, N, d) with H a multiple of Hkv")
    return Hkv


def _window(causal: bool, window: int) -> int:
    if window < 0 or (window > 0 and not causal):
        raise ValueError("window > 0 is a causal sliding window (causal=True)")
    return int(window)


def fwd(q, k, v, causal: bool = True, scale: float | None = None, out=None, lse=None,
        window: int = 0):
    """O, L = attention(q, k, v) for (B, H, N, d) fp16/bf16 CUDA tensors.

    L is (B, H, N) fp32, the natural-log logsumexp of each row's scaled scores.
    k and v may have fewer heads, (B, Hkv, N, d) with H a multiple of Hkv: each
    group of H/Hkv consecutive query heads shares one K/V head (GQA; Hkv = 1 is MQA).
    ``window`` > 0 (causal only) limits each query to the ``window`` most recent keys,
    itself included (sliding-window attention).
    ``scale`` defaults to 1/sqrt(d).  Runs asynchronously on torch's current stream.
    """
    import torch
    _need_cuda(q, k, v)
    Hkv = _kv_heads(q, k, v)
    window = _window(causal, window)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _need_cuda(out, lse)
    if out.shape != q.shape or out.dtype != q.dtype or lse.shape != (B, H, N) \
            or lse.dtype != torch.float32:
        raise ValueError("out must match q; lse must be (B, H, N) fp32")
    lib = load_library()
    if window > 0:
        _check(lib.fa_fwd_swa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, N, d,
                              window, float(scale), _dtype_code(q), _stream()), "fa_fwd_swa")
    elif Hkv == H:
        _check(lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, int(causal),
                          float(scale), _dtype_code(q), _stream()), "fa_fwd")
    else:
        _check(lib.fa_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Hkv, N, d,
                              int(causal), float(scale), _dtype_code(q), _stream()), "fa_fwd_gqa")
    return out, lse


def bwd_workspace_size(B: int, H: int, N: int, d: int, causal: bool = True) -> int:
    return int(load_library().fa_bwd_workspace_size(B, H, N, d, int(causal)))


def bwd(q, k, v, o, lse, do, causal: bool = True, scale: float | None = None,
        dq=None, dk=None, dv=None, workspace=None, window: int = 0):
    """dQ, dK, dV of attention for upstream gradient ``do``.

    q, o, do, dq are (B, H, N, d); k, v, dk, dv are (B, Hkv, N, d) (Hkv = H unless
    K/V heads are shared, as in ``fwd``; a shared head's dK and dV sum over its
    query heads; ``window`` as in ``fwd``).  ``o`` and ``lse`` are the forward's
    outputs.  ``workspace`` (optional) is a CUDA uint8 tensor of at least
    ``bwd_workspace_size`` bytes; without it the library takes scratch from the
    stream-ordered allocator.
    """
    import torch
    _need_cuda(q, k, v, o, lse, do)
    Hkv = _kv_heads(q, k, v)
    window = _window(causal, window)
    B, H, N, d = q.shape
    for t in (k, v, o, do):
        if t.dtype != q.dtype:
            raise ValueError("q, k, v, o, do must share one dtype")
    if o.shape != q.shape or do.shape != q.shape:
        raise ValueError("o and do must match q")
    if lse.shape != (B, H, N) or lse.dtype != torch.float32:
        raise ValueError("lse must be (B, H, N) fp32")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need_cuda(dq, dk, dv)
    if dq.shape != q.shape or dk.shape != k.shape or dv.shape != v.shape:
        raise ValueError("dq must match q, dk and dv must match k and v")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        _need_cuda(workspace)
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    lib = load_library()
    if window > 0:
        _check(lib.fa_bwd_swa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                              _ptr(dk), _ptr(dv), ws_ptr, ws_bytes, B, H, Hkv, N, d, window,
                              float(scale), _dtype_code(q), _stream()), "fa_bwd_swa")
    elif Hkv == H:
        _check(lib.fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                          _ptr(dk), _ptr(dv), ws_ptr, ws_bytes, B, H, N, d, int(causal),
                          float(scale), _dtype_code(q), _stream()), "fa_bwd")
    else:
        _check(lib.fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                              _ptr(dk), _ptr(dv), ws_ptr, ws_bytes, B, H, Hkv, N, d, int(causal),
                              float(scale), _dtype_code(q), _stream()), "fa_bwd_gqa")
    return dq, dk, dv


def _packed(q, k, v, cu_seqlens):
    """(B, total, H, Hkv, d) of packed sequences q (total, H, d), k, v (total, Hkv, d)."""
    import torch
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape:
        raise ValueError("packed q must be (total, H, d) and k, v one (total, Hkv, d) shape")
    total, H, d = q.shape
    Hkv = k.shape[1]
    if k.shape[0] != total or k.shape[2] != d or Hkv < 1 or H % Hkv:
        raise ValueError("k, v must be (total, Hkv, d) with H a multiple of Hkv")
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor of B+1 offsets")
    return cu_seqlens.numel() - 1, total, H, Hkv, d


def fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = True,
               scale: float | None = None, window: int = 0, out=None, lse=None):
    """O, L of packed variable-length sequences: q (total, H, d), k and v (total, Hkv, d),
    sequence b at rows cu_seqlens[b] .. cu_seqlens[b+1]-1 (int32 CUDA tensor, B+1
    entries), each attending only to its own keys; max_seqlen bounds every length.
    L is (H, total) fp32.  ``window`` and shared K/V heads as in ``fwd``."""
    import torch
    _need_cuda(q, k, v, cu_seqlens)
    B, total, H, Hkv, d = _packed(q, k, v, cu_seqlens)
    window = _window(causal, window)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, total), dtype=torch.float32, device=q.device) if lse is None else lse
    _need_cuda(out, lse)
    if out.shape != q.shape or out.dtype != q.dtype or lse.shape != (H, total) \
            or lse.dtype != torch.float32:
        raise ValueError("out must match q; lse must be (H, total) fp32")
    _check(load_library().fa_fwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens), B, total,
        int(max_seqlen), H, Hkv, d, int(causal), window, float(scale), _dtype_code(q), _stream()),
        "fa_fwd_varlen")
    return out, lse


def bwd_varlen(q, k, v, o, lse, do, cu_seqlens, max_seqlen: int, causal: bool = True,
               scale: float | None = None, window: int = 0, dq=None, dk=None, dv=None,
               workspace=None):
    """dQ (total, H, d), dK, dV (total, Hkv, d) of packed variable-length sequences (see
    ``fwd_varlen``); ``o`` and ``lse`` are its outputs.  ``workspace``: optional CUDA
    uint8 tensor of fa_bwd_varlen_workspace_size bytes."""
    import torch
    _need_cuda(q, k, v, o, lse, do, cu_seqlens)
    B, total, H, Hkv, d = _packed(q, k, v, cu_seqlens)
    window = _window(causal, window)
    if o.shape != q.shape or do.shape != q.shape or lse.shape != (H, total):
        raise ValueError("o and do must match q; lse must be (H, total)")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _need_cuda(dq, dk, dv)
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        _need_cuda(workspace)
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check(load_library().fa_bwd_varlen(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
        ws_ptr, ws_bytes, _ptr(cu_seqlens), B, total, int(max_seqlen), H, Hkv, d, int(causal),
        window, float(scale), _dtype_code(q), _stream()), "fa_bwd_varlen")
    return dq, dk, dv


def fwd_fp8(q8, k8, vt8, q_scale: float, k_scale: float, v_scale: float, causal: bool = True,
            scale: float | None = None, out=None, lse=None):
    """O (bf16, B x H x N x 128) and L (fp32, B x H x N) of attention on 8-bit E4M3 codes:
    q8 (B, H, N, 128), k8 (B, Hkv, N, 128) and vt8 (B, Hkv, 128, N) -- V with its last two
    axes swapped -- as uint8 (or float8_e4m3fn) CUDA tensors standing for q_scale * Q,
    k_scale * K and v_scale * V.  N must be a multiple of 16."""
    import torch
    _need_cuda(q8, k8, vt8)
    if q8.dim() != 4 or k8.dim() != 4 or vt8.dim() != 4:
        raise ValueError("q8, k8 must be (B, H|Hkv, N, 128) and vt8 (B, Hkv, 128, N)")
    for t in (q8, k8, vt8):
        if t.element_size() != 1:
            raise ValueError("FP8 inputs must be 1-byte tensors (uint8 or float8_e4m3fn)")
    B, H, N, d = q8.shape
    Hkv = k8.shape[1]
    if k8.shape != (B, Hkv, N, d) or vt8.shape != (B, Hkv, d, N) or Hkv < 1 or H % Hkv:
        raise ValueError("k8 must be (B, Hkv, N, d) and vt8 (B, Hkv, d, N), H a multiple of Hkv")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device) if lse is None else lse
    _need_cuda(out, lse)
    if out.shape != (B, H, N, d) or out.dtype != torch.bfloat16 or lse.shape != (B, H, N) \
            or lse.dtype != torch.float32:
        raise ValueError("out must be (B, H, N, d) bf16 and lse (B, H, N) fp32")
    _check(load_library().fa_fwd_fp8(
        _ptr(q8), _ptr(k8), _ptr(vt8), _ptr(out), _ptr(lse), B, H, Hkv, N, d, int(causal),
        float(scale), float(q_scale), float(k_scale), float(v_scale), _stream()), "fa_fwd_fp8")
    return out, lse


def quantize_fp8(x, inv_scale: float, transpose: bool = False, out=None):
    """E4M3 codes (uint8) of x * inv_scale, rounded to nearest even and saturated at
    +-448, for a 16-bit CUDA tensor x of shape (..., rows, cols); with ``transpose``
    the result is (..., cols, rows)."""
    import torch
    _need_cuda(x)
    if x.dim() < 2:
        raise ValueError("x must have at least two dimensions")
    rows, cols = x.shape[-2], x.shape[-1]
    mats = x.numel() // max(rows * cols, 1)
    shape = tuple(x.shape[:-2]) + ((cols, rows) if transpose else (rows, cols))
    out = torch.empty(shape, dtype=torch.uint8, device=x.device) if out is None else out
    _need_cuda(out)
    if tuple(out.shape) != shape or out.element_size() != 1:
        raise ValueError("out must be a 1-byte tensor of the result's shape")
    _check(load_library().fa_quantize_fp8(
        _ptr(x), _ptr(out), mats, rows, cols, float(inv_scale), int(transpose), _dtype_code(x),
        _stream()), "fa_quantize_fp8")
    return out


def decode_workspace_size(B: int, H: int, Hkv: int, Nmax: int, d: int) -> int:
    return int(load_library().fa_decode_workspace_size(B, H, Hkv, Nmax, d))


def decode(q, k_cache, v_cache, cache_seqlens, scale: float | None = None, out=None, lse=None,
           workspace=None):
    """O (B, H, d), L (B, H) fp32 of one query row per (batch, head) against the first
    cache_seqlens[b] rows of k_cache, v_cache (B, Hkv, Nmax, d); cache_seqlens is an
    int32 CUDA tensor of B lengths.  Query head h uses K/V head h // (H // Hkv).  A
    sequence with no cached key gets O = 0, L = -inf.  ``workspace``: an optional uint8
    CUDA tensor of at least decode_workspace_size(...) bytes (else one is allocated
    per call on the current stream)."""
    import torch
    _need_cuda(q, k_cache, v_cache, cache_seqlens)
    if q.dim() != 3 or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("q must be (B, H, d) and the caches one (B, Hkv, Nmax, d) shape")
    B, H, d = q.shape
    Bk, Hkv, Nmax, dk = k_cache.shape
    if Bk != B or dk != d or Hkv < 1 or H % Hkv:
        raise ValueError("caches must be (B, Hkv, Nmax, d) with H a multiple of Hkv")
    if cache_seqlens.dtype != torch.int32 or cache_seqlens.shape != (B,):
        raise ValueError("cache_seqlens must be an int32 tensor of B lengths")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    _need_cuda(out, lse)
    if out.shape != q.shape or out.dtype != q.dtype or lse.shape != (B, H) \
            or lse.dtype != torch.float32:
        raise ValueError("out must match q; lse must be (B, H) fp32")
    ws, ws_bytes = None, 0
    if workspace is not None:
        _need_cuda(workspace)
        ws, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check(load_library().fa_decode(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_seqlens), _ptr(out), _ptr(lse), ws,
        ws_bytes, B, H, Hkv, Nmax, d, float(scale), _dtype_code(q), _stream()), "fa_decode")
    return out, lse


def decode_fp8(q, k_cache8, v_cache8, cache_seqlens, k_scale: float, v_scale: float,
               scale: float | None = None, out=None, lse=None, workspace=None):
    """As ``decode``, with caches of 8-bit E4M3 codes (uint8 or float8_e4m3fn CUDA tensors,
    (B, Hkv, Nmax, 128)) standing for k_scale * K and v_scale * V."""
    import torch
    _need_cuda(q, k_cache8, v_cache8, cache_seqlens)
    if q.dim() != 3 or k_cache8.dim() != 4 or v_cache8.shape != k_cache8.shape:
        raise ValueError("q must be (B, H, d) and the caches one (B, Hkv, Nmax, d) shape")
    if k_cache8.element_size() != 1 or v_cache8.element_size() != 1:
        raise ValueError("E4M3 caches must be 1-byte tensors")
    B, H, d = q.shape
    Bk, Hkv, Nmax, dk = k_cache8.shape
    if Bk != B or dk != d or Hkv < 1 or H % Hkv:
        raise ValueError("caches must be (B, Hkv, Nmax, d) with H a multiple of Hkv")
    if cache_seqlens.dtype != torch.int32 or cache_seqlens.shape != (B,):
        raise ValueError("cache_seqlens must be an int32 tensor of B lengths")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H), dtype=torch.float32, device=q.device) if lse is None else lse
    _need_cuda(out, lse)
    if out.shape != q.shape or out.dtype != q.dtype or lse.shape != (B, H) \
            or lse.dtype != torch.float32:
        raise ValueError("out must match q; lse must be (B, H) fp32")
    ws, ws_bytes = None, 0
    if workspace is not None:
        _need_cuda(workspace)
        ws, ws_bytes = _ptr(workspace), workspace.numel() * workspace.element_size()
    _check(load_library().fa_decode_fp8(
        _ptr(q), _ptr(k_cache8), _ptr(v_cache8), _ptr(cache_seqlens), _ptr(out), _ptr(lse), ws,
        ws_bytes, B, H, Hkv, Nmax, d, float(scale), float(k_scale), float(v_scale),
        _dtype_code(q), _stream()), "fa_decode_fp8")
    return out, lse


def device_status() -> int:
    """Synchronise the current stream; return (and clear) the device status code."""
    return int(load_library().fa_device_status(_stream()))


def set_wait_limit_ns(ns: int) -> None:
    _check(load_library().fa_set_wait_limit_ns(int(ns)), "fa_set_wait_limit_ns")


def trace_enable(on: bool = True) -> None:
    """Start (clearing earlier records) or stop the per-kernel CUDA-event trace."""
    _check(load_library().fa_trace_enable(int(on)), "fa_trace_enable")


def trace_read() -> dict:
    """{kernel name: (total GPU ms, launches)} of the traced launches."""
    lib = load_library()
    out = {}
    k = 0
    while True:
        name = lib.fa_trace_kind_name(k)
        if name is None:
            break
        ms, n = ctypes.c_double(), ctypes.c_longlong()
        _check(lib.fa_trace_read(k, ctypes.byref(ms), ctypes.byref(n)), "fa_trace_read")
        out[name.decode()] = (ms.value, n.value)
        k += 1
    return out


def selftest_timeout(limit_ns: int = 1_000_000) -> int:
    """Run the bounded-wait self test; returns the status code (5 = timeout seen)."""
    return int(load_library().fa_selftest_timeout(int(limit_ns), _stream()))
