"""Exact tiled attention forward (FlashAttention forward) for GB300 / sm_103a.

The compute path is the C-ABI library ``libfa`` (``include/fa.h``): hand-written
CUDA kernels built for sm_103a by ``build.py``. This module is a thin binding
with the same entry-point names; it only marshals arguments (device pointers,
sizes, the current CUDA stream). There is no fallback: if ``libfa.so`` is
missing or fails to load, every call raises.

    import exact_tiled_attention_forward_gb300 as fa
    o, lse = fa.fa_forward(q, k, v, causal=False)          # torch CUDA tensors

Tensors: q ``[B, H_q, N_q, d]``, k/v ``[B, H_kv, N_k, d]`` BF16 (or FP16, through
``fa_forward_fp16``) contiguous; returns o ``[B, H_q, N_q, d]`` of the same type
and lse ``[B, H_q, N_q]`` FP32.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libfa.so")
LIB_SINGLE_GPU_PATH = os.path.join(_PKG, "_build", "libfa_single_gpu.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "fa.h")
HEADER_SINGLE_GPU = os.path.join(os.path.dirname(_PKG), "include", "fa_single_gpu.h")

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_CUDA = -3
FA_ERR_NO_MEMORY = -4
FA_ERR_TIMEOUT = -5
FA_ERR_TOO_LARGE = -6
FA_ERR_BOUNDS = -7

FA_DTYPE_BF16 = 0
FA_DTYPE_FP16 = 1

_lib = None
_lib_single = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = lib().fa_status_string(status).decode()
        if status == FA_ERR_CUDA:
            msg += f" (cudaError {lib().fa_get_last_cuda_error()})"
        super().__init__(f"{what}: {msg}" if what else msg)


_c_int, _c_float, _c_size, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

_SIGNATURES = {
    "fa_forward": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 7 + [_c_float, _vp]),
    "fa_forward_fp16": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 7 + [_c_float, _vp]),
    "fa_forward_fp8": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 7 + [_c_float] * 4 + [_vp]),
    "fa_forward_host": (_c_int, [_c_int] + [ctypes.POINTER(_vp)] * 5 + [_c_int] * 7 +
                        [_c_float, _c_int, _vp]),
    "fa_forward_host_packed": (_c_int, [_c_int] + [ctypes.POINTER(_vp)] * 2 + [_c_int] * 7 +
                               [_c_float, _c_int, _vp]),
    "fa_forward_noalloc": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 7 + [_c_float, _vp]),
    "fa_backward": (_c_int, [_vp] * 9 + [_c_int] * 7 + [_c_float, _c_int, _vp]),
    "fa_decode_paged": (_c_int, [_vp] * 7 + [_c_int] * 8 + [_c_float, _c_int, _vp]),
    "fa_naive_forward": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 7 +
                         [_c_float, _vp, _c_size, _vp]),
    "fa_naive_workspace_bytes": (_c_size, [_c_int] * 4),
    "fa_forward_plan": (_c_int, [_c_int] * 7 + [ctypes.POINTER(ctypes.c_longlong),
                                                ctypes.POINTER(_c_int), ctypes.POINTER(_c_size)]),
    "fa_selftest_wait_timeout": (_c_int, [ctypes.c_ulonglong, _vp]),
    "fa_selftest_bounds": (_c_int, [_vp]),
    "fa_debug_build": (_c_int, []),
    "fa_status_string": (ctypes.c_char_p, [_c_int]),
    "fa_get_last_cuda_error": (_c_int, []),
    "fa_device_status": (_c_int, [_c_int]),
    "fa_version": (_c_int, []),
}


def lib() -> ctypes.CDLL:
    """Load libfa.so (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libfa.so not found at {LIB_PATH}: build it first "
                              "(python -m exact_tiled_attention_forward_gb300.build)")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def lib_single_gpu() -> ctypes.CDLL:
    """Load libfa_single_gpu.so (once): libfa plus the cluster-multicast forward
    of ``include/fa_single_gpu.h``. Only for a process that uses one GPU."""
    global _lib_single
    if _lib_single is None:
        if not os.path.exists(LIB_SINGLE_GPU_PATH):
            raise ImportError(f"libfa_single_gpu.so not found at {LIB_SINGLE_GPU_PATH}: build it first "
                              "(python -m exact_tiled_attention_forward_gb300.build)")
        l = ctypes.CDLL(LIB_SINGLE_GPU_PATH)
        sigs = dict(_SIGNATURES)
        sigs["fa_forward_cluster_multicast"] = _SIGNATURES["fa_forward"]
        for name, (res, args) in sigs.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib_single = l
    return _lib_single


def header_functions(header: str = HEADER) -> list[str]:
    """Names of the functions a header (default ``include/fa.h``) declares."""
    text = open(header).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(fa_\w+)\s*\(", text, re.M)))


def _check(status: int, what: str):
    if status != FA_OK:
        raise FaError(status, what)


def _stream_ptr(stream):
    """Raw handle of `stream` (a torch stream or an int), or of the current
    stream of the current device when None."""
    if stream is None:
        import torch
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)   # ~10x cheaper than current_stream()
        if raw is not None:
            return raw(torch.cuda.current_device())
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _dims(q, k):
    B, H_q, N_q, d = q.shape
    Bk, H_kv, N_k, dk = k.shape
    if Bk != B or dk != d:
        raise ValueError("q and k/v disagree on batch or head dim")
    return B, H_q, H_kv, N_q, N_k, d


def _ptr(t):
    """Device address of a tensor as an int (0 for None or an empty tensor); the
    c_void_p argtypes take ints directly."""
    return t.data_ptr() if t is not None and t.numel() > 0 else 0


def _check_dtypes(dtype, q, k, v, out, lse):
    """All of q, k, v, out in `dtype`, lse FP32 (or None): libfa reads raw memory."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if t is not None and t.dtype != dtype:
            raise TypeError(f"{name} is {t.dtype}, expected {dtype}")
    if lse is not None and lse.dtype != torch.float32:
        raise TypeError(f"lse is {lse.dtype}, expected torch.float32")


def fa_forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
               return_lse: bool = True, stream=None):
    """Fused forward on the current CUDA stream. Returns ``(o, lse)``.
    BF16 tensors; FP16 tensors are passed on to ``fa_forward_fp16``."""
    import torch
    if q.dtype == torch.float16:
        return fa_forward_fp16(q, k, v, causal=causal, scale=scale, out=out, lse=lse,
                               return_lse=return_lse, stream=stream)
    _check_dtypes(torch.bfloat16, q, k, v, out, lse)
    B, H_q, H_kv, N_q, N_k, d = _dims(q, k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H_q, N_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H_q, N_q), dtype=torch.float32, device=q.device)
    st = lib().fa_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H_q, H_kv, N_q, N_k,
                          d, int(bool(causal)), float(scale), _stream_ptr(stream))
    _check(st, "fa_forward")
    return out, lse


def fa_forward_fp16(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                    return_lse: bool = True, stream=None):
    """Fused forward on FP16 q, k, v (FP16 o, FP32 lse). Returns ``(o, lse)``."""
    import torch
    _check_dtypes(torch.float16, q, k, v, out, lse)
    B, H_q, H_kv, N_q, N_k, d = _dims(q, k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H_q, N_q, d), dtype=torch.float16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H_q, N_q), dtype=torch.float32, device=q.device)
    st = lib().fa_forward_fp16(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H_q, H_kv, N_q,
                               N_k, d, int(bool(causal)), float(scale), _stream_ptr(stream))
    _check(st, "fa_forward_fp16")
    return out, lse


def fa_forward_fp8(q, k, v, descale, causal: bool = False, scale: float | None = None, out=None, lse=None,
                   return_lse: bool = True, stream=None):
    """Fused forward on FP8 E4M3 inputs: q, k, v hold E4M3 codes (torch.uint8 or
    torch.float8_e4m3fn, one byte each) standing for code * factor, with
    ``descale = (factor_q, factor_k, factor_v)``. Returns ``(o, lse)``: o BF16,
    lse FP32. d must be 64 or 128."""
    import torch
    allowed = {torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)}
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype not in allowed:
            raise TypeError(f"{name} is {t.dtype}, expected E4M3 codes (torch.uint8 or torch.float8_e4m3fn)")
    if out is not None and out.dtype != torch.bfloat16:
        raise TypeError(f"out is {out.dtype}, expected torch.bfloat16")
    if lse is not None and lse.dtype != torch.float32:
        raise TypeError(f"lse is {lse.dtype}, expected torch.float32")
    B, H_q, H_kv, N_q, N_k, d = _dims(q, k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H_q, N_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H_q, N_q), dtype=torch.float32, device=q.device)
    dq, dk, dv = (float(x) for x in descale)
    st = lib().fa_forward_fp8(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H_q, H_kv, N_q, N_k,
                              d, int(bool(causal)), float(scale), dq, dk, dv, _stream_ptr(stream))
    _check(st, "fa_forward_fp8")
    return out, lse


def fa_forward_host(qs, ks, vs, outs, lses=None, causal: bool = False, scale: float | None = None,
                    stream=None) -> None:
    """n requests whose tensors are in host memory (lists of CPU tensors of one
    shape and type, BF16 or FP16; page-locked memory lets the copies overlap the
    kernels). Results land in ``outs`` (and ``lses`` when given) once ``stream``
    has been synchronised; see ``include/fa.h``."""
    import torch
    n = len(qs)
    if not (len(ks) == len(vs) == len(outs) == n) or (lses is not None and len(lses) != n):
        raise ValueError("qs, ks, vs, outs (and lses) must have one entry per request")
    if n == 0:
        return
    dtype = qs[0].dtype
    if dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"q is {dtype}, expected torch.bfloat16 or torch.float16")
    B, H_q, H_kv, N_q, N_k, d = _dims(qs[0], ks[0])
    for i in range(n):
        _check_dtypes(dtype, qs[i], ks[i], vs[i], outs[i], None if lses is None else lses[i])
        group = [qs[i], ks[i], vs[i], outs[i]] + ([] if lses is None or lses[i] is None else [lses[i]])
        for t in group:
            if t.device.type != "cpu" or not t.is_contiguous():
                raise ValueError("fa_forward_host takes contiguous CPU tensors")
        if (qs[i].shape != qs[0].shape or ks[i].shape != ks[0].shape or vs[i].shape != ks[0].shape
                or tuple(outs[i].shape) != (B, H_q, N_q, d)
                or (lses is not None and lses[i] is not None and tuple(lses[i].shape) != (B, H_q, N_q))):
            raise ValueError(f"request {i} does not have the shape of request 0")
    if scale is None:
        scale = 1.0 / math.sqrt(d)

    def arr(ts):
        return (_vp * n)(*[t.data_ptr() if t is not None else 0 for t in ts])

    st = lib().fa_forward_host(n, arr(qs), arr(ks), arr(vs), arr(outs),
                               None if lses is None else arr(lses), B, H_q, H_kv, N_q, N_k, d,
                               int(bool(causal)), float(scale),
                               FA_DTYPE_FP16 if dtype == torch.float16 else FA_DTYPE_BF16,
                               _stream_ptr(stream))
    _check(st, "fa_forward_host")


def fa_forward_host_packed(qkvs, outs, shape, causal: bool = False, scale: float | None = None,
                           dtype=None, stream=None) -> None:
    """``fa_forward_host`` with each request packed in two contiguous CPU
    buffers: ``qkvs[i]`` holds Q, K, V back to back and ``outs[i]`` receives O
    then LSE (FP32). ``shape`` = (B, H_q, H_kv, N_q, N_k, d); ``dtype``
    torch.bfloat16 (default) or torch.float16 names the element type."""
    import torch
    dtype = torch.bfloat16 if dtype is None else dtype
    if dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"dtype is {dtype}, expected torch.bfloat16 or torch.float16")
    B, H_q, H_kv, N_q, N_k, d = (int(x) for x in shape)
    n = len(qkvs)
    if len(outs) != n:
        raise ValueError("qkvs and outs must have one entry per request")
    if n == 0:
        return
    in_bytes = (B * H_q * N_q + 2 * B * H_kv * N_k) * d * 2
    out_bytes = B * H_q * N_q * (d * 2 + 4)
    for t, need in [(t, in_bytes) for t in qkvs] + [(t, out_bytes) for t in outs]:
        if t.device.type != "cpu" or not t.is_contiguous():
            raise ValueError("fa_forward_host_packed takes contiguous CPU buffers")
        if t.numel() * t.element_size() < need:
            raise ValueError(f"a buffer holds {t.numel() * t.element_size()} bytes, needs {need}")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    ptrs = lambda ts: (_vp * n)(*[t.data_ptr() for t in ts])
    st = lib().fa_forward_host_packed(n, ptrs(qkvs), ptrs(outs), B, H_q, H_kv, N_q, N_k, d,
                                      int(bool(causal)), float(scale),
                                      FA_DTYPE_FP16 if dtype == torch.float16 else FA_DTYPE_BF16,
                                      _stream_ptr(stream))
    _check(st, "fa_forward_host_packed")


def _check_layout(what, **tensors):
    """Each named tensor (name -> (tensor, expected shape)) is a contiguous CUDA
    tensor of that shape: libfa derives every size from the shapes of q and k."""
    given = [(name, t, shape) for name, (t, shape) in tensors.items() if t is not None]
    for name, t, shape in given:
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{what}: {name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    for name, t, _ in given:
        if not t.is_contiguous():
            raise ValueError(f"{what}: {name} must be contiguous")
    for name, t, _ in given:
        if t.numel() > 0 and t.device.type != "cuda":
            raise ValueError(f"{what}: {name} must be a CUDA tensor")


def fa_backward(q, k, v, o, lse, do, causal: bool = False, scale: float | None = None, dq=None,
                dk=None, dv=None, stream=None):
    """Gradients (dq, dk, dv) of the forward given its o and lse and the upstream
    gradient do; BF16 or FP16 tensors (all one type), FP32 lse. Returns (dq, dk, dv)."""
    import torch
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"q is {dtype}, expected torch.bfloat16 or torch.float16")
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do), ("dq", dq), ("dk", dk), ("dv", dv)):
        if t is not None and t.dtype != dtype:
            raise TypeError(f"{name} is {t.dtype}, expected {dtype}")
    if lse is None or lse.dtype != torch.float32:
        raise TypeError("lse (FP32, from the forward) is required")
    B, H_q, H_kv, N_q, N_k, d = _dims(q, k)
    qs, ks = (B, H_q, N_q, d), (B, H_kv, N_k, d)
    _check_layout("fa_backward", q=(q, qs), k=(k, ks), v=(v, ks), o=(o, qs), lse=(lse, (B, H_q, N_q)),
                  do=(do, qs), dq=(dq, qs), dk=(dk, ks), dv=(dv, ks))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    st = lib().fa_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq), _ptr(dk),
                           _ptr(dv), B, H_q, H_kv, N_q, N_k, d, int(bool(causal)), float(scale),
                           FA_DTYPE_FP16 if dtype == torch.float16 else FA_DTYPE_BF16,
                           _stream_ptr(stream))
    _check(st, "fa_backward")
    return dq, dk, dv


def fa_decode_paged(q, k_cache, v_cache, block_table, seqlens_k, causal: bool = False,
                    scale: float | None = None, out=None, lse=None, return_lse: bool = True, stream=None):
    """Decode over a paged K/V cache. q ``[B, H_q, N_q, d]``; k_cache, v_cache
    ``[num_pages, H_kv, 128, d]`` (BF16 or FP16, q's type); block_table int32
    ``[B, max_pages]``; seqlens_k int32 ``[B]``; all on the device. Returns
    ``(o, lse)`` as ``fa_forward`` does."""
    import torch
    dtype = q.dtype
    if dtype not in (torch.bfloat16, torch.float16):
        raise TypeError(f"q is {dtype}, expected torch.bfloat16 or torch.float16")
    _check_dtypes(dtype, q, k_cache, v_cache, out, lse)
    for name, t in (("block_table", block_table), ("seqlens_k", seqlens_k)):
        if t.dtype != torch.int32:
            raise TypeError(f"{name} is {t.dtype}, expected torch.int32")
    B, H_q, N_q, d = q.shape
    num_pages, H_kv, page, dk = k_cache.shape
    if page != 128 or dk != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache / v_cache must be [num_pages, H_kv, 128, d] with q's d")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(seqlens_k.shape) != (B,):
        raise ValueError("block_table must be [B, max_pages] and seqlens_k [B]")
    _check_layout("fa_decode_paged", q=(q, q.shape), k_cache=(k_cache, k_cache.shape),
                  v_cache=(v_cache, k_cache.shape), block_table=(block_table, block_table.shape),
                  seqlens_k=(seqlens_k, (B,)), out=(out, q.shape), lse=(lse, (B, H_q, N_q)))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H_q, N_q), dtype=torch.float32, device=q.device)
    st = lib().fa_decode_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table), _ptr(seqlens_k),
                               _ptr(out), _ptr(lse), B, H_q, H_kv, N_q, num_pages, block_table.shape[1], d,
                               int(bool(causal)), float(scale),
                               FA_DTYPE_FP16 if dtype == torch.float16 else FA_DTYPE_BF16, _stream_ptr(stream))
    _check(st, "fa_decode_paged")
    return out, lse


def fa_forward_noalloc(q, k, v, causal: bool = False, scale: float | None = None, out=None,
                       lse=None, return_lse: bool = True, stream=None):
    """``fa_forward`` that allocates no device memory inside libfa: split
    partials use libfa's fixed 32 MiB device array (see ``include/fa.h``).
    Concurrent calls race on that array; keep them on one stream. Returns ``(o, lse)``."""
    import torch
    _check_dtypes(torch.bfloat16, q, k, v, out, lse)
    B, H_q, H_kv, N_q, N_k, d = _dims(q, k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H_q, N_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H_q, N_q), dtype=torch.float32, device=q.device)
    st = lib().fa_forward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H_q, H_kv,
                                  N_q, N_k, d, int(bool(causal)), float(scale), _stream_ptr(stream))
    _check(st, "fa_forward_noalloc")
    return out, lse


def fa_forward_cluster_multicast(q, k, v, causal: bool = False, scale: float | None = None, out=None,
                                 lse=None, return_lse: bool = True, stream=None):
    """``fa_forward`` (BF16) with CTA pairs sharing K/V tile loads by cluster
    multicast, from libfa_single_gpu.so (``include/fa_single_gpu.h``): for a
    process that uses one GPU only. Returns ``(o, lse)``."""
    import torch
    _check_dtypes(torch.bfloat16, q, k, v, out, lse)
    B, H_q, H_kv, N_q, N_k, d = _dims(q, k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H_q, N_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H_q, N_q), dtype=torch.float32, device=q.device)
    l = lib_single_gpu()
    st = l.fa_forward_cluster_multicast(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H_q, H_kv,
                                        N_q, N_k, d, int(bool(causal)), float(scale), _stream_ptr(stream))
    if st != FA_OK:
        raise FaError(st, "fa_forward_cluster_multicast")
    return out, lse


def fa_forward_plan(B: int, H_q: int, H_kv: int, N_q: int, N_k: int, d: int,
                    causal: bool = False) -> dict:
    """How fa_forward runs this request on the current device: CTAs of its main
    kernel, kernels it launches, workspace bytes it allocates (the scratch that
    fa_forward_noalloc needs)."""
    ctas, launches, ws = ctypes.c_longlong(0), _c_int(0), _c_size(0)
    st = lib().fa_forward_plan(B, H_q, H_kv, N_q, N_k, d, int(bool(causal)), ctypes.byref(ctas),
                               ctypes.byref(launches), ctypes.byref(ws))
    _check(st, "fa_forward_plan")
    return {"ctas": int(ctas.value), "launches": int(launches.value), "workspace_bytes": int(ws.value)}


def fa_naive_workspace_bytes(B: int, H_q: int, N_q: int, N_k: int) -> int:
    return int(lib().fa_naive_workspace_bytes(B, H_q, N_q, N_k))


def fa_naive_forward(q, k, v, causal: bool = False, scale: float | None = None, out=None,
                     lse=None, workspace=None, return_lse: bool = True, stream=None):
    """Unfused three-kernel baseline (BF16). Returns ``(o, lse)``."""
    import torch
    _check_dtypes(torch.bfloat16, q, k, v, out, lse)
    B, H_q, H_kv, N_q, N_k, d = _dims(q, k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H_q, N_q, d), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H_q, N_q), dtype=torch.float32, device=q.device)
    nbytes = fa_naive_workspace_bytes(B, H_q, N_q, N_k)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    st = lib().fa_naive_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H_q, H_kv, N_q,
                                N_k, d, int(bool(causal)), float(scale), _ptr(workspace),
                                workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    _check(st, "fa_naive_forward")
    return out, lse


def fa_device_status(reset: bool = True) -> int:
    """Synchronise and return the device status word (FA_OK or FA_ERR_TIMEOUT)."""
    return int(lib().fa_device_status(int(bool(reset))))


def fa_status_string(status: int) -> str:
    return lib().fa_status_string(status).decode()


def fa_version() -> tuple[int, int]:
    v = int(lib().fa_version())
    return v >> 16, v & 0xFFFF
