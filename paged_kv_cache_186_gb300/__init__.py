"""Python binding of the sm_103a paged-KV-cache attention library.

Thin ctypes marshalling over the C ABI declared in include/pa.h: tensors are
passed as device pointers, the stream is torch's current CUDA stream. Every
step of the computation runs in the library's CUDA kernels; this module never
computes attention itself and has no fallback. If libpa_gb300.so is missing,
every call raises (build it with ``python -m paged_kv_cache_186_gb300.build``).

Names follow the C ABI: store_kv, decode, decode_window, decode_append,
decode_workspace_size, prefill_varlen, decode_noalloc, get_device_error,
debug_inject_wait_timeout.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa_gb300.so")

PA_KV_BF16 = 0
PA_KV_FP8_E4M3 = 1
PA_KV_INT8 = 2

PA_DEVERR_SLOT_RANGE = 0x1
PA_DEVERR_WAIT_TIMEOUT = 0x2
PA_DEVERR_BLOCK_RANGE = 0x4

STATUS = {0: "PA_OK", 1: "PA_ERR_NULL", 2: "PA_ERR_SHAPE", 3: "PA_ERR_DTYPE",
          4: "PA_ERR_UNSUPPORTED", 5: "PA_ERR_CUDA", 6: "PA_ERR_WORKSPACE", 7: "PA_ERR_ALIGN",
          8: "PA_ERR_TOO_LARGE"}

# Size of the static scratch buffer pa_decode_noalloc uses (PA_DECODE_NOALLOC_SCRATCH_BYTES).
DECODE_NOALLOC_SCRATCH_BYTES = 32 << 20

# Every symbol include/pa.h declares.
EXPORTED = ("pa_abi_version", "pa_status_string", "pa_store_kv", "pa_decode_workspace_size",
            "pa_decode", "pa_decode_window", "pa_decode_append", "pa_decode_window_append",
            "pa_prefill_varlen",
            "pa_decode_noalloc", "pa_get_device_error", "pa_debug_inject_wait_timeout")


class PAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}")


class KVCache(ctypes.Structure):
    """Mirror of pa_kv_cache."""
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libpa_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m paged_kv_cache_186_gb300.build` (needs nvcc)")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.pa_abi_version.restype = i32
    L.pa_abi_version.argtypes = []
    L.pa_status_string.restype = ctypes.c_char_p
    L.pa_status_string.argtypes = [ctypes.c_int]
    L.pa_store_kv.restype = ctypes.c_int
    L.pa_store_kv.argtypes = [P, P, P, P, P, i32, ctypes.POINTER(KVCache), P]
    L.pa_decode_workspace_size.restype = ctypes.c_size_t
    L.pa_decode_workspace_size.argtypes = [ctypes.POINTER(KVCache), i32, i32, i32, i32]
    L.pa_decode.restype = ctypes.c_int
    L.pa_decode.argtypes = [P, ctypes.POINTER(KVCache), P, i32, P, i32, i32, i32, ctypes.c_float,
                            P, P, ctypes.c_size_t, P]
    L.pa_decode_window.restype = ctypes.c_int
    L.pa_decode_window.argtypes = [P, ctypes.POINTER(KVCache), P, i32, P, i32, i32, i32,
                                   ctypes.c_float, i32, i32, P, P, ctypes.c_size_t, P]
    L.pa_decode_append.restype = ctypes.c_int
    L.pa_decode_append.argtypes = [P, P, P, P, P, ctypes.POINTER(KVCache), P, i32, P, i32, i32,
                                   i32, ctypes.c_float, P, P, ctypes.c_size_t, P]
    L.pa_decode_window_append.restype = ctypes.c_int
    L.pa_decode_window_append.argtypes = [P, P, P, P, P, ctypes.POINTER(KVCache), P, i32, P, i32,
                                          i32, i32, ctypes.c_float, i32, i32, P, P,
                                          ctypes.c_size_t, P]
    L.pa_prefill_varlen.restype = ctypes.c_int
    L.pa_prefill_varlen.argtypes = [P, ctypes.POINTER(KVCache), P, i32, P, P, i32, i32, i32, i32,
                                    ctypes.c_float, P, P]
    L.pa_decode_noalloc.restype = ctypes.c_int
    L.pa_decode_noalloc.argtypes = [P, ctypes.POINTER(KVCache), P, i32, P, i32, i32, i32,
                                    ctypes.c_float, P, P]
    L.pa_get_device_error.restype = ctypes.c_int
    L.pa_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    L.pa_debug_inject_wait_timeout.restype = ctypes.c_int
    L.pa_debug_inject_wait_timeout.argtypes = [i32, ctypes.c_uint64]
    del i64
    _lib = L
    return L


def _ptr(t: torch.Tensor | None):
    # a plain int: the prototypes declare c_void_p, which ctypes fills from it
    return None if t is None else t.data_ptr()


# The raw handle of the current stream, without building a torch.cuda.Stream
# object per call (a tenth of the cost; the public call is the fallback).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream():
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _check(code: int, what: str):
    if code != 0:
        raise PAError(code, what)


def make_cache(k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: torch.Tensor | None = None,
               v_scale: torch.Tensor | None = None) -> KVCache:
    """Describe caches of shape (num_blocks, block_size, num_kv_heads, head_dim):
    bf16, or uint8 E4M3 / int8 codes with fp32 scales (num_blocks, num_kv_heads,
    block_size)."""
    if k_cache.dtype == torch.bfloat16:
        dt = PA_KV_BF16
    elif k_cache.dtype in (torch.uint8, torch.float8_e4m3fn):
        dt = PA_KV_FP8_E4M3
    elif k_cache.dtype == torch.int8:
        dt = PA_KV_INT8
    else:
        raise TypeError(f"unsupported cache dtype {k_cache.dtype}")
    for t in (k_cache, v_cache, k_scale, v_scale):
        if t is not None and not t.is_contiguous():
            raise ValueError("cache tensors must be contiguous")
    nb, bs, hkv, d = k_cache.shape
    return KVCache(nb, bs, hkv, d, dt, k_cache.data_ptr(), v_cache.data_ptr(),
                   None if k_scale is None else k_scale.data_ptr(),
                   None if v_scale is None else v_scale.data_ptr())


def store_kv(k, v, slot_mapping, k_cache, v_cache, k_scale_new=None, v_scale_new=None,
             k_scale=None, v_scale=None) -> None:
    """pa_store_kv: write k/v (T, Hkv, D) to their slots (int64 (T,)), in place."""
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    k, v = k.contiguous(), v.contiguous()
    sm = slot_mapping.contiguous()
    _check(lib().pa_store_kv(_ptr(k), _ptr(v), _ptr(k_scale_new), _ptr(v_scale_new), _ptr(sm),
                             int(sm.numel()), ctypes.byref(cache), _stream()), "pa_store_kv")


def decode_workspace_size(k_cache, batch: int, num_heads: int, max_blocks_per_seq: int,
                          max_context_len: int = 0, v_cache=None, k_scale=None,
                          v_scale=None) -> int:
    cache = make_cache(k_cache, k_cache if v_cache is None else v_cache, k_scale, v_scale)
    return int(lib().pa_decode_workspace_size(ctypes.byref(cache), batch, num_heads,
                                              max_blocks_per_seq, max_context_len))


def decode(q, k_cache, v_cache, block_tables, context_lens, scale: float, *,
           max_context_len: int = 0, out=None, workspace=None, k_scale=None,
           v_scale=None) -> torch.Tensor:
    """pa_decode: q (B, H, D) bf16 -> out (B, H, D) bf16.

    max_context_len is the host-side bound of context_lens (0 = block-table
    capacity). A workspace (uint8 tensor) is allocated when none is given.
    """
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    B, H, D = q.shape
    bt = block_tables.contiguous()
    cl = context_lens.contiguous()
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.bfloat16, device=q.device)
    if workspace is None:  # a caller-provided workspace is checked by the library
        need = int(lib().pa_decode_workspace_size(ctypes.byref(cache), B, H, bt.shape[1],
                                                  max_context_len))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pa_decode(_ptr(q.contiguous()), ctypes.byref(cache), _ptr(bt), bt.shape[1],
                           _ptr(cl), int(max_context_len), B, H, float(scale), _ptr(out),
                           _ptr(workspace), ws_bytes, _stream()), "pa_decode")
    return out


def decode_window(q, k_cache, v_cache, block_tables, context_lens, scale: float, window: int,
                  sinks: int = 0, *, max_context_len: int = 0, out=None, workspace=None,
                  k_scale=None, v_scale=None) -> torch.Tensor:
    """pa_decode_window: decode attention over the last `window` keys and the
    first `sinks` keys of each sequence (window <= 0: all keys)."""
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    B, H, D = q.shape
    bt = block_tables.contiguous()
    cl = context_lens.contiguous()
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.bfloat16, device=q.device)
    if workspace is None:
        need = int(lib().pa_decode_workspace_size(ctypes.byref(cache), B, H, bt.shape[1],
                                                  max_context_len))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().pa_decode_window(_ptr(q.contiguous()), ctypes.byref(cache), _ptr(bt),
                                  bt.shape[1], _ptr(cl), int(max_context_len), B, H, float(scale),
                                  int(window), int(sinks), _ptr(out), _ptr(workspace), ws_bytes,
                                  _stream()), "pa_decode_window")
    return out


def decode_append(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                  scale: float, *, max_context_len: int = 0, out=None, workspace=None,
                  k_scale_new=None, v_scale_new=None, k_scale=None,
                  v_scale=None) -> torch.Tensor:
    """pa_decode_append: write each sequence's new K/V row (k_new/v_new
    (B, Hkv, D), cache dtype) at position context_len-1 through the block
    table, in place, and return decode attention over context_len keys."""
    return decode_window_append(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                                scale, 0, 0, max_context_len=max_context_len, out=out,
                                workspace=workspace, k_scale_new=k_scale_new,
                                v_scale_new=v_scale_new, k_scale=k_scale, v_scale=v_scale)


def decode_window_append(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens,
                         scale: float, window: int, sinks: int = 0, *, max_context_len: int = 0,
                         out=None, workspace=None, k_scale_new=None, v_scale_new=None,
                         k_scale=None, v_scale=None) -> torch.Tensor:
    """pa_decode_window_append (window 0: pa_decode_append): write each
    sequence's new K/V row at position context_len-1 through the block table,
    in place, and return decode attention over the last `window` keys and the
    first `sinks` keys (window <= 0: all context_len keys)."""
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    B, H, D = q.shape
    bt = block_tables.contiguous()
    cl = context_lens.contiguous()
    k_new, v_new = k_new.contiguous(), v_new.contiguous()
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.bfloat16, device=q.device)
    if workspace is None:
        need = int(lib().pa_decode_workspace_size(ctypes.byref(cache), B, H, bt.shape[1],
                                                  max_context_len))
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if int(window) > 0:
        rc = lib().pa_decode_window_append(
            _ptr(q.contiguous()), _ptr(k_new), _ptr(v_new), _ptr(k_scale_new), _ptr(v_scale_new),
            ctypes.byref(cache), _ptr(bt), bt.shape[1], _ptr(cl), int(max_context_len), B, H,
            float(scale), int(window), int(sinks), _ptr(out), _ptr(workspace), ws_bytes,
            _stream())
        _check(rc, "pa_decode_window_append")
    else:
        rc = lib().pa_decode_append(
            _ptr(q.contiguous()), _ptr(k_new), _ptr(v_new), _ptr(k_scale_new), _ptr(v_scale_new),
            ctypes.byref(cache), _ptr(bt), bt.shape[1], _ptr(cl), int(max_context_len), B, H,
            float(scale), _ptr(out), _ptr(workspace), ws_bytes, _stream())
        _check(rc, "pa_decode_append")
    return out


def prefill_varlen(q, k_cache, v_cache, block_tables, cu_seqlens_q, cu_seqlens_k,
                   scale: float, *, max_q_len: int = 0, out=None) -> torch.Tensor:
    """pa_prefill_varlen: packed q (total_q, H, D) bf16 -> out (total_q, H, D) bf16,
    attending over each sequence's paged K/V with the bottom-right causal mask.
    The new tokens' K/V must already be in the cache (store_kv)."""
    cache = make_cache(k_cache, v_cache)
    T, H, D = q.shape
    bt = block_tables.contiguous()
    cq, ck = cu_seqlens_q.contiguous(), cu_seqlens_k.contiguous()
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=q.device)
    _check(lib().pa_prefill_varlen(_ptr(q.contiguous()), ctypes.byref(cache), _ptr(bt),
                                   bt.shape[1], _ptr(cq), _ptr(ck), cq.numel() - 1, H, T,
                                   int(max_q_len), float(scale), _ptr(out), _stream()),
           "pa_prefill_varlen")
    return out


def decode_noalloc(q, k_cache, v_cache, block_tables, context_lens, scale: float, *,
                   max_context_len: int = 0, out=None, k_scale=None,
                   v_scale=None) -> torch.Tensor:
    """pa_decode_noalloc: pa_decode with the split-K scratch taken from the
    library's static device buffer instead of a caller workspace. For callers
    that cannot allocate device memory; `out` should then be passed in."""
    cache = make_cache(k_cache, v_cache, k_scale, v_scale)
    B, H, D = q.shape
    bt = block_tables.contiguous()
    cl = context_lens.contiguous()
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.bfloat16, device=q.device)
    _check(lib().pa_decode_noalloc(_ptr(q.contiguous()), ctypes.byref(cache), _ptr(bt),
                                   bt.shape[1], _ptr(cl), int(max_context_len), B, H,
                                   float(scale), _ptr(out), _stream()), "pa_decode_noalloc")
    return out


def debug_inject_wait_timeout(skip_copy: int, wait_limit_ns: int = 0) -> None:
    """pa_debug_inject_wait_timeout: arm (skip_copy >= 0) or disarm (< 0) the
    failure-detection test hook of the decode kernels."""
    _check(lib().pa_debug_inject_wait_timeout(int(skip_copy), int(wait_limit_ns)),
           "pa_debug_inject_wait_timeout")


def get_device_error() -> int:
    """Synchronise the device, return and clear its PA_DEVERR_* word."""
    code = ctypes.c_uint32(0)
    _check(lib().pa_get_device_error(ctypes.byref(code)), "pa_get_device_error")
    return int(code.value)
