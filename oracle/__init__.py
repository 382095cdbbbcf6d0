"""CPU oracle for paged-KV-cache attention (test infrastructure).

This package is the ground truth the CUDA library is checked against. Only the
test-suite, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may
import it; the library itself never does. It shares no code with the CUDA
path: the arithmetic lives in ``pa_oracle.c`` (plain C, IEEE double, straight
loops), compiled here with gcc into ``_pa_oracle.so`` and called via ctypes.

Every function takes numpy arrays holding the raw stored bits (bf16 as
uint16, FP8-E4M3 as uint8) and returns float64 results.

Page references (titles of the source pages):
  * "Decode Phase Attention Forward Pass": decode semantics, GQA head map,
    context_lens including the just-stored token, the zero-padding caveat.
  * "tiny-vllm part 05": block / offset arithmetic of the K/V append.
  * "Prefill Forward Prefix Caching Explained": packed varlen prefill and the
    bottom-right causal mask.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_pa_oracle.so")
_lock = threading.Lock()
_lib = None

KV_BF16 = 0
KV_E4M3 = 1
KV_INT8 = 2

_ERRORS = {1: "bad argument", 2: "index or length out of range", 3: "out of memory"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with gcc (no fast-math: IEEE double semantics)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_e4m3_to_double.restype = dbl
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode_array.restype = None
        lib.oracle_e4m3_decode_array.argtypes = [P, i64, P]
        lib.oracle_store_kv.restype = i32
        lib.oracle_store_kv.argtypes = [P, P, P, i64, i64, i64, i64, P, P, P, P, P, P, i64]
        lib.oracle_decode.restype = i32
        lib.oracle_decode.argtypes = [P, P, P, i32, P, P, i64, i32, i32, i32, P, i32, P, i32, i32,
                                      dbl, P, i32]
        lib.oracle_decode_window.restype = i32
        lib.oracle_decode_window.argtypes = [P, P, P, i32, P, P, i64, i32, i32, i32, P, i32, P,
                                             i32, i32, ctypes.c_double, i64, i64, P, i32]
        lib.oracle_decode_split.restype = i32
        lib.oracle_decode_split.argtypes = [P, P, P, i32, P, P, i64, i32, i32, i32, P, i32, P, i32,
                                            i32, dbl, i32, P]
        lib.oracle_causal_mask.restype = i32
        lib.oracle_causal_mask.argtypes = [i32, i32, P]
        lib.oracle_prefill.restype = i32
        lib.oracle_prefill.argtypes = [P, P, P, i32, P, P, i64, i32, i32, i32, P, i32, P, P, i32,
                                       i32, dbl, P, i32]
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _check(rc):
    if rc != 0:
        raise OracleError(_ERRORS.get(rc, f"error {rc}"))


def default_threads() -> int:
    return len(os.sched_getaffinity(0))


def e4m3_to_double(codes) -> np.ndarray:
    """Decode OCP E4M3 byte codes to float64 (from the format definition)."""
    codes = _c(codes, np.uint8)
    out = np.empty(codes.shape, np.float64)
    _load().oracle_e4m3_decode_array(_ptr(codes), codes.size, _ptr(out))
    return out


def store_kv(k, v, slot_mapping, k_cache, v_cache, k_scale_new=None, v_scale_new=None,
             k_scale_cache=None, v_scale_cache=None) -> None:
    """Write new K/V rows into cache slots in place (byte copy).

    k, v: (T, Hkv, D) uint16 (bf16 bits) or uint8 (E4M3); caches:
    (num_blocks, block_size, Hkv, D) of the same dtype, modified in place;
    slot_mapping (T,) int64, slot = block * block_size + offset, < 0 skips.
    FP8 scales: new (T, Hkv) fp32 -> caches (num_blocks, Hkv, block_size).
    """
    T = k.shape[0]
    row_bytes = k[0].nbytes if T else k_cache[0, 0].nbytes
    num_slots = k_cache.shape[0] * k_cache.shape[1]
    block_size = k_cache.shape[1]
    hkv = k_cache.shape[2]
    for a in (k_cache, v_cache, k_scale_cache, v_scale_cache):
        if a is not None and not a.flags.c_contiguous:
            raise OracleError("caches must be C-contiguous (modified in place)")
    k, v = np.ascontiguousarray(k), np.ascontiguousarray(v)
    sm = _c(slot_mapping, np.int64)
    ks = None if k_scale_new is None else _c(k_scale_new, np.float32)
    vs = None if v_scale_new is None else _c(v_scale_new, np.float32)
    _check(_load().oracle_store_kv(_ptr(k), _ptr(v), _ptr(sm), T, row_bytes, num_slots,
                                   block_size, _ptr(k_cache), _ptr(v_cache), _ptr(ks), _ptr(vs),
                                   _ptr(k_scale_cache), _ptr(v_scale_cache), hkv))


def _cache_args(k_cache, v_cache, k_scale, v_scale):
    if k_cache.dtype == np.uint16:
        dtype = KV_BF16
    elif k_cache.dtype == np.uint8:
        dtype = KV_E4M3
    elif k_cache.dtype == np.int8:
        dtype = KV_INT8
    else:
        raise OracleError("cache must hold bf16 bits (uint16), E4M3 bytes (uint8) or INT8 "
                          "codes (int8)")
    kc, vc = np.ascontiguousarray(k_cache), np.ascontiguousarray(v_cache)
    ks = None if k_scale is None else _c(k_scale, np.float32)
    vs = None if v_scale is None else _c(v_scale, np.float32)
    nb, bs, hkv, d = kc.shape
    return (kc, vc, ks, vs), (_ptr(kc), _ptr(vc), dtype, _ptr(ks), _ptr(vs), nb, bs, hkv, d)


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale=None, v_scale=None,
           threads: int | None = None, window: int = 0, sinks: int = 0) -> np.ndarray:
    """Single-query paged decode attention in float64.

    q: (B, H, D) uint16 bf16 bits. Caches (num_blocks, block_size, Hkv, D):
    bf16 bits (uint16), E4M3 bytes (uint8) or INT8 codes (int8), the latter two
    with scales (num_blocks, Hkv, block_size). block_tables (B, max_blocks)
    int32; context_lens (B,) int32. window > 0: only the last `window` keys and
    the first `sinks` keys of each sequence are attended.
    Returns (B, H, D) float64.
    """
    q = _c(q, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    keep, cargs = _cache_args(k_cache, v_cache, k_scale, v_scale)
    B, H, D = q.shape
    out = np.zeros((B, H, D), np.float64)
    _check(_load().oracle_decode_window(_ptr(q), *cargs, _ptr(bt), bt.shape[1], _ptr(cl), B, H,
                                        float(scale), int(window), int(sinks), _ptr(out),
                                        threads or default_threads()))
    del keep
    return out


def decode_split(q, k_cache, v_cache, block_tables, context_lens, scale, split_tokens,
                 k_scale=None, v_scale=None) -> np.ndarray:
    """Decode computed per chunk of split_tokens keys, then merged (flash-decoding)."""
    q = _c(q, np.uint16)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    keep, cargs = _cache_args(k_cache, v_cache, k_scale, v_scale)
    B, H, D = q.shape
    out = np.zeros((B, H, D), np.float64)
    _check(_load().oracle_decode_split(_ptr(q), *cargs, _ptr(bt), bt.shape[1], _ptr(cl), B, H,
                                       float(scale), int(split_tokens), _ptr(out)))
    del keep
    return out


def causal_mask(q_len: int, kv_len: int) -> np.ndarray:
    """Bottom-right-aligned causal mask, (q_len, kv_len) uint8, 1 = visible."""
    m = np.zeros((q_len, kv_len), np.uint8)
    _check(_load().oracle_causal_mask(q_len, kv_len, _ptr(m)))
    return m


def prefill(q, k_cache, v_cache, block_tables, cu_seqlens_q, cu_seqlens_k, scale, k_scale=None,
            v_scale=None, threads: int | None = None) -> np.ndarray:
    """Varlen prefix-cached prefill with the bottom-right causal mask, float64.

    q: (total_q, H, D) uint16 bf16 bits, packed by cu_seqlens_q (B+1,).
    cu_seqlens_k (B+1,) gives each sequence's kv_len = cached + new.
    Returns (total_q, H, D) float64.
    """
    q = _c(q, np.uint16)
    bt = _c(block_tables, np.int32)
    cq = _c(cu_seqlens_q, np.int32)
    ck = _c(cu_seqlens_k, np.int32)
    keep, cargs = _cache_args(k_cache, v_cache, k_scale, v_scale)
    T, H, D = q.shape
    B = cq.shape[0] - 1
    if cq[-1] != T:
        raise OracleError("cu_seqlens_q[-1] must equal the number of packed rows")
    out = np.zeros((T, H, D), np.float64)
    _check(_load().oracle_prefill(_ptr(q), *cargs, _ptr(bt), bt.shape[1], _ptr(cq), _ptr(ck), B,
                                  H, float(scale), _ptr(out), threads or default_threads()))
    del keep
    return out
