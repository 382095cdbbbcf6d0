"""pa_decode_noalloc: the decode entry point for callers that cannot allocate.

Some callers have no device allocator of their own (a plain C program that
is handed device pointers by another runtime), or run inside a serving
engine whose KV-block pool has reserved nearly all device memory, so they
cannot give pa_decode a workspace. This entry point takes the split-K
scratch from a static buffer inside the library instead.

The tests call it through the C ABI twice in a row (the second call finds
the first call's partials still in the buffer) and check each output against
pa_decode's with the decode tolerance, and against the oracle; then a run of
calls whose batch, head grouping and cache type change from call to call
(so the buffer's layout moves between calls) through the Python binding.
This file is collected last; it also passes alone in a fresh process (its
first call does the per-device set-up).
"""
import ctypes

import pytest
import torch

import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import ATOL, REL_L2, assert_attention_close, oracle_store_and_decode, to_device

pytestmark = pytest.mark.gpu


def _noalloc_c_abi(g, out, max_context_len):
    cache = pa.make_cache(g.k_cache, g.v_cache, g.k_scale, g.v_scale)
    B, H, _ = g.q.shape
    return pa.lib().pa_decode_noalloc(
        ctypes.c_void_p(g.q.data_ptr()), ctypes.byref(cache),
        ctypes.c_void_p(g.block_tables.data_ptr()), g.block_tables.shape[1],
        ctypes.c_void_p(g.context_lens.data_ptr()), max_context_len, B, H, g.scale,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _close(a, b):
    d = (a.float() - b.float()).abs()
    rel = float(torch.linalg.vector_norm(a.float() - b.float()) /
                torch.linalg.vector_norm(b.float()))
    return float(d.max()) <= ATOL and rel <= REL_L2


def _prepare(lens, H, Hkv, bs, kv, seed):
    h = W.make_decode(len(lens), H, Hkv, 128, bs, lens, seed=seed, kv_dtype=kv)
    want = oracle_store_and_decode(h)
    g = to_device(h)
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, g.k_scale_new,
                g.v_scale_new, g.k_scale, g.v_scale)
    return g, want


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_noalloc_matches_decode_on_two_calls_in_a_row(kv):
    # lengths long enough that several sequences need split-K scratch
    lens = [3000, 17, 4096, 1, 1500, 2200]
    H, Hkv, bs = (32, 8, 16) if kv == "bf16" else (64, 8, 32)
    g, want = _prepare(lens, H, Hkv, bs, kv, seed=70)
    assert pa.decode_workspace_size(g.k_cache, len(lens), H, g.block_tables.shape[1],
                                    max(lens), k_scale=g.k_scale, v_scale=g.v_scale) > 0
    ref = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                    max_context_len=max(lens), k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    assert_attention_close(ref, want, "pa_decode")
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_c_abi(g, out, max(lens)) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert _close(out, ref), f"call {call} differs from pa_decode"
        assert_attention_close(out, want, f"noalloc call {call}")
    assert pa.get_device_error() == 0


def test_noalloc_calls_with_changing_shapes():
    # each call lays the static buffer out for its own shape (partial slots,
    # then counters): a shrinking batch and a changing head grouping leave
    # the previous call's partials where this call's counters now sit
    shapes = [
        ([4096, 3000, 2500, 1700, 900, 4000, 3500, 2048] * 8, 32, 8, 16, "bf16"),
        ([5000, 1200, 3300, 800, 2600, 64], 64, 8, 32, "fp8"),
        ([2049, 4000, 777], 8, 1, 16, "bf16"),
        ([6000, 3000], 32, 8, 16, "int8"),
        ([4096, 3000, 2500, 1700, 900, 4000, 3500, 2048] * 8, 32, 8, 16, "bf16"),
    ]
    for i, (lens, H, Hkv, bs, kv, ) in enumerate(shapes):
        g, want = _prepare(lens, H, Hkv, bs, kv, seed=72 + i)
        ref = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                        max_context_len=max(lens), k_scale=g.k_scale, v_scale=g.v_scale)
        out = torch.full_like(ref, float("nan"))
        out = pa.decode_noalloc(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens,
                                g.scale, max_context_len=max(lens), out=out, k_scale=g.k_scale,
                                v_scale=g.v_scale)
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        assert _close(out, ref), f"shape {i} differs from pa_decode"
        assert_attention_close(out, want, f"noalloc shape {i} ({kv}, {H}/{Hkv}, B={len(lens)})")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    g = to_device(W.make_decode(2, 64, 8, 128, 32, [40, 70], seed=71, kv_dtype="fp8"))
    # claimed shape: a batch above the persistent kernel's 16384 sequences (the
    # grid-split path), whose split-K scratch grows with batch x context and
    # far exceeds the static buffer
    B, H = 17000, 64
    need = pa.decode_workspace_size(g.k_cache, B, H, 512, 16384, k_scale=g.k_scale,
                                    v_scale=g.v_scale)
    assert need > pa.DECODE_NOALLOC_SCRATCH_BYTES
    cache = pa.make_cache(g.k_cache, g.v_cache, g.k_scale, g.v_scale)
    rc = pa.lib().pa_decode_noalloc(ctypes.c_void_p(g.q.data_ptr()), ctypes.byref(cache),
                                    ctypes.c_void_p(g.block_tables.data_ptr()), 512,
                                    ctypes.c_void_p(g.context_lens.data_ptr()), 16384, B, H,
                                    g.scale, ctypes.c_void_p(g.q.data_ptr()), None)
    assert rc == 8  # PA_ERR_TOO_LARGE, nothing launched
