"""pa_decode_noalloc: the decode entry point for callers that cannot allocate.

Callers without a device allocator of their own (a plain C program handed
device pointers by another runtime), or whose device memory is fully reserved
by a serving engine's KV pool, cannot pass pa_decode a workspace. This entry
point takes the split-K scratch from a static buffer inside the library. The
test calls it through the C ABI twice in a row (the second call finds the
first call's partials still in the buffer) and checks each output against
pa_decode's with the decode tolerance. It runs last in the suite and also
passes alone in a fresh process (its first call does the per-device set-up).
"""
import ctypes

import pytest
import torch

import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import ATOL, REL_L2, to_device

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


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_noalloc_matches_decode_on_two_calls_in_a_row(kv):
    # lengths long enough that several sequences need split-K scratch
    lens = [3000, 17, 4096, 1, 1500, 2200]
    H, Hkv, bs = (32, 8, 16) if kv == "bf16" else (64, 8, 32)
    g = to_device(W.make_decode(len(lens), H, Hkv, 128, bs, lens, seed=70, kv_dtype=kv))
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, g.k_scale_new,
                g.v_scale_new, g.k_scale, g.v_scale)
    assert pa.decode_workspace_size(g.k_cache, len(lens), H, g.block_tables.shape[1],
                                    max(lens), k_scale=g.k_scale, v_scale=g.v_scale) > 0
    ref = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                    max_context_len=max(lens), k_scale=g.k_scale, v_scale=g.v_scale)
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _noalloc_c_abi(g, out, max(lens)) == 0
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        assert _close(out, ref)
    assert pa.get_device_error() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch():
    g = to_device(W.make_decode(2, 64, 8, 128, 32, [40, 70], seed=71, kv_dtype="fp8"))
    # claimed shape: a batch large enough for the grid-split path, whose split-K
    # scratch grows with batch x context and far exceeds the static buffer
    B, H = 4096, 64
    need = pa.decode_workspace_size(g.k_cache, B, H, 512, 16384, k_scale=g.k_scale,
                                    v_scale=g.v_scale)
    assert need > pa.DECODE_NOALLOC_SCRATCH_BYTES
    cache = pa.make_cache(g.k_cache, g.v_cache, g.k_scale, g.v_scale)
    rc = pa.lib().pa_decode_noalloc(ctypes.c_void_p(g.q.data_ptr()), ctypes.byref(cache),
                                    ctypes.c_void_p(g.block_tables.data_ptr()), 512,
                                    ctypes.c_void_p(g.context_lens.data_ptr()), 16384, B, H,
                                    g.scale, ctypes.c_void_p(g.q.data_ptr()), None)
    assert rc == 8  # PA_ERR_TOO_LARGE, nothing launched
