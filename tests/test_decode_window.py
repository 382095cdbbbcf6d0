"""GPU sliding-window / attention-sink decode (pa_decode_window) against the
fp64 oracle's window reading: keys p < sinks and p >= context_len - window.

Tolerance as for pa_decode: max-abs 1e-2 beyond the bf16 output rounding and
relative L2 5e-3 over each call's outputs.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import assert_attention_close, host_copy, to_device

pytestmark = pytest.mark.gpu


def oracle_window(h, window, sinks):
    """The oracle's append of the new tokens, then its windowed decode."""
    if h.kv_dtype == "bf16":
        kc, vc = W.bf16_bits(h.k_cache).copy(), W.bf16_bits(h.v_cache).copy()
        oracle.store_kv(W.bf16_bits(h.k_new), W.bf16_bits(h.v_new), h.slot_mapping.numpy(), kc, vc)
        return oracle.decode(W.bf16_bits(h.q), kc, vc, h.block_tables.numpy(),
                             h.context_lens.numpy(), h.scale, window=window, sinks=sinks)
    kc, vc = W.u8(h.k_cache).copy(), W.u8(h.v_cache).copy()
    ks, vs = h.k_scale.numpy().copy(), h.v_scale.numpy().copy()
    oracle.store_kv(W.u8(h.k_new), W.u8(h.v_new), h.slot_mapping.numpy(), kc, vc,
                    h.k_scale_new.numpy(), h.v_scale_new.numpy(), ks, vs)
    return oracle.decode(W.bf16_bits(h.q), kc, vc, h.block_tables.numpy(),
                         h.context_lens.numpy(), h.scale, k_scale=ks, v_scale=vs,
                         window=window, sinks=sinks)


def gpu_window(g, window, sinks, max_context_len=0):
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, g.k_scale_new,
                g.v_scale_new, g.k_scale, g.v_scale)
    out = pa.decode_window(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                           window, sinks, max_context_len=max_context_len, k_scale=g.k_scale,
                           v_scale=g.v_scale)
    torch.cuda.synchronize()
    return out


CASES = [
    # (H, Hkv, D, bs, kv, lens, window, sinks)
    (8, 2, 64, 16, "bf16", [1, 17, 33, 100, 16, 15], 8, 0),       # window inside one block
    (8, 2, 64, 16, "bf16", [1, 17, 33, 100, 16, 15], 16, 4),      # sink and window blocks
    (32, 8, 128, 16, "bf16", [1, 15, 16, 17, 255, 3000, 4096], 100, 4),
    (32, 8, 128, 16, "bf16", [40, 41, 300], 20, 10),               # hole inside one block
    (32, 8, 128, 32, "bf16", [1, 31, 33, 65, 2049, 5000], 512, 3),
    (32, 8, 128, 32, "bf16", [70, 100], 64, 40),                   # sinks reach the window
    (8, 1, 128, 16, "bf16", [9, 300, 1025], 1, 0),                 # newest key only
    (64, 8, 128, 32, "fp8", [1, 31, 33, 1000, 5000], 256, 4),
    (16, 2, 128, 16, "fp8", [1, 16, 17, 300, 2500], 33, 17),
]


@pytest.mark.parametrize("case", CASES,
                         ids=lambda c: f"H{c[0]}kv{c[1]}D{c[2]}bs{c[3]}{c[4]}w{c[6]}s{c[7]}")
def test_window_decode_matches_oracle(case):
    H, Hkv, D, bs, kv, lens, window, sinks = case
    h = W.make_decode(len(lens), H, Hkv, D, bs, lens, seed=200 + window + sinks, kv_dtype=kv)
    want = oracle_window(h, window, sinks)
    got = gpu_window(to_device(h), window, sinks)
    assert pa.get_device_error() == 0
    assert_attention_close(got, want, str(case))


def test_window_zero_is_bit_identical_to_decode():
    lens = [5, 300, 1000, 4097]
    g = to_device(W.make_decode(4, 32, 8, 128, 16, lens, seed=210))
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    ref = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale)
    for window, sinks in [(0, 0), (0, 7), (-3, 2), (5000, 0)]:
        got = pa.decode_window(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                               window, sinks)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (window, sinks)


def test_window_changes_the_result():
    lens = [2000, 3000]
    h = W.make_decode(2, 32, 8, 128, 16, lens, seed=211)
    g = to_device(h)
    full = gpu_window(to_device(h), 0, 0)
    win = gpu_window(g, 256, 4)
    assert (full.float() - win.float()).abs().max() > 1e-2


def test_window_long_sequences_split_across_warps():
    lens = [70001, 30000]
    h = W.make_decode(2, 32, 8, 128, 16, lens, seed=212)
    want = oracle_window(h, 40000, 4)
    got = gpu_window(to_device(h), 40000, 4, max_context_len=max(lens))
    assert_attention_close(got, want, "long window")


def test_window_empty_and_short_sequences():
    gen = torch.Generator().manual_seed(213)
    lens = torch.randint(0, 80, (300,), generator=gen)
    lens[::13] = 0
    h = W.make_decode(300, 8, 2, 64, 16, lens.tolist(), seed=214)
    want = oracle_window(h, 24, 2)
    got = gpu_window(to_device(h), 24, 2)
    assert torch.all(got[lens == 0].float() == 0)
    assert_attention_close(got, want, "short window")


def test_window_full_size_long_context_every_sequence():
    g = W.make_workload("long_context_decode_b8", device="cuda")
    lens = g.meta["lens"]
    h = host_copy(g)  # before the GPU appends the new tokens
    window, sinks = 4096, 4
    got = gpu_window(g, window, sinks, max_context_len=max(lens))
    assert pa.get_device_error() == 0
    want = oracle_window(h, window, sinks)
    assert_attention_close(got, want, "long_context window")


def test_window_rejects_negative_sinks_and_large_batches():
    g = to_device(W.make_decode(2, 8, 2, 64, 16, [20, 40], seed=215))
    cache = pa.make_cache(g.k_cache, g.v_cache)
    L = pa.lib()
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    rc = L.pa_decode_window(ctypes.c_void_p(g.q.data_ptr()), ctypes.byref(cache),
                            ctypes.c_void_p(g.block_tables.data_ptr()), g.block_tables.shape[1],
                            ctypes.c_void_p(g.context_lens.data_ptr()), 0, 2, 8, g.scale, 8, -1,
                            ctypes.c_void_p(g.q.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                            ws.numel(), None)
    assert rc == 2  # PA_ERR_SHAPE
    B = 16500  # grid-split path: no window support
    need = pa.decode_workspace_size(g.k_cache, B, 8, g.block_tables.shape[1], 64)
    big = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    rc = L.pa_decode_window(ctypes.c_void_p(g.q.data_ptr()), ctypes.byref(cache),
                            ctypes.c_void_p(g.block_tables.data_ptr()), g.block_tables.shape[1],
                            ctypes.c_void_p(g.context_lens.data_ptr()), 64, B, 8, g.scale, 8, 0,
                            ctypes.c_void_p(g.q.data_ptr()), ctypes.c_void_p(big.data_ptr()),
                            big.numel(), None)
    assert rc == 4  # PA_ERR_UNSUPPORTED, nothing launched


APPEND_CASES = [
    # (H, Hkv, bs, kv, lens, window, sinks)
    (32, 8, 16, "bf16", [1, 5, 300, 1100, 5000, 2049, 0, 4100], 1024, 4),
    (32, 8, 16, "bf16", [40, 41, 300, 17], 20, 10),               # hole inside one block
    (8, 1, 16, "bf16", [9, 300, 1025], 1, 0),                     # newest key only
    (64, 8, 32, "fp8", [1, 31, 33, 1000, 5000], 256, 4),
    (64, 8, 32, "int8", [2, 64, 65, 3000], 100, 3),
]


@pytest.mark.parametrize("case", APPEND_CASES,
                         ids=lambda c: f"{c[3]}_w{c[5]}s{c[6]}_H{c[0]}kv{c[1]}bs{c[2]}")
def test_window_append_equals_store_then_window(case):
    # pa_decode_window_append: the new rows written by the decode's own warps,
    # then the window; bit-identical to pa_store_kv + pa_decode_window (outputs
    # and cache bytes) and within tolerance of the oracle
    H, Hkv, bs, kv, lens, window, sinks = case
    h = W.make_decode(len(lens), H, Hkv, 128, bs, lens, seed=211 + H + bs + window, kv_dtype=kv)
    want = oracle_window(h, window, sinks)
    fused, sep = to_device(h), to_device(h)
    got = pa.decode_window_append(fused.q, fused.k_new, fused.v_new, fused.k_cache, fused.v_cache,
                                  fused.block_tables, fused.context_lens, fused.scale, window,
                                  sinks, k_scale_new=fused.k_scale_new,
                                  v_scale_new=fused.v_scale_new, k_scale=fused.k_scale,
                                  v_scale=fused.v_scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    ref = gpu_window(sep, window, sinks)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(fused.k_cache.view(torch.uint8), sep.k_cache.view(torch.uint8))
    assert torch.equal(fused.v_cache.view(torch.uint8), sep.v_cache.view(torch.uint8))
    if kv != "bf16":
        assert torch.equal(fused.k_scale, sep.k_scale) and torch.equal(fused.v_scale, sep.v_scale)
    assert_attention_close(got, want, f"window append {case}")
    assert torch.all(got[torch.tensor(lens) == 0].float() == 0)
