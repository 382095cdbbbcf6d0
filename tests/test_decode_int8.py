"""GPU decode over an INT8 KV cache (signed codes, one fp32 scale per (slot,
kv head)) against the fp64 oracle's INT8 reading: element = code * scale.

Store is bit-exact (codes and scales); attention outputs use the decode
tolerance (max-abs 1e-2 beyond the bf16 output rounding, relative L2 5e-3).
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import assert_attention_close, host_copy, oracle_store_and_decode, to_device
from test_decode_window import gpu_window, oracle_window

pytestmark = pytest.mark.gpu


def gpu_store_decode(g, max_context_len=0):
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, g.k_scale_new,
                g.v_scale_new, g.k_scale, g.v_scale)
    out = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                    max_context_len=max_context_len, k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    return out


CASES = [
    # (H, Hkv, bs, lens): head_dim 128
    (64, 8, 32, [1, 31, 32, 33, 1000, 5000]),
    (16, 2, 16, [1, 16, 17, 300, 2500]),
    (32, 8, 16, [2, 255, 4096]),
    (8, 8, 32, [7, 64, 65]),  # group 1
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"H{c[0]}kv{c[1]}bs{c[2]}")
def test_int8_decode_matches_oracle(case):
    H, Hkv, bs, lens = case
    h = W.make_decode(len(lens), H, Hkv, 128, bs, lens, seed=300 + H + bs, kv_dtype="int8")
    want = oracle_store_and_decode(h)
    got = gpu_store_decode(to_device(h))
    assert pa.get_device_error() == 0
    assert_attention_close(got, want, str(case))


def test_int8_store_is_bit_exact():
    lens = [1, 17, 40]
    h = W.make_decode(3, 16, 2, 128, 16, lens, seed=310, kv_dtype="int8")
    g = to_device(h)
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, g.k_scale_new,
                g.v_scale_new, g.k_scale, g.v_scale)
    torch.cuda.synchronize()
    kf = g.k_cache.view(-1, 2, 128)
    for i, s in enumerate(h.slot_mapping.tolist()):
        assert torch.equal(kf[s], g.k_new[i])
        blk, off = s // 16, s % 16
        assert torch.equal(g.k_scale[blk, :, off], g.k_scale_new[i])
        assert torch.equal(g.v_scale[blk, :, off], g.v_scale_new[i])


def test_int8_context_len_one_returns_dequantised_v():
    h = W.make_decode(2, 16, 2, 128, 32, [1, 1], seed=311, kv_dtype="int8")
    want = oracle_store_and_decode(h)
    got = gpu_store_decode(to_device(h)).float().cpu().double().numpy()
    # the exact result is one V row, code * scale. The kernel folds the V
    # scale into the probability in f16 (relative rounding <= 2^-11) and
    # rounds the output to bf16 (<= 2^-8): within one bf16 step of it.
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -7)


def test_int8_fused_append_matches_separate_calls():
    lens = [1, 31, 32, 33, 1000]
    h = W.make_decode(len(lens), 64, 8, 128, 32, lens, seed=312, kv_dtype="int8")
    a, b = to_device(h), to_device(h)
    got = pa.decode_append(a.q, a.k_new, a.v_new, a.k_cache, a.v_cache, a.block_tables,
                           a.context_lens, a.scale, k_scale_new=a.k_scale_new,
                           v_scale_new=a.v_scale_new, k_scale=a.k_scale, v_scale=a.v_scale)
    ref = gpu_store_decode(b)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(a.k_cache, b.k_cache) and torch.equal(a.v_cache, b.v_cache)
    assert torch.equal(a.k_scale, b.k_scale) and torch.equal(a.v_scale, b.v_scale)


def test_int8_window_matches_oracle():
    lens = [1, 31, 33, 1000, 5000]
    h = W.make_decode(len(lens), 64, 8, 128, 32, lens, seed=313, kv_dtype="int8")
    want = oracle_window(h, 200, 4)
    got = gpu_window(to_device(h), 200, 4)
    assert_attention_close(got, want, "int8 window")


def test_int8_full_size_workload_every_sequence():
    g = W.make_workload("llama3_70b_int8_decode_b256", device="cuda")
    lens = g.meta["lens"]
    h = host_copy(g)  # before the GPU appends the new tokens
    got = gpu_store_decode(g, max_context_len=max(lens))
    assert pa.get_device_error() == 0
    want = oracle_store_and_decode(h)
    assert_attention_close(got, want, "llama3_70b_int8_decode_b256")
