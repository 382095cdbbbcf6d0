"""GPU store_kv (pa_store_kv) against the oracle's byte copy: bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import to_device

pytestmark = pytest.mark.gpu


def _gpu_store(d):
    pa.store_kv(d.k_new, d.v_new, d.slot_mapping, d.k_cache, d.v_cache, d.k_scale_new,
                d.v_scale_new, d.k_scale, d.v_scale)
    torch.cuda.synchronize()


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("dims", [(2, 64, 16), (8, 128, 16), (8, 128, 32)])
def test_store_kv_bit_exact_with_padding_slots(kv_dtype, dims):
    hkv, d, bs = dims
    if kv_dtype == "fp8" and d != 128:
        pytest.skip("FP8 caches are head_dim 128")
    lens = [1, 5, 16, 17, 33, 64, 3, 9]
    h = W.make_decode(len(lens), hkv, hkv, d, bs, lens, seed=40, kv_dtype=kv_dtype,
                      num_blocks=64)
    h.slot_mapping[2] = -1  # padding token
    g = to_device(h)
    _gpu_store(g)
    assert pa.get_device_error() == 0
    if kv_dtype == "bf16":
        kc, vc = W.bf16_bits(h.k_cache).copy(), W.bf16_bits(h.v_cache).copy()
        oracle.store_kv(W.bf16_bits(h.k_new), W.bf16_bits(h.v_new), h.slot_mapping.numpy(), kc, vc)
        np.testing.assert_array_equal(W.bf16_bits(g.k_cache), kc)
        np.testing.assert_array_equal(W.bf16_bits(g.v_cache), vc)
    else:
        kc, vc = W.u8(h.k_cache).copy(), W.u8(h.v_cache).copy()
        ks, vs = h.k_scale.numpy().copy(), h.v_scale.numpy().copy()
        oracle.store_kv(W.u8(h.k_new), W.u8(h.v_new), h.slot_mapping.numpy(), kc, vc,
                        h.k_scale_new.numpy(), h.v_scale_new.numpy(), ks, vs)
        np.testing.assert_array_equal(W.u8(g.k_cache), kc)
        np.testing.assert_array_equal(W.u8(g.v_cache), vc)
        np.testing.assert_array_equal(g.k_scale.cpu().numpy().view(np.uint32), ks.view(np.uint32))
        np.testing.assert_array_equal(g.v_scale.cpu().numpy().view(np.uint32), vs.view(np.uint32))


def test_store_kv_prefill_sized_batch_bit_exact():
    h = W.make_prefill(8, 32, 8, 128, 16, [0, 100, 2048, 7, 500, 1, 1000, 64],
                       [128, 1024, 300, 999, 129, 512, 640, 777], seed=41)
    g = to_device(h)
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    torch.cuda.synchronize()
    kc, vc = W.bf16_bits(h.k_cache).copy(), W.bf16_bits(h.v_cache).copy()
    oracle.store_kv(W.bf16_bits(h.k_new), W.bf16_bits(h.v_new), h.slot_mapping.numpy(), kc, vc)
    np.testing.assert_array_equal(W.bf16_bits(g.k_cache), kc)
    np.testing.assert_array_equal(W.bf16_bits(g.v_cache), vc)


def test_store_kv_slot_beyond_pool_is_skipped_and_flagged():
    h = W.make_decode(3, 2, 2, 64, 16, [4, 8, 12], seed=42, num_blocks=4)
    g = to_device(h)
    before = g.k_cache.clone()
    bad = g.slot_mapping.clone()
    bad[1] = 4 * 16  # one past the last slot of the pool
    pa.store_kv(g.k_new, g.v_new, bad, g.k_cache, g.v_cache)
    assert pa.get_device_error() & pa.PA_DEVERR_SLOT_RANGE
    assert pa.get_device_error() == 0  # the word was cleared
    flat_b, flat_a = before.view(-1, 2, 64), g.k_cache.view(-1, 2, 64)
    for t in (0, 2):
        s = int(bad[t])
        assert torch.equal(flat_a[s], g.k_new[t])
    changed = (flat_a != flat_b).any(dim=(1, 2)).nonzero().flatten().tolist()
    assert sorted(changed) == sorted(int(bad[t]) for t in (0, 2))
