"""Seeded random prefill cases against the fp64 oracle.

Each case draws the head grouping (1, 2, 4, 8 or 16 query heads per kv head),
the kv heads, the block size and a batch of sequences whose cached prefix
(0 to ~1500 tokens) and new-token count (0 to ~400) are drawn independently,
so query tiles start at varied offsets inside a sequence, cross sequence
boundaries in the packed rows, and meet the bottom-right mask at varied key
offsets. The new tokens are stored with pa_store_kv, pa_prefill_varlen runs
once, and every output row is compared with the oracle's store then prefill.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import assert_attention_close, to_device

pytestmark = pytest.mark.gpu


def draw_case(seed):
    rng = np.random.default_rng(seed)
    G = int(rng.choice([1, 2, 4, 8, 16]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    while G * Hkv > 64:
        Hkv //= 2
    bs = int(rng.choice([16, 32]))
    B = int(rng.integers(1, 7))
    kind = rng.random(B)
    cached = np.where(kind < 0.25, 0, rng.integers(1, 1500, B))
    q_lens = np.where(rng.random(B) < 0.1, 0,
                      np.where(rng.random(B) < 0.3, rng.integers(1, 9, B), rng.integers(9, 400, B)))
    if q_lens.sum() == 0:
        q_lens[0] = 1
    return dict(H=G * Hkv, Hkv=Hkv, bs=bs, cached=[int(x) for x in cached],
                q_lens=[int(x) for x in q_lens])


@pytest.mark.parametrize("seed", range(20))
def test_random_prefill_matches_oracle(seed):
    c = draw_case(3000 + seed)
    h = W.make_prefill(len(c["q_lens"]), c["H"], c["Hkv"], 128, c["bs"], c["cached"], c["q_lens"],
                       seed=4000 + seed)
    kc, vc = W.bf16_bits(h.k_cache).copy(), W.bf16_bits(h.v_cache).copy()
    oracle.store_kv(W.bf16_bits(h.k_new), W.bf16_bits(h.v_new), h.slot_mapping.numpy(), kc, vc)
    want = oracle.prefill(W.bf16_bits(h.q), kc, vc, h.block_tables.numpy(),
                          h.cu_seqlens_q.numpy(), h.cu_seqlens_k.numpy(), h.scale)
    g = to_device(h)
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    got = pa.prefill_varlen(g.q, g.k_cache, g.v_cache, g.block_tables, g.cu_seqlens_q,
                            g.cu_seqlens_k, g.scale, max_q_len=max(c["q_lens"]))
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    assert_attention_close(got, want, str(c))
