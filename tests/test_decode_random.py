"""Seeded random decode cases against the fp64 oracle.

Each case draws a batch size, head counts and grouping, a block size, a KV
type (bf16, E4M3 or INT8 codes), a mix of context lengths (empty, within one
block, a few blocks, thousands of tokens) and, for half of the cases, a
sliding window with sinks; the fused store-and-attend call
(pa_decode_window_append, window 0 = pa_decode_append) runs once and every
output row is compared with the oracle's store then decode. The length mixes
put segment ends and warp-range boundaries in varied places, so the split of
the flattened blocks by work units, the straddling segments' partials and
their merges (with and without the arrival fast path) are all exercised.
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
    kv = ["bf16", "fp8", "int8"][seed % 3]
    if kv == "bf16":
        D = int(rng.choice([64, 128]))
        bs = int(rng.choice([16, 32]))
    else:
        D, bs = 128, int(rng.choice([16, 32]))
    Hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([1, 2, 3, 4, 8]))
    B = int(rng.choice([1, 3, 17, 64, 200, 700, 2600]))
    kind = rng.random(B)
    if rng.random() < 0.25:  # every segment under 8 blocks: blocks alone weigh the split
        lens = np.where(kind < 0.1, 0, rng.integers(1, 8 * bs, B))
    else:
        long_hi = 6000 if B <= 700 else 1500
        lens = np.where(kind < 0.1, 0,
                        np.where(kind < 0.3, rng.integers(1, bs + 1, B),
                                 np.where(kind < 0.8, rng.integers(bs, 8 * bs, B),
                                          rng.integers(500, long_hi, B))))
    window, sinks = 0, 0
    if rng.random() < 0.5:
        window = int(rng.choice([1, 7, 64, 300, 1024]))
        sinks = int(rng.choice([0, 1, 4, 16]))
    return dict(kv=kv, D=D, bs=bs, Hkv=Hkv, H=Hkv * G, B=B, lens=[int(x) for x in lens],
                window=window, sinks=sinks)


def oracle_case(h, c):
    if c["kv"] == "bf16":
        kc, vc = W.bf16_bits(h.k_cache).copy(), W.bf16_bits(h.v_cache).copy()
        oracle.store_kv(W.bf16_bits(h.k_new), W.bf16_bits(h.v_new), h.slot_mapping.numpy(), kc, vc)
        return oracle.decode(W.bf16_bits(h.q), kc, vc, h.block_tables.numpy(),
                             h.context_lens.numpy(), h.scale, window=c["window"],
                             sinks=c["sinks"])
    kc, vc = W.u8(h.k_cache).copy(), W.u8(h.v_cache).copy()
    ks, vs = h.k_scale.numpy().copy(), h.v_scale.numpy().copy()
    oracle.store_kv(W.u8(h.k_new), W.u8(h.v_new), h.slot_mapping.numpy(), kc, vc,
                    h.k_scale_new.numpy(), h.v_scale_new.numpy(), ks, vs)
    return oracle.decode(W.bf16_bits(h.q), kc, vc, h.block_tables.numpy(),
                         h.context_lens.numpy(), h.scale, k_scale=ks, v_scale=vs,
                         window=c["window"], sinks=c["sinks"])


@pytest.mark.parametrize("seed", range(32))
def test_random_case_matches_oracle(seed):
    c = draw_case(1000 + seed)
    h = W.make_decode(c["B"], c["H"], c["Hkv"], c["D"], c["bs"], c["lens"], seed=2000 + seed,
                      kv_dtype=c["kv"])
    want = oracle_case(h, c)
    g = to_device(h)
    got = pa.decode_window_append(g.q, g.k_new, g.v_new, g.k_cache, g.v_cache, g.block_tables,
                                  g.context_lens, g.scale, c["window"], c["sinks"],
                                  max_context_len=max(max(c["lens"]), 1),
                                  k_scale_new=g.k_scale_new, v_scale_new=g.v_scale_new,
                                  k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    assert torch.all(got[torch.tensor(c["lens"]) == 0].float() == 0)
    assert_attention_close(got, want, str({k: v for k, v in c.items() if k != "lens"}))
