"""GPU varlen prefix-cached prefill (pa_store_kv + pa_prefill_varlen) against
the fp64 oracle, with the decode tolerance (bf16 output, fp32 accumulation).

Small cases are compared in full. The full-size workload is compared on every
row of its two shortest sequences and on sampled query rows of every
sequence: row i of sequence b sees keys 0..i+cached, which the oracle's
prefill computes as a one-row sequence with kv_len = i + cached + 1 over the
same block-table row (a pinned identity of the oracle).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import assert_attention_close, oracle_store_and_decode, to_device

pytestmark = pytest.mark.gpu


def oracle_full(h):
    kc, vc = W.bf16_bits(h.k_cache).copy(), W.bf16_bits(h.v_cache).copy()
    oracle.store_kv(W.bf16_bits(h.k_new), W.bf16_bits(h.v_new), h.slot_mapping.numpy(), kc, vc)
    return oracle.prefill(W.bf16_bits(h.q), kc, vc, h.block_tables.numpy(),
                          h.cu_seqlens_q.numpy(), h.cu_seqlens_k.numpy(), h.scale)


def gpu_prefill(g, max_q_len=0):
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    out = pa.prefill_varlen(g.q, g.k_cache, g.v_cache, g.block_tables, g.cu_seqlens_q,
                            g.cu_seqlens_k, g.scale, max_q_len=max_q_len)
    torch.cuda.synchronize()
    return out


def run_case(H, Hkv, bs, cached, q_lens, seed):
    h = W.make_prefill(len(q_lens), H, Hkv, 128, bs, cached, q_lens, seed=seed)
    want = oracle_full(h)
    g = to_device(h)
    got = gpu_prefill(g, max_q_len=max(q_lens))
    assert pa.get_device_error() == 0
    return got, want


def test_single_tile_prefill():
    # one 128-row tile (32 tokens x 4 heads), one 128-key tile
    got, want = run_case(4, 1, 16, [40], [32], seed=80)
    assert_attention_close(got, want, "single tile")


def test_no_prefix_is_causal_attention():
    got, want = run_case(8, 2, 16, [0, 0], [77, 128], seed=81)
    assert_attention_close(got, want, "cached=0")


CASES = [
    # (H, Hkv, bs, cached, q_lens)
    (32, 8, 16, [0, 100, 2048, 7], [128, 300, 129, 1000]),
    (32, 8, 32, [5, 1000], [1, 255]),
    (8, 8, 16, [64, 0], [33, 17]),          # group 1
    (16, 8, 16, [300], [200]),              # group 2
    (64, 8, 32, [128, 900], [256, 65]),     # group 8
    (16, 1, 16, [17], [40]),                # group 16
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"H{c[0]}kv{c[1]}bs{c[2]}")
def test_prefill_matches_oracle(case):
    H, Hkv, bs, cached, q_lens = case
    got, want = run_case(H, Hkv, bs, cached, q_lens, seed=82 + H + bs)
    assert_attention_close(got, want, str(case))


def test_single_query_rows_equal_decode():
    # q_len = 1 per sequence: prefill degenerates to decode over kv_len keys;
    # both are checked against the oracle's decode of the same cache
    lens = [1, 100, 2049]
    d = W.make_decode(3, 32, 8, 128, 16, lens, seed=83)
    want = oracle_store_and_decode(d)
    g = to_device(d)
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache)
    dec = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale)
    cu_q = torch.arange(4, dtype=torch.int32, device="cuda")
    cu_k = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
    pre = pa.prefill_varlen(g.q, g.k_cache, g.v_cache, g.block_tables, cu_q, cu_k, g.scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    assert_attention_close(pre, want, "prefill with q_len 1")
    assert_attention_close(dec, want, "decode")
    diff = (pre.float() - dec.float()).abs().max().item()
    assert diff <= 2e-2  # two bf16 results of the same attention


def test_full_size_workload_rows():
    # every row of the two shortest sequences, plus sampled rows of every
    # sequence (row i of sequence b sees keys 0 .. cached_b + i: the oracle's
    # prefill of a one-row sequence with that kv_len over the same table row)
    g = W.make_workload("varlen_prefill_b8", device="cuda")
    m = g.meta
    h_cache = (g.k_cache.cpu(), g.v_cache.cpu())  # before the GPU stores the new tokens
    got = gpu_prefill(g, max_q_len=max(m["q_lens"]))
    assert pa.get_device_error() == 0
    assert torch.isfinite(got.float()).all()
    kc, vc = W.bf16_bits(h_cache[0]).copy(), W.bf16_bits(h_cache[1]).copy()
    oracle.store_kv(W.bf16_bits(g.k_new), W.bf16_bits(g.v_new), g.slot_mapping.cpu().numpy(),
                    kc, vc)
    cu_q_all = g.cu_seqlens_q.cpu().numpy()
    cu_k_all = g.cu_seqlens_k.cpu().numpy()
    bt_all = g.block_tables.cpu().numpy()
    q_bits = W.bf16_bits(g.q)
    # the two shortest sequences in full
    short = sorted(np.argsort(m["q_lens"], kind="stable")[:2].tolist())
    rows = np.concatenate([np.arange(cu_q_all[b], cu_q_all[b + 1]) for b in short])
    cu_q = np.concatenate([[0], np.cumsum([cu_q_all[b + 1] - cu_q_all[b] for b in short])])
    cu_k = np.concatenate([[0], np.cumsum([cu_k_all[b + 1] - cu_k_all[b] for b in short])])
    want = oracle.prefill(q_bits[rows], kc, vc, bt_all[short], cu_q.astype(np.int32),
                          cu_k.astype(np.int32), g.scale)
    assert_attention_close(got[torch.as_tensor(rows)], want, "two shortest sequences in full")
    # sampled rows of every sequence
    gen = torch.Generator().manual_seed(7)
    rows, seqs, kvs = [], [], []
    for b in range(len(m["q_lens"])):
        ql = m["q_lens"][b]
        picks = sorted(set([0, ql - 1] + torch.randint(0, ql, (4,), generator=gen).tolist()))
        for i in picks:
            rows.append(int(cu_q_all[b]) + i)
            seqs.append(b)
            kvs.append(m["cached"][b] + i + 1)
    cu_q = np.arange(len(rows) + 1, dtype=np.int32)
    cu_k = np.concatenate([[0], np.cumsum(kvs)]).astype(np.int32)
    want = oracle.prefill(q_bits[rows], kc, vc, bt_all[seqs], cu_q, cu_k, g.scale)
    assert_attention_close(got[rows], want, "varlen_prefill_b8 sampled rows")
