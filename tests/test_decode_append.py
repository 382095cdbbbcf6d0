"""GPU fused append + decode (pa_decode_append) against pa_store_kv + pa_decode
and against the fp64 oracle.

pa_decode_append must leave the cache exactly as pa_store_kv with the slot
of position context_len-1 does, and return exactly pa_decode's output
afterwards (the same kernel attends to the same bytes), so both comparisons
are bit-exact. The oracle comparison uses the attention tolerance (max-abs
1e-2 beyond the bf16 output rounding, relative L2 5e-3).
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import assert_attention_close, host_copy, oracle_store_and_decode, to_device

pytestmark = pytest.mark.gpu


def _clone(g):
    d = {k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in g.__dict__.items()}
    return type(g)(**d)


def fused(g, max_context_len=0):
    out = pa.decode_append(g.q, g.k_new, g.v_new, g.k_cache, g.v_cache, g.block_tables,
                           g.context_lens, g.scale, max_context_len=max_context_len,
                           k_scale_new=g.k_scale_new, v_scale_new=g.v_scale_new,
                           k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    return out


def separate(g, max_context_len=0):
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, g.k_scale_new,
                g.v_scale_new, g.k_scale, g.v_scale)
    out = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                    max_context_len=max_context_len, k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    return out


def assert_same_as_separate(g, max_context_len=0):
    """Run both paths on copies of the same device inputs; bit-exact compare."""
    a, b = _clone(g), _clone(g)
    got = fused(a, max_context_len)
    assert pa.get_device_error() == 0
    ref = separate(b, max_context_len)
    assert pa.get_device_error() == 0
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), "outputs differ"
    assert torch.equal(a.k_cache.view(torch.uint8), b.k_cache.view(torch.uint8)), "k cache differs"
    assert torch.equal(a.v_cache.view(torch.uint8), b.v_cache.view(torch.uint8)), "v cache differs"
    if g.k_scale is not None:
        assert torch.equal(a.k_scale, b.k_scale) and torch.equal(a.v_scale, b.v_scale)
    return got


CASES = [
    # (H, Hkv, D, bs, kv, lens): new token at the start, middle and end of a block
    (8, 2, 64, 16, "bf16", [1, 17, 33, 100, 16, 15]),
    (32, 8, 128, 16, "bf16", [1, 15, 16, 17, 255, 256, 257, 3000, 700, 4096]),
    (32, 8, 128, 32, "bf16", [1, 31, 32, 33, 63, 64, 65, 2049, 5000]),
    (8, 1, 128, 16, "bf16", [9, 300, 1025]),
    (64, 8, 128, 32, "fp8", [1, 31, 32, 33, 1000, 5000]),
    (16, 2, 128, 16, "fp8", [1, 16, 17, 300, 2500]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"H{c[0]}kv{c[1]}D{c[2]}bs{c[3]}{c[4]}")
def test_append_matches_oracle_and_separate_calls(case):
    H, Hkv, D, bs, kv, lens = case
    h = W.make_decode(len(lens), H, Hkv, D, bs, lens, seed=150 + H + D + bs, kv_dtype=kv)
    want = oracle_store_and_decode(h)
    g = to_device(h)
    got = assert_same_as_separate(g)
    assert_attention_close(got, want, str(case))


def test_append_cache_rows_equal_the_new_tokens():
    lens = [1, 16, 17, 40, 0, 33]
    h = W.make_decode(len(lens), 8, 2, 128, 16, lens, seed=161)
    g = to_device(h)
    fused(g)
    assert pa.get_device_error() == 0
    kflat = g.k_cache.view(-1, 2, 128)
    vflat = g.v_cache.view(-1, 2, 128)
    for i, L in enumerate(lens):
        if L == 0:
            continue
        s = int(h.slot_mapping[i])
        assert torch.equal(kflat[s].view(torch.int16), g.k_new[i].view(torch.int16))
        assert torch.equal(vflat[s].view(torch.int16), g.v_new[i].view(torch.int16))


def test_append_leaves_other_slots_untouched():
    lens = [5, 70, 33]
    h = W.make_decode(len(lens), 8, 2, 64, 16, lens, seed=162)
    g = to_device(h)
    before_k, before_v = g.k_cache.clone(), g.v_cache.clone()
    fused(g)
    assert pa.get_device_error() == 0
    mask = torch.ones(g.k_cache.numel() // (2 * 64), dtype=torch.bool, device="cuda")
    mask[h.slot_mapping.cuda()] = False
    kf, vf = g.k_cache.view(-1, 2 * 64), g.v_cache.view(-1, 2 * 64)
    assert torch.equal(kf[mask].view(torch.int16), before_k.view(-1, 2 * 64)[mask].view(torch.int16))
    assert torch.equal(vf[mask].view(torch.int16), before_v.view(-1, 2 * 64)[mask].view(torch.int16))


def test_append_empty_and_short_sequences():
    gen = torch.Generator().manual_seed(163)
    lens = torch.randint(0, 60, (300,), generator=gen)
    lens[::17] = 0
    lens[5] = 1
    h = W.make_decode(300, 8, 2, 64, 16, lens.tolist(), seed=164)
    want = oracle_store_and_decode(h)
    got = assert_same_as_separate(to_device(h))
    assert torch.all(got[lens == 0].float() == 0)
    assert_attention_close(got, want, "short/empty")


def test_append_long_sequence_split_across_warps():
    # the last block belongs to a different warp than the first ones
    h = W.make_decode(2, 32, 8, 128, 16, [30001, 12345], seed=165)
    want = oracle_store_and_decode(h)
    got = assert_same_as_separate(to_device(h), max_context_len=30001)
    assert_attention_close(got, want, "split segments")


def test_append_batch_above_persistent_limit():
    gen = torch.Generator().manual_seed(166)
    lens = torch.randint(1, 40, (16500,), generator=gen).tolist()
    lens[7] = 700
    h = W.make_decode(16500, 8, 2, 64, 16, lens, seed=167)
    want = oracle_store_and_decode(h)
    got = assert_same_as_separate(to_device(h), max_context_len=max(lens))
    assert_attention_close(got, want, "large batch")


def test_append_bad_block_id_is_flagged_not_faulted():
    h = W.make_decode(2, 8, 2, 64, 16, [20, 40], seed=168)
    g = to_device(h)
    g.block_tables[1, 2] = 10 ** 6  # the block of position 39
    fused(g)
    assert pa.get_device_error() & pa.PA_DEVERR_BLOCK_RANGE


@pytest.mark.parametrize("name", ["llama3_8b_decode_b64", "llama3_70b_fp8_decode_b256"])
def test_append_full_size_workload(name):
    g = W.make_workload(name, device="cuda")
    lens = g.meta["lens"]
    h = host_copy(g)  # before the GPU appends the new tokens
    got = assert_same_as_separate(g, max_context_len=max(lens))
    want = oracle_store_and_decode(h)
    assert_attention_close(got, want, name)


def test_back_to_back_calls_see_lengths_and_tables_rewritten_in_between():
    # Decode launches let the next one start early and read context_lens and
    # block_tables before waiting. Rewriting both on the device (ordinary
    # kernels) between two calls, with no host synchronisation, must still be
    # seen by the second call.
    lens = [40, 700, 1500, 33]
    h = W.make_decode(len(lens), 32, 8, 128, 16, lens, seed=170)
    g = to_device(h)
    pa.decode_append(g.q, g.k_new, g.v_new, g.k_cache, g.v_cache, g.block_tables,
                     g.context_lens, g.scale)
    g.context_lens[1:2].fill_(300)  # shorten one sequence
    n2 = (lens[2] + 15) // 16
    g.block_tables[2, :n2] = g.block_tables[2, :n2].flip(0)  # reorder another's blocks
    out = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    # the oracle over the same (appended) cache with the rewritten inputs
    want = oracle.decode(W.bf16_bits(g.q.cpu()), W.bf16_bits(g.k_cache.cpu()),
                         W.bf16_bits(g.v_cache.cpu()), g.block_tables.cpu().numpy(),
                         g.context_lens.cpu().numpy(), g.scale)
    assert int(g.context_lens[1]) == 300
    assert_attention_close(out, want, "rewritten lengths/tables")
