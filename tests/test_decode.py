"""GPU paged decode (pa_store_kv + pa_decode) against the fp64 oracle.

Tolerance (bf16 output, fp32 accumulation): max-abs <= 1e-2 and relative L2
<= 5e-3 over all outputs of a call. Every case, the full-size workloads in
the bench's launch configuration included, is compared element by element
over every output row.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import assert_attention_close, host_copy, oracle_store_and_decode, to_device

pytestmark = pytest.mark.gpu


def gpu_store_decode(g, max_context_len=0, out=None, workspace=None):
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, g.k_scale_new,
                g.v_scale_new, g.k_scale, g.v_scale)
    out = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                    max_context_len=max_context_len, out=out, workspace=workspace,
                    k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    return out


def run_case(h, max_context_len=0):
    want = oracle_store_and_decode(h)
    g = to_device(h)
    got = gpu_store_decode(g, max_context_len)
    assert pa.get_device_error() == 0
    return got, want


def test_tiny_workload_full_parity():
    h = W.make_workload("tiny_decode")
    got, want = run_case(h)
    assert_attention_close(got, want, "tiny_decode")


CASES = [
    # (H, Hkv, D, bs, kv, lens)
    (8, 2, 64, 16, "bf16", [1, 17, 33, 100, 16, 15]),
    (32, 8, 128, 16, "bf16", [1, 15, 16, 17, 255, 256, 257, 3000, 700, 4096]),
    (32, 8, 128, 32, "bf16", [1, 31, 32, 33, 63, 64, 65, 2049, 5000]),
    (4, 4, 64, 32, "bf16", [2, 40, 1000, 77]),        # MHA, group 1
    (8, 1, 128, 16, "bf16", [9, 300, 1025]),          # MQA, group 8
    (6, 2, 128, 16, "bf16", [5, 513, 129]),           # group 3
    (64, 8, 128, 32, "fp8", [1, 31, 32, 33, 1000, 5000]),
    (16, 2, 128, 16, "fp8", [1, 16, 17, 300, 2500]),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"H{c[0]}kv{c[1]}D{c[2]}bs{c[3]}{c[4]}")
def test_decode_matches_oracle(case):
    H, Hkv, D, bs, kv, lens = case
    h = W.make_decode(len(lens), H, Hkv, D, bs, lens, seed=50 + H + D + bs, kv_dtype=kv)
    got, want = run_case(h)
    assert_attention_close(got, want, str(case))


def test_decode_with_context_len_hint():
    lens = [100, 3000, 17, 2048]
    h = W.make_decode(4, 32, 8, 128, 16, lens, seed=61)
    got, want = run_case(h, max_context_len=max(lens))
    assert_attention_close(got, want, "hint")


def test_context_len_zero_row_is_zero():
    h = W.make_decode(3, 8, 2, 64, 16, [0, 5, 40], seed=62)
    got, want = run_case(h)
    assert torch.all(got[0] == 0)
    assert_attention_close(got, want, "len0")


def test_context_len_one_returns_stored_v_bit_exactly():
    for kv in ("bf16",):
        h = W.make_decode(4, 32, 8, 128, 16, [1, 1, 1, 1], seed=63, kv_dtype=kv)
        g = to_device(h)
        got = gpu_store_decode(g)
        want = g.v_new.repeat_interleave(4, dim=1)  # (B, H, D): head h reads kv head h // 4
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_identical_keys_give_mean_of_v():
    h = W.make_decode(2, 8, 2, 128, 16, [37, 300], seed=64)
    h.k_cache[:] = h.k_new[0, 0]
    h.k_new[:] = h.k_new[0, 0]
    got, want = run_case(h)
    assert_attention_close(got, want, "identical keys")


def test_repeat_calls_are_deterministic():
    h = W.make_decode(6, 32, 8, 128, 16, [100, 4000, 600, 1, 2222, 3333], seed=65)
    g = to_device(h)
    a = gpu_store_decode(g).clone()
    b = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_workspace_contents_on_entry_are_ignored():
    # zeros, all-ones bytes, random bytes and a workspace an earlier call left
    # behind: the same output, equal to the oracle's (segments split across warps)
    lens = [3000, 17, 4096, 1, 1500, 2200, 700, 64]
    h = W.make_decode(len(lens), 32, 8, 128, 16, lens, seed=73)
    want = oracle_store_and_decode(h)
    g = to_device(h)
    n = pa.decode_workspace_size(g.k_cache, len(lens), 32, g.block_tables.shape[1])
    assert n > 0
    first = gpu_store_decode(g).clone()
    assert_attention_close(first, want, "first call")
    gen = torch.Generator().manual_seed(74)
    left_behind = torch.empty(n, dtype=torch.uint8, device="cuda")
    pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
              workspace=left_behind)
    fills = [torch.zeros(n, dtype=torch.uint8), torch.full((n,), 255, dtype=torch.uint8),
             torch.randint(0, 256, (n,), generator=gen, dtype=torch.uint8)]
    for ws in [f.cuda() for f in fills] + [left_behind]:
        got = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                        workspace=ws)
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        assert torch.equal(got.view(torch.int16), first.view(torch.int16))


def test_workspace_too_small_is_rejected():
    h = to_device(W.make_decode(2, 32, 8, 128, 16, [4000, 4000], seed=66))
    need = pa.decode_workspace_size(h.k_cache, 2, 32, h.block_tables.shape[1])
    assert need > 0
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.lib()  # loaded
        import ctypes
        cache = pa.make_cache(h.k_cache, h.v_cache)
        rc = pa.lib().pa_decode(ctypes.c_void_p(h.q.data_ptr()), ctypes.byref(cache),
                                ctypes.c_void_p(h.block_tables.data_ptr()), h.block_tables.shape[1],
                                ctypes.c_void_p(h.context_lens.data_ptr()), 0, 2, 32, h.scale,
                                ctypes.c_void_p(h.q.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                ws.numel(), None)
        pa._check(rc, "pa_decode")
    assert e.value.code == 6


def test_block_table_entry_outside_pool_is_flagged_not_faulted():
    h = W.make_decode(2, 8, 2, 64, 16, [40, 20], seed=67, num_blocks=8)
    g = to_device(h)
    g.block_tables[0, 1] = 8  # pool has blocks 0..7
    pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale)
    assert pa.get_device_error() & pa.PA_DEVERR_BLOCK_RANGE
    assert pa.get_device_error() == 0


def _full_size(name):
    g = W.make_workload(name, device="cuda")
    lens = g.meta["lens"]
    h = host_copy(g)  # before the GPU appends the new tokens
    got = gpu_store_decode(g, max_context_len=max(lens))
    assert pa.get_device_error() == 0
    want = oracle_store_and_decode(h)
    return got, want


@pytest.mark.parametrize("name", ["llama3_8b_decode_b64", "long_context_decode_b8",
                                  "llama3_70b_fp8_decode_b256", "llama3_8b_short_decode_b2304",
                                  "llama3_8b_short_decode_b9216",
                                  "llama3_8b_short_decode_b17408"])
def test_full_size_workload_every_sequence(name):
    # the bench's launch configuration; every output row against the oracle
    got, want = _full_size(name)
    assert_attention_close(got, want, name)


def test_many_short_and_empty_sequences():
    # many segments per CTA, zero-length sequences in between, tiny pieces
    gen = torch.Generator().manual_seed(90)
    lens = torch.randint(0, 60, (300,), generator=gen)
    lens[::17] = 0
    lens[5] = 1
    h = W.make_decode(300, 8, 2, 64, 16, lens.tolist(), seed=91)
    got, want = run_case(h)
    assert torch.all(got[lens == 0].float() == 0)
    assert_attention_close(got, want, "short/empty")


@pytest.mark.parametrize("kv,H,bs", [("bf16", 32, 16), ("fp8", 64, 32), ("int8", 64, 32)])
def test_empty_sequences_between_long_ones(kv, H, bs):
    # segments long enough for the split to count a cost per segment end,
    # with empty sequences (work units but no blocks) between them, in runs
    lens = [0, 0, 0, 700, 0, 4100, 0, 0, 0, 0, 33, 2500, 0, 1, 0, 0, 9000, 0]
    h = W.make_decode(len(lens), H, 8, 128, bs, lens, seed=88, kv_dtype=kv)
    got, want = run_case(h)
    assert torch.all(got[torch.tensor(lens) == 0].float() == 0)
    assert_attention_close(got, want, f"empty between long ({kv})")


def test_one_long_sequence_spread_over_all_ctas():
    h = W.make_decode(1, 32, 8, 128, 16, [70001], seed=92)
    got, want = run_case(h, max_context_len=70001)
    assert_attention_close(got, want, "one long sequence")


@pytest.mark.parametrize("H,Hkv,bs,kv,L", [
    (32, 8, 16, "bf16", 100000),
    (8, 1, 16, "bf16", 100003),   # one segment split into hundreds of parts
    (8, 8, 32, "bf16", 65537),    # group 1
    (6, 2, 16, "bf16", 50001),    # group 3
    (64, 8, 32, "fp8", 99999),
])
def test_one_long_sequence_merges_in_groups(H, Hkv, bs, kv, L):
    # far more than 16 warps per (sequence, kv head): partials merge per
    # group of 16 and then across groups
    h = W.make_decode(1, H, Hkv, 128, bs, [L], seed=95 + H + bs, kv_dtype=kv)
    got, want = run_case(h, max_context_len=L)
    assert_attention_close(got, want, f"one sequence of {L}")


@pytest.mark.parametrize("H,Hkv,kv,L", [
    (32, 8, "bf16", 2048),   # 128 blocks per segment: 32 parts, one merge
    (32, 8, "bf16", 2112),   # 33 parts: groups of 16, 16 and a 1-part tail
    (32, 8, "bf16", 2176),   # 34 parts: 16, 16, 2
    (32, 8, "bf16", 2065),   # 130 blocks, the last one partly filled
    (8, 8, "bf16", 2112),    # group 1
    (64, 8, "fp8", 2112),
])
def test_merge_group_boundaries(H, Hkv, kv, L):
    # one sequence of fewer than 4 * (persistent CTAs) blocks over all kv
    # heads: one warp per 4 blocks, so a segment of n blocks has n / 4 parts
    bs = 32 if kv == "fp8" else 16
    h = W.make_decode(1, H, Hkv, 128, bs, [L * bs // 16], seed=97 + L + H, kv_dtype=kv)
    got, want = run_case(h, max_context_len=L * bs // 16)
    assert_attention_close(got, want, f"one sequence of {L * bs // 16} ({kv})")


def test_batch_at_persistent_limit():
    # 16384 sequences: the largest batch of the persistent kernel (its prefix
    # sums fill 64 KB of shared memory, 1 CTA per SM)
    gen = torch.Generator().manual_seed(95)
    lens = torch.randint(0, 40, (16384,), generator=gen).tolist()
    lens[4000] = 3000  # one segment split over many warps
    h = W.make_decode(16384, 8, 2, 64, 16, lens, seed=96)
    got, want = run_case(h, max_context_len=max(lens))
    assert torch.all(got[torch.tensor(lens) == 0].float() == 0)
    assert_attention_close(got, want, "batch 16384")


def test_batch_above_persistent_limit_uses_grid_split():
    gen = torch.Generator().manual_seed(93)
    lens = torch.randint(1, 40, (16500,), generator=gen).tolist()
    lens[7] = 700  # one sequence long enough to need several splits
    h = W.make_decode(16500, 8, 2, 64, 16, lens, seed=94)
    got, want = run_case(h, max_context_len=max(lens))
    assert_attention_close(got, want, "large batch")
