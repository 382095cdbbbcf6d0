"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against what the source pages fix or what the
mathematics fixes (closed forms, invariants, a textbook routine in an
independent library, brute force on tiny inputs). No GPU is involved.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(t):
    return W.bf16_bits(t)


def _f64(t):
    return t.detach().cpu().to(torch.float64)


def _dense_kv(inp, b, L):
    """Dense (L, Hkv, D) K and V of sequence b, gathered block by block from the
    pool: logical block j of the sequence is physical block block_tables[b, j]."""
    bs = inp.k_cache.shape[1]
    ks, vs = [], []
    for j in range(-(-L // bs)):
        phys = int(inp.block_tables[b, j])
        ks.append(inp.k_cache[phys])
        vs.append(inp.v_cache[phys])
    k = torch.cat(ks)[:L] if ks else inp.k_cache[0, :0]
    v = torch.cat(vs)[:L] if vs else inp.v_cache[0, :0]
    return _f64(k), _f64(v)


def _store_new(inp):
    """Append the new token via the oracle's store (positions L-1)."""
    kc = _bits(inp.k_cache).copy()
    vc = _bits(inp.v_cache).copy()
    oracle.store_kv(_bits(inp.k_new), _bits(inp.v_new), inp.slot_mapping.numpy(), kc, vc)
    return kc, vc


def _with_new(inp):
    """Same inputs with the new token written by plain tensor indexing."""
    kc = inp.k_cache.clone()
    vc = inp.v_cache.clone()
    hkv, d = kc.shape[2], kc.shape[3]
    for t, s in enumerate(inp.slot_mapping.tolist()):
        if s >= 0:
            kc.view(-1, hkv, d)[s] = inp.k_new[t]
            vc.view(-1, hkv, d)[s] = inp.v_new[t]
    out = W.DecodeInputs(**{**inp.__dict__, "k_cache": kc, "v_cache": vc})
    return out


def _oracle_decode(inp, **kw):
    kc, vc = _store_new(inp)
    return oracle.decode(_bits(inp.q), kc, vc, inp.block_tables.numpy(),
                         inp.context_lens.numpy(), inp.scale, **kw)


# ---------------------------------------------------------------- the mask
def test_mask_matches_printed_2x5_example():
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "bottom_right_mask_2x5.txt"))
            if ln.strip() and not ln.startswith("#")]
    want = np.array([[int(x) for x in r] for r in rows], np.uint8)
    assert want.shape == (2, 5)
    np.testing.assert_array_equal(oracle.causal_mask(2, 5), want)


def test_mask_square_case_is_lower_triangular():
    # cached_len = 0: ordinary causal mask
    np.testing.assert_array_equal(oracle.causal_mask(6, 6), np.tril(np.ones((6, 6), np.uint8)))


def test_mask_matches_tril_with_offset():
    for ql, kl in [(1, 1), (1, 9), (3, 7), (5, 5), (4, 20)]:
        want = torch.ones(ql, kl).tril(diagonal=kl - ql).to(torch.uint8).numpy()
        np.testing.assert_array_equal(oracle.causal_mask(ql, kl), want)


def test_mask_rejects_more_queries_than_keys():
    with pytest.raises(oracle.OracleError):
        oracle.causal_mask(3, 2)


# ---------------------------------------------------------------- decode
@pytest.mark.parametrize("dims", [(3, 4, 2, 16, 4), (2, 8, 8, 8, 16), (4, 6, 1, 32, 8)])
def test_decode_equals_dense_softmax_attention(dims):
    B, H, Hkv, D, bs = dims
    lens = [1, 7, 13, 40][:B]
    inp = _with_new(W.make_decode(B, H, Hkv, D, bs, lens, seed=11))
    got = oracle.decode(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache),
                        inp.block_tables.numpy(), inp.context_lens.numpy(), inp.scale)
    G = H // Hkv
    for b, L in enumerate(lens):
        k, v = _dense_kv(inp, b, L)
        k = k.repeat_interleave(G, dim=1)  # (L, H, D): head h uses kv head h // G
        v = v.repeat_interleave(G, dim=1)
        q = _f64(inp.q[b])  # (H, D)
        s = torch.einsum("hd,lhd->hl", q, k) * inp.scale
        p = torch.softmax(s, dim=-1)
        o = torch.einsum("hl,lhd->hd", p, v)
        np.testing.assert_allclose(got[b], o.numpy(), rtol=0, atol=1e-12)


def test_store_then_decode_uses_the_new_token():
    inp = W.make_decode(3, 4, 2, 16, 4, [5, 8, 9], seed=5)
    a = _oracle_decode(inp)
    ref = _with_new(inp)
    b = oracle.decode(_bits(ref.q), _bits(ref.k_cache), _bits(ref.v_cache),
                      ref.block_tables.numpy(), ref.context_lens.numpy(), ref.scale)
    np.testing.assert_array_equal(a, b)


def test_context_len_one_returns_v_exactly():
    inp = _with_new(W.make_decode(2, 4, 2, 32, 16, [1, 1], seed=3))
    got = oracle.decode(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache),
                        inp.block_tables.numpy(), inp.context_lens.numpy(), inp.scale)
    for b in range(2):
        v = _f64(inp.v_new[b]).repeat_interleave(2, dim=0)
        np.testing.assert_array_equal(got[b], v.numpy())


def test_identical_keys_give_mean_of_v():
    inp = _with_new(W.make_decode(2, 4, 2, 16, 4, [9, 23], seed=4))
    kc = inp.k_cache.clone()
    kc[:] = kc[0, 0]  # every key row identical
    got = oracle.decode(_bits(inp.q), _bits(kc), _bits(inp.v_cache), inp.block_tables.numpy(),
                        inp.context_lens.numpy(), inp.scale)
    for b, L in enumerate([9, 23]):
        _, v = _dense_kv(inp, b, L)
        mean = v.mean(dim=0).repeat_interleave(2, dim=0)
        np.testing.assert_allclose(got[b], mean.numpy(), rtol=0, atol=1e-12)


def test_gqa_equals_mha_with_repeated_kv_heads():
    B, H, Hkv, D, bs = 3, 8, 2, 16, 4
    lens = [3, 10, 17]
    inp = _with_new(W.make_decode(B, H, Hkv, D, bs, lens, seed=8))
    gqa = oracle.decode(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache),
                        inp.block_tables.numpy(), inp.context_lens.numpy(), inp.scale)
    G = H // Hkv
    k_mha = inp.k_cache.repeat_interleave(G, dim=2)
    v_mha = inp.v_cache.repeat_interleave(G, dim=2)
    mha = oracle.decode(_bits(inp.q), _bits(k_mha), _bits(v_mha), inp.block_tables.numpy(),
                        inp.context_lens.numpy(), inp.scale)
    np.testing.assert_array_equal(gqa, mha)
    # and the map is h // G, not h % Hkv: swapping kv heads changes the answer
    k_sw = inp.k_cache.flip(2)
    v_sw = inp.v_cache.flip(2)
    other = oracle.decode(_bits(inp.q), _bits(k_sw), _bits(v_sw), inp.block_tables.numpy(),
                          inp.context_lens.numpy(), inp.scale)
    assert np.abs(other - gqa).max() > 1e-3


def test_invariant_under_physical_block_permutation():
    inp = _with_new(W.make_decode(4, 4, 2, 16, 4, [2, 9, 16, 31], seed=9, num_blocks=40))
    base = oracle.decode(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache),
                         inp.block_tables.numpy(), inp.context_lens.numpy(), inp.scale)
    perm = torch.randperm(40, generator=torch.Generator().manual_seed(1))
    inv = torch.argsort(perm)  # new position of old block i is inv[i]
    kc = inp.k_cache[perm]
    vc = inp.v_cache[perm]
    bt = inp.block_tables.clone()
    m = bt >= 0
    bt[m] = inv[bt[m].long()].to(torch.int32)
    got = oracle.decode(_bits(inp.q), _bits(kc), _bits(vc), bt.numpy(), inp.context_lens.numpy(),
                        inp.scale)
    np.testing.assert_array_equal(got, base)


def test_context_len_zero_gives_zero_row():
    inp = _with_new(W.make_decode(2, 4, 2, 16, 4, [0, 5], seed=2))
    got = oracle.decode(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache),
                        inp.block_tables.numpy(), inp.context_lens.numpy(), inp.scale)
    assert np.all(got[0] == 0.0)
    assert np.abs(got[1]).max() > 0


def test_zero_padding_to_max_len_distorts_result():
    # The decode page warns that zero-padded keys steal softmax weight; the
    # oracle must not do that: with lengths {1, 100} the padded version differs.
    inp = _with_new(W.make_decode(2, 4, 2, 16, 4, [1, 100], seed=12))
    got = oracle.decode(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache),
                        inp.block_tables.numpy(), inp.context_lens.numpy(), inp.scale)
    k, v = _dense_kv(inp, 0, 1)
    kp = torch.zeros(100, *k.shape[1:], dtype=torch.float64)
    vp = torch.zeros_like(kp)
    kp[:1], vp[:1] = k, v
    q = _f64(inp.q[0])
    s = torch.einsum("hd,lhd->hl", q, kp.repeat_interleave(2, dim=1)) * inp.scale
    padded = torch.einsum("hl,lhd->hd", torch.softmax(s, -1), vp.repeat_interleave(2, dim=1))
    assert np.abs(padded.numpy() - got[0]).max() > 1e-2
    np.testing.assert_array_equal(got[0], v[0].repeat_interleave(2, dim=0).numpy())


@pytest.mark.parametrize("split", [1, 3, 16, 17, 64, 1000])
def test_split_merge_equals_unsplit(split):
    inp = _with_new(W.make_decode(3, 8, 2, 16, 4, [1, 50, 123], seed=21))
    a = oracle.decode(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache),
                      inp.block_tables.numpy(), inp.context_lens.numpy(), inp.scale)
    b = oracle.decode_split(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache),
                            inp.block_tables.numpy(), inp.context_lens.numpy(), inp.scale, split)
    np.testing.assert_allclose(b, a, rtol=0, atol=1e-12)


def test_decode_rejects_block_out_of_pool():
    inp = _with_new(W.make_decode(1, 2, 1, 8, 4, [6], seed=1, num_blocks=4))
    bt = inp.block_tables.clone()
    bt[0, 1] = 4  # pool has blocks 0..3
    with pytest.raises(oracle.OracleError):
        oracle.decode(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache), bt.numpy(),
                      inp.context_lens.numpy(), inp.scale)


# ---------------------------------------------------------------- store_kv
def test_store_kv_is_indexed_assignment_and_leaves_other_slots():
    inp = W.make_decode(5, 4, 2, 16, 4, [3, 4, 5, 12, 1], seed=6, num_blocks=12)
    sm = inp.slot_mapping.clone()
    sm[2] = -1  # a padding token writes nothing
    kc = torch.full_like(inp.k_cache, 7.0)  # sentinel bytes everywhere
    vc = torch.full_like(inp.v_cache, -3.0)
    kb, vb = _bits(kc).copy(), _bits(vc).copy()
    oracle.store_kv(_bits(inp.k_new), _bits(inp.v_new), sm.numpy(), kb, vb)
    hkv, d = kc.shape[2], kc.shape[3]
    for t, s in enumerate(sm.tolist()):
        if s >= 0:
            kc.view(-1, hkv, d)[s] = inp.k_new[t]
            vc.view(-1, hkv, d)[s] = inp.v_new[t]
    np.testing.assert_array_equal(kb, _bits(kc))
    np.testing.assert_array_equal(vb, _bits(vc))
    # block/offset arithmetic of the append: logical block p // bs, offset p % bs
    L = 12
    p = L - 1
    assert int(inp.slot_mapping[3]) == int(inp.block_tables[3, p // 4]) * 4 + p % 4


def test_store_kv_rejects_slot_beyond_pool():
    inp = W.make_decode(1, 2, 1, 8, 4, [3], seed=1, num_blocks=2)
    kc, vc = _bits(inp.k_cache).copy(), _bits(inp.v_cache).copy()
    with pytest.raises(oracle.OracleError):
        oracle.store_kv(_bits(inp.k_new), _bits(inp.v_new), np.array([8], np.int64), kc, vc)


# ---------------------------------------------------------------- FP8
def test_e4m3_codec_matches_torch_for_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_to_double(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2
    np.testing.assert_array_equal(got[~nan], want[~nan])
    # a few values written out from the format definition
    assert got[0x38] == 1.0 and got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9
    assert got[0xB8] == -1.0 and got[0x08] == 2.0 ** -6


def test_fp8_decode_equals_dense_attention_on_dequantised_values():
    B, H, Hkv, D, bs = 3, 8, 2, 32, 8
    lens = [1, 9, 30]
    inp = W.make_decode(B, H, Hkv, D, bs, lens, seed=14, kv_dtype="fp8")
    kc, vc = W.u8(inp.k_cache).copy(), W.u8(inp.v_cache).copy()
    ksc, vsc = inp.k_scale.numpy().copy(), inp.v_scale.numpy().copy()
    oracle.store_kv(W.u8(inp.k_new), W.u8(inp.v_new), inp.slot_mapping.numpy(), kc, vc,
                    inp.k_scale_new.numpy(), inp.v_scale_new.numpy(), ksc, vsc)
    got = oracle.decode(_bits(inp.q), kc, vc, inp.block_tables.numpy(), inp.context_lens.numpy(),
                        inp.scale, k_scale=ksc, v_scale=vsc)
    # scales are stored (NB, Hkv, bs); bring them to the cache's (NB, bs, Hkv)
    kd = torch.from_numpy(kc).view(torch.float8_e4m3fn).to(torch.float64) * \
        torch.from_numpy(ksc).double().permute(0, 2, 1)[..., None]
    vd = torch.from_numpy(vc).view(torch.float8_e4m3fn).to(torch.float64) * \
        torch.from_numpy(vsc).double().permute(0, 2, 1)[..., None]
    dense = W.DecodeInputs(**{**inp.__dict__, "k_cache": kd, "v_cache": vd})
    G = H // Hkv
    for b, L in enumerate(lens):
        k, v = _dense_kv(dense, b, L)
        k, v = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
        s = torch.einsum("hd,lhd->hl", _f64(inp.q[b]), k) * inp.scale
        o = torch.einsum("hl,lhd->hd", torch.softmax(s, -1), v)
        np.testing.assert_allclose(got[b], o.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- window / sinks
# "Decode Phase" glossary, long-context bullets: a sliding window attends to
# the most recent W tokens; attention sinks (StreamingLLM) keep the initial
# tokens as well. Visible keys of a sequence of L tokens: p < S or p >= L - W.
def _visible(L, window, sinks):
    if window <= 0:
        return list(range(L))
    return [p for p in range(L) if p < sinks or p >= L - window]


@pytest.mark.parametrize("window,sinks", [(1, 0), (5, 0), (8, 2), (13, 4), (40, 3), (3, 40),
                                          (6, 6)])
def test_window_decode_equals_dense_attention_over_visible_keys(window, sinks):
    B, H, Hkv, D, bs = 4, 6, 2, 16, 4
    lens = [1, 9, 17, 38]
    inp = _with_new(W.make_decode(B, H, Hkv, D, bs, lens, seed=21))
    got = oracle.decode(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache),
                        inp.block_tables.numpy(), inp.context_lens.numpy(), inp.scale,
                        window=window, sinks=sinks)
    G = H // Hkv
    for b, L in enumerate(lens):
        k, v = _dense_kv(inp, b, L)
        idx = torch.tensor(_visible(L, window, sinks), dtype=torch.long)
        k = k[idx].repeat_interleave(G, dim=1)
        v = v[idx].repeat_interleave(G, dim=1)
        s = torch.einsum("hd,lhd->hl", _f64(inp.q[b]), k) * inp.scale
        o = torch.einsum("hl,lhd->hd", torch.softmax(s, -1), v)
        np.testing.assert_allclose(got[b], o.numpy(), rtol=0, atol=1e-12)


def test_window_of_one_returns_newest_v_exactly():
    inp = _with_new(W.make_decode(3, 4, 2, 32, 8, [1, 20, 70], seed=22))
    got = oracle.decode(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache),
                        inp.block_tables.numpy(), inp.context_lens.numpy(), inp.scale,
                        window=1)
    for b in range(3):
        np.testing.assert_array_equal(got[b], _f64(inp.v_new[b]).repeat_interleave(2, 0).numpy())


def test_window_covering_everything_equals_full_decode():
    inp = _with_new(W.make_decode(3, 8, 2, 16, 4, [5, 30, 31], seed=23))
    args = (_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache), inp.block_tables.numpy(),
            inp.context_lens.numpy(), inp.scale)
    full = oracle.decode(*args)
    np.testing.assert_array_equal(oracle.decode(*args, window=31), full)
    np.testing.assert_array_equal(oracle.decode(*args, window=20, sinks=11), full)
    np.testing.assert_array_equal(oracle.decode(*args, window=0, sinks=3), full)


def test_window_equals_full_decode_of_the_visible_tokens_repacked():
    # the visible keys copied into a fresh, compact cache form a sequence of
    # their own; full decode over it must give the windowed result
    B, H, Hkv, D, bs = 3, 4, 2, 16, 4
    lens = [12, 29, 40]
    window, sinks = 7, 3
    inp = _with_new(W.make_decode(B, H, Hkv, D, bs, lens, seed=24))
    want = oracle.decode(_bits(inp.q), _bits(inp.k_cache), _bits(inp.v_cache),
                         inp.block_tables.numpy(), inp.context_lens.numpy(), inp.scale,
                         window=window, sinks=sinks)
    for b, L in enumerate(lens):
        vis = _visible(L, window, sinks)
        n = len(vis)
        nb = -(-n // bs)
        kc = torch.zeros((nb, bs, Hkv, D), dtype=torch.bfloat16)
        vc = torch.zeros_like(kc)
        for i, p in enumerate(vis):
            phys = int(inp.block_tables[b, p // bs])
            kc[i // bs, i % bs] = inp.k_cache[phys, p % bs]
            vc[i // bs, i % bs] = inp.v_cache[phys, p % bs]
        bt = np.arange(nb, dtype=np.int32)[None]
        got = oracle.decode(_bits(inp.q[b:b + 1]), _bits(kc), _bits(vc), bt,
                            np.array([n], np.int32), inp.scale)
        np.testing.assert_allclose(got[0], want[b], rtol=0, atol=1e-13)


# ---------------------------------------------------------------- INT8 KV
def test_int8_quantiser_round_trip_bound():
    g = torch.Generator().manual_seed(25)
    codes, scales = W._randn_int8((50, 64), g, "cpu")
    g = torch.Generator().manual_seed(25)
    x = torch.randn((50, 64), generator=g, dtype=torch.float32).double()
    c = codes.double()
    assert c.abs().max() <= 127
    # the row maximum lands on +-127 exactly; every value within half a step
    np.testing.assert_array_equal(c.abs().amax(1).numpy(), np.full(50, 127.0))
    err = (c * scales.double()[:, None] - x).abs()
    assert bool((err <= scales.double()[:, None] * 0.5 * (1 + 1e-6)).all())


def test_int8_decode_equals_dense_attention_on_dequantised_values():
    B, H, Hkv, D, bs = 3, 8, 2, 32, 8
    lens = [1, 9, 30]
    inp = W.make_decode(B, H, Hkv, D, bs, lens, seed=26, kv_dtype="int8")
    kc, vc = W.u8(inp.k_cache).copy(), W.u8(inp.v_cache).copy()
    assert kc.dtype == np.int8
    ksc, vsc = inp.k_scale.numpy().copy(), inp.v_scale.numpy().copy()
    oracle.store_kv(W.u8(inp.k_new), W.u8(inp.v_new), inp.slot_mapping.numpy(), kc, vc,
                    inp.k_scale_new.numpy(), inp.v_scale_new.numpy(), ksc, vsc)
    got = oracle.decode(_bits(inp.q), kc, vc, inp.block_tables.numpy(), inp.context_lens.numpy(),
                        inp.scale, k_scale=ksc, v_scale=vsc)
    kd = torch.from_numpy(kc).double() * torch.from_numpy(ksc).double().permute(0, 2, 1)[..., None]
    vd = torch.from_numpy(vc).double() * torch.from_numpy(vsc).double().permute(0, 2, 1)[..., None]
    dense = W.DecodeInputs(**{**inp.__dict__, "k_cache": kd, "v_cache": vd})
    G = H // Hkv
    for b, L in enumerate(lens):
        k, v = _dense_kv(dense, b, L)
        k, v = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
        s = torch.einsum("hd,lhd->hl", _f64(inp.q[b]), k) * inp.scale
        o = torch.einsum("hl,lhd->hd", torch.softmax(s, -1), v)
        np.testing.assert_allclose(got[b], o.numpy(), rtol=0, atol=1e-12)
    # context_len 1: the newest V row, dequantised, exactly
    v1 = W.u8(inp.v_new[0]).astype(np.float64) * inp.v_scale_new[0].double().numpy()[:, None]
    np.testing.assert_array_equal(got[0], np.repeat(v1, G, axis=0))


# ---------------------------------------------------------------- prefill
def _stored_prefill(inp):
    kc, vc = _bits(inp.k_cache).copy(), _bits(inp.v_cache).copy()
    oracle.store_kv(_bits(inp.k_new), _bits(inp.v_new), inp.slot_mapping.numpy(), kc, vc)
    return kc, vc


def test_cu_seqlens_example_rows():
    lines = {ln.split()[0]: [int(x) for x in ln.split()[1:]]
             for ln in open(os.path.join(GOLDEN, "cu_seqlens_example.txt"))
             if ln.strip() and not ln.startswith("#")}
    cu = lines["cu_seqlens_q"]
    inp = W.make_prefill(2, 2, 1, 8, 4, [0, 0], [cu[1] - cu[0], cu[2] - cu[1]], seed=3)
    # make every V of sequence 0 equal 1 and of sequence 1 equal 2
    inp.v_new[:4] = 1.0
    inp.v_new[4:] = 2.0
    kc, vc = _stored_prefill(inp)
    out = oracle.prefill(_bits(inp.q), kc, vc, inp.block_tables.numpy(), np.array(cu, np.int32),
                         inp.cu_seqlens_k.numpy(), inp.scale)
    for r in lines["rows_of_seq0"]:
        np.testing.assert_allclose(out[r], 1.0, rtol=0, atol=1e-12)
    for r in lines["rows_of_seq1"]:
        np.testing.assert_allclose(out[r], 2.0, rtol=0, atol=1e-12)


def test_prefill_without_prefix_equals_causal_sdpa():
    B, H, Hkv, D, bs = 2, 4, 2, 16, 4
    qls = [5, 11]
    inp = W.make_prefill(B, H, Hkv, D, bs, [0, 0], qls, seed=17)
    kc, vc = _stored_prefill(inp)
    out = oracle.prefill(_bits(inp.q), kc, vc, inp.block_tables.numpy(),
                         inp.cu_seqlens_q.numpy(), inp.cu_seqlens_k.numpy(), inp.scale)
    G = H // Hkv
    for b in range(B):
        r0, r1 = int(inp.cu_seqlens_q[b]), int(inp.cu_seqlens_q[b + 1])
        q = _f64(inp.q[r0:r1]).transpose(0, 1)  # (H, n, D)
        k = _f64(inp.k_new[r0:r1]).repeat_interleave(G, dim=1).transpose(0, 1)
        v = _f64(inp.v_new[r0:r1]).repeat_interleave(G, dim=1).transpose(0, 1)
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                             scale=inp.scale)
        np.testing.assert_allclose(out[r0:r1], o.transpose(0, 1).numpy(), rtol=0, atol=1e-12)


def test_prefill_with_prefix_equals_bruteforce_bottom_right_mask():
    B, H, Hkv, D, bs = 3, 4, 1, 16, 4
    cached, qls = [0, 6, 13], [3, 7, 2]
    inp = W.make_prefill(B, H, Hkv, D, bs, cached, qls, seed=19)
    kc, vc = _stored_prefill(inp)
    out = oracle.prefill(_bits(inp.q), kc, vc, inp.block_tables.numpy(),
                         inp.cu_seqlens_q.numpy(), inp.cu_seqlens_k.numpy(), inp.scale)
    kt = torch.from_numpy(kc.view(np.int16)).view(torch.bfloat16)
    vt = torch.from_numpy(vc.view(np.int16)).view(torch.bfloat16)
    stored = W.DecodeInputs(q=inp.q, k_new=None, v_new=None, slot_mapping=None, k_cache=kt,
                            v_cache=vt, block_tables=inp.block_tables, context_lens=None,
                            scale=inp.scale)
    for b in range(B):
        kl = cached[b] + qls[b]
        k, v = _dense_kv(stored, b, kl)
        k, v = k.repeat_interleave(H, dim=1), v.repeat_interleave(H, dim=1)
        r0 = int(inp.cu_seqlens_q[b])
        q = _f64(inp.q[r0:r0 + qls[b]])
        s = torch.einsum("nhd,lhd->hnl", q, k) * inp.scale
        vis = torch.ones(qls[b], kl, dtype=torch.bool).tril(diagonal=kl - qls[b])
        s = s.masked_fill(~vis, float("-inf"))
        o = torch.einsum("hnl,lhd->nhd", torch.softmax(s, -1), v)
        np.testing.assert_allclose(out[r0:r0 + qls[b]], o.numpy(), rtol=0, atol=1e-12)


def test_prefill_single_query_equals_decode():
    # q_len = 1 with cached_len = L - 1 sees all L keys: the decode problem.
    lens = [1, 6, 19]
    dec = W.make_decode(3, 4, 2, 16, 4, lens, seed=23)
    kc, vc = _store_new(dec)
    d_out = oracle.decode(_bits(dec.q), kc, vc, dec.block_tables.numpy(),
                          dec.context_lens.numpy(), dec.scale)
    cu_q = np.arange(4, dtype=np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    p_out = oracle.prefill(_bits(dec.q), kc, vc, dec.block_tables.numpy(), cu_q, cu_k, dec.scale)
    np.testing.assert_array_equal(p_out, d_out)


def test_prefill_rejects_more_queries_than_keys():
    inp = W.make_prefill(1, 2, 1, 8, 4, [0], [4], seed=2)
    kc, vc = _stored_prefill(inp)
    with pytest.raises(oracle.OracleError):
        oracle.prefill(_bits(inp.q), kc, vc, inp.block_tables.numpy(),
                       np.array([0, 4], np.int32), np.array([0, 3], np.int32), inp.scale)


# ---------------------------------------------------------------- workloads
def test_workload_shapes_and_sinks():
    w = W.make_decode(2, 4, 2, 16, 4, [40, 64], seed=30, sinks=4)
    assert [len(s) for s in w.meta["sink_positions"]] == [4, 4]
    ref = W.make_decode(2, 4, 2, 16, 4, [40, 64], seed=30, sinks=0)
    for b, L in enumerate([40, 64]):
        k, _ = _dense_kv(_with_new(w), b, L)
        k0, _ = _dense_kv(_with_new(ref), b, L)
        for p in range(L):
            f = 4.0 if p in w.meta["sink_positions"][b] else 1.0
            assert torch.equal(k[p], k0[p] * f)


def test_tiny_workload_matches_its_description():
    w = W.make_workload("tiny_decode")
    assert w.q.shape == (4, 8, 64) and w.k_cache.shape == (64, 16, 2, 64)
    assert w.context_lens.tolist() == [1, 17, 33, 100]
    used = w.block_tables[w.block_tables >= 0]
    assert used.numel() == 1 + 2 + 3 + 7 and len(set(used.tolist())) == used.numel()
    assert math.isclose(w.scale, 1 / 8)
