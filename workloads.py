"""Seeded synthetic inputs for paged-KV-cache attention.

This module only builds inputs: shapes, random values, block assignments and
slot numbers. It contains none of the attention arithmetic, so both the CUDA
library's tests/bench and the CPU oracle can consume what it produces.

Layouts (the library's boundary):
  * k_cache, v_cache: (num_blocks, block_size, num_kv_heads, head_dim),
    bf16 or FP8-E4M3 (stored as uint8 codes); FP8 adds fp32 scales, one per
    (slot, kv head), laid out (num_blocks, num_kv_heads, block_size).
  * block_tables: (batch, max_blocks) int32, unused entries -1.
  * slot = physical_block * block_size + offset (int64), one per new token.

Recipe, common to all workloads: values are drawn from torch's Philox/MT
generators seeded per workload; bulk tensors are drawn in fp32 N(0, 1) and
rounded to bf16 (round-to-nearest-even); physical blocks are a random
permutation of the pool, handed out to sequences in order, so consecutive
logical blocks of a sequence are scattered over the pool.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# The five workloads, by what they are.
WORKLOADS = {
    # Tiny paged decode: 1 layer, B=4, H=8, Hkv=2, D=64, bs=16, pool of 64 blocks.
    "tiny_decode": dict(kind="decode", seed=0, batch=4, num_heads=8, num_kv_heads=2, head_dim=64,
                        block_size=16, context_lens=[1, 17, 33, 100], num_blocks=64,
                        scale=1.0 / 8.0, kv_dtype="bf16"),
    # Llama-3-8B-shaped decode: 32 q heads / 8 kv heads, D=128, bs=16, batch 64,
    # context_len uniform in [512, 4096], pool of 20k blocks.
    "llama3_8b_decode_b64": dict(kind="decode", seed=1, batch=64, num_heads=32, num_kv_heads=8,
                                 head_dim=128, block_size=16, lens=("uniform", 512, 4096),
                                 num_blocks=20000, scale=1.0 / math.sqrt(128), kv_dtype="bf16"),
    # Long-context split-K decode: batch 8, context_len uniform in [32768, 131072],
    # 4 random 'sink' key positions per sequence with 4x the key norm.
    "long_context_decode_b8": dict(kind="decode", seed=2, batch=8, num_heads=32, num_kv_heads=8,
                                   head_dim=128, block_size=16, lens=("uniform", 32768, 131072),
                                   pool_factor=1.1, sinks=4, scale=1.0 / math.sqrt(128),
                                   kv_dtype="bf16"),
    # Llama-3-70B-shaped continuous-batch decode with FP8-E4M3 KV: 64 q heads /
    # 8 kv heads, D=128, bs=32, batch 256, context_len lognormal(median 1024,
    # sigma 1) clipped to [1, 16384].
    "llama3_70b_fp8_decode_b256": dict(kind="decode", seed=3, batch=256, num_heads=64,
                                       num_kv_heads=8, head_dim=128, block_size=32,
                                       lens=("lognormal", 1024.0, 1.0, 1, 16384), pool_factor=1.1,
                                       scale=1.0 / math.sqrt(128), kv_dtype="fp8"),
    # The same continuous batch with an INT8 KV cache (symmetric codes, one
    # fp32 scale per (token, head)): the glossary's other KV quantisation.
    "llama3_70b_int8_decode_b256": dict(kind="decode", seed=3, batch=256, num_heads=64,
                                        num_kv_heads=8, head_dim=128, block_size=32,
                                        lens=("lognormal", 1024.0, 1.0, 1, 16384),
                                        pool_factor=1.1, scale=1.0 / math.sqrt(128),
                                        kv_dtype="int8"),
    # A large continuous batch: 2304 mostly short sequences, Llama-3-8B heads,
    # context_len lognormal (median 96, sigma 1) clipped to [8, 1536]. The
    # persistent decode with 9 KB of per-sequence prefix sums in each CTA's
    # shared memory.
    "llama3_8b_short_decode_b2304": dict(kind="decode", seed=5, batch=2304, num_heads=32,
                                         num_kv_heads=8, head_dim=128, block_size=16,
                                         lens=("lognormal", 96.0, 1.0, 8, 1536),
                                         pool_factor=1.1, scale=1.0 / math.sqrt(128),
                                         kv_dtype="bf16"),
    # 9216 sequences, Llama-3-8B heads, short contexts (lognormal, median 64,
    # sigma 0.5, clipped to [8, 512]): the persistent decode at 2 CTAs per SM.
    "llama3_8b_short_decode_b9216": dict(kind="decode", seed=6, batch=9216, num_heads=32,
                                         num_kv_heads=8, head_dim=128, block_size=16,
                                         lens=("lognormal", 64.0, 0.5, 8, 512),
                                         pool_factor=1.1, scale=1.0 / math.sqrt(128),
                                         kv_dtype="bf16"),
    # More sequences than the persistent decode's per-sequence prefix sums
    # hold (16384): the grid-split decode. Llama-3-8B heads, short contexts
    # (lognormal, median 48, sigma 0.5, clipped to [8, 384]).
    "llama3_8b_short_decode_b17408": dict(kind="decode", seed=8, batch=17408, num_heads=32,
                                          num_kv_heads=8, head_dim=128, block_size=16,
                                          lens=("lognormal", 48.0, 0.5, 8, 384),
                                          pool_factor=1.1, scale=1.0 / math.sqrt(128),
                                          kv_dtype="bf16"),
    # Varlen prefix-cached prefill: 8 sequences, 32/8 heads, D=128, bs=16,
    # cached_len uniform in [0, 2048], q_len uniform in [128, 1024].
    "varlen_prefill_b8": dict(kind="prefill", seed=4, batch=8, num_heads=32, num_kv_heads=8,
                              head_dim=128, block_size=16, cached=(0, 2048), q_lens=(128, 1024),
                              pool_factor=1.1, scale=1.0 / math.sqrt(128), kv_dtype="bf16"),
}

FP8_MAX = 448.0  # largest finite E4M3 magnitude


@dataclass
class DecodeInputs:
    q: torch.Tensor                 # (B, H, D) bf16
    k_new: torch.Tensor             # (B, Hkv, D) bf16 or uint8 codes
    v_new: torch.Tensor
    slot_mapping: torch.Tensor      # (B,) int64: slot of position context_len-1
    k_cache: torch.Tensor           # (NB, bs, Hkv, D)
    v_cache: torch.Tensor
    block_tables: torch.Tensor      # (B, max_blocks) int32
    context_lens: torch.Tensor      # (B,) int32, includes the new token
    scale: float
    kv_dtype: str = "bf16"
    k_scale: torch.Tensor | None = None       # (NB, Hkv, bs) fp32 (FP8 only)
    v_scale: torch.Tensor | None = None
    k_scale_new: torch.Tensor | None = None   # (B, Hkv) fp32 (FP8 only)
    v_scale_new: torch.Tensor | None = None
    meta: dict = field(default_factory=dict)

    @property
    def batch(self):
        return self.q.shape[0]

    @property
    def num_heads(self):
        return self.q.shape[1]


@dataclass
class PrefillInputs:
    q: torch.Tensor                 # (total_q, H, D) bf16, packed
    k_new: torch.Tensor             # (total_q, Hkv, D) bf16: K of the new tokens
    v_new: torch.Tensor
    slot_mapping: torch.Tensor      # (total_q,) int64
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    block_tables: torch.Tensor      # (B, max_blocks) int32
    cu_seqlens_q: torch.Tensor      # (B+1,) int32
    cu_seqlens_k: torch.Tensor      # (B+1,) int32
    scale: float
    meta: dict = field(default_factory=dict)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, g, device, chunk_rows: int = 1 << 22) -> torch.Tensor:
    """N(0,1) drawn in fp32, rounded to bf16; drawn in row chunks to bound memory."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(shape[0], -1)
    rows = max(1, chunk_rows // max(1, flat.shape[1]))
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device,
                                  dtype=torch.float32).to(torch.bfloat16)
    return out


def _randn_fp8(shape, g, device, chunk_rows: int = 1 << 22):
    """N(0,1) in fp32 quantised to E4M3 with one fp32 scale per row of the last axis.

    scale = amax / 448 (1 if the row is all zero); code = E4M3(x / scale) by
    torch's round-to-nearest-even cast, after clamping to +-448.
    Returns (codes uint8 of `shape`, scales fp32 of shape[:-1]).
    """
    codes = torch.empty(shape, dtype=torch.uint8, device=device)
    scales = torch.empty(shape[:-1], dtype=torch.float32, device=device)
    d = shape[-1]
    fc = codes.view(-1, d)
    fs = scales.view(-1)
    rows = max(1, chunk_rows // d)
    for r0 in range(0, fc.shape[0], rows):
        r1 = min(fc.shape[0], r0 + rows)
        x = torch.randn((r1 - r0, d), generator=g, device=device, dtype=torch.float32)
        amax = x.abs().amax(dim=1)
        s = torch.where(amax > 0, amax / FP8_MAX, torch.ones_like(amax))
        y = (x / s[:, None]).clamp_(-FP8_MAX, FP8_MAX)
        fc[r0:r1] = y.to(torch.float8_e4m3fn).view(torch.uint8)
        fs[r0:r1] = s
    return codes, scales


INT8_MAX = 127.0


def _randn_int8(shape, g, device, chunk_rows: int = 1 << 22):
    """N(0,1) in fp32 quantised to symmetric INT8 with one fp32 scale per row of
    the last axis: scale = amax / 127 (1 if the row is all zero), code =
    round-half-to-even(x / scale), in [-127, 127].
    Returns (codes int8 of `shape`, scales fp32 of shape[:-1])."""
    codes = torch.empty(shape, dtype=torch.int8, device=device)
    scales = torch.empty(shape[:-1], dtype=torch.float32, device=device)
    d = shape[-1]
    fc = codes.view(-1, d)
    fs = scales.view(-1)
    rows = max(1, chunk_rows // d)
    for r0 in range(0, fc.shape[0], rows):
        r1 = min(fc.shape[0], r0 + rows)
        x = torch.randn((r1 - r0, d), generator=g, device=device, dtype=torch.float32)
        amax = x.abs().amax(dim=1)
        s = torch.where(amax > 0, amax / INT8_MAX, torch.ones_like(amax))
        fc[r0:r1] = torch.round(x / s[:, None]).clamp_(-INT8_MAX, INT8_MAX).to(torch.int8)
        fs[r0:r1] = s
    return codes, scales


def draw_lengths(spec, n: int, g_cpu: torch.Generator) -> list[int]:
    kind = spec[0]
    if kind == "uniform":
        lo, hi = spec[1], spec[2]
        return torch.randint(lo, hi + 1, (n,), generator=g_cpu).tolist()
    if kind == "lognormal":
        median, sigma, lo, hi = spec[1], spec[2], spec[3], spec[4]
        z = torch.randn((n,), generator=g_cpu, dtype=torch.float64)
        x = torch.exp(math.log(median) + sigma * z)
        return torch.clamp(torch.round(x), lo, hi).to(torch.int64).tolist()
    raise ValueError(kind)


def _assign_blocks(blocks_needed: list[int], num_blocks: int, g_cpu) -> torch.Tensor:
    perm = torch.randperm(num_blocks, generator=g_cpu).to(torch.int32)
    width = max(1, max(blocks_needed) if blocks_needed else 1)
    bt = torch.full((len(blocks_needed), width), -1, dtype=torch.int32)
    pos = 0
    for i, nb in enumerate(blocks_needed):
        bt[i, :nb] = perm[pos:pos + nb]
        pos += nb
    if pos > num_blocks:
        raise ValueError("pool too small for the requested lengths")
    return bt


def _slot(bt_row: torch.Tensor, p: int, bs: int) -> int:
    return int(bt_row[p // bs]) * bs + p % bs


def make_decode(batch: int, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                context_lens, *, num_blocks: int | None = None, pool_factor: float = 1.1,
                seed: int = 0, device="cpu", kv_dtype: str = "bf16", sinks: int = 0,
                scale: float | None = None) -> DecodeInputs:
    """Decode inputs for one step: the cache holds positions 0..L-2 of every
    sequence and the new token (position L-1) comes as k_new/v_new with its slot,
    to be appended by store_kv before attention."""
    g_cpu = _gen(seed, "cpu")
    lens = [int(x) for x in context_lens]
    need = [max(1, -(-L // block_size)) for L in lens]
    if num_blocks is None:
        num_blocks = max(1, math.ceil(sum(need) * pool_factor))
    bt = _assign_blocks(need, num_blocks, g_cpu)
    sink_pos = []
    for L in lens:
        k = min(sinks, L)
        sink_pos.append(sorted(torch.randperm(L, generator=g_cpu)[:k].tolist()) if k else [])
    g = _gen(seed + 1000, device)
    cache_shape = (num_blocks, block_size, num_kv_heads, head_dim)
    ks = vs = ksn = vsn = None
    if kv_dtype == "bf16":
        k_cache = _randn_bf16(cache_shape, g, device)
        v_cache = _randn_bf16(cache_shape, g, device)
        k_new = _randn_bf16((batch, num_kv_heads, head_dim), g, device)
        v_new = _randn_bf16((batch, num_kv_heads, head_dim), g, device)
    elif kv_dtype == "fp8":
        k_cache, ks = _randn_fp8(cache_shape, g, device)
        v_cache, vs = _randn_fp8(cache_shape, g, device)
        ks = ks.permute(0, 2, 1).contiguous()  # (NB, Hkv, bs)
        vs = vs.permute(0, 2, 1).contiguous()
        k_new, ksn = _randn_fp8((batch, num_kv_heads, head_dim), g, device)
        v_new, vsn = _randn_fp8((batch, num_kv_heads, head_dim), g, device)
    elif kv_dtype == "int8":
        k_cache, ks = _randn_int8(cache_shape, g, device)
        v_cache, vs = _randn_int8(cache_shape, g, device)
        ks = ks.permute(0, 2, 1).contiguous()  # (NB, Hkv, bs)
        vs = vs.permute(0, 2, 1).contiguous()
        k_new, ksn = _randn_int8((batch, num_kv_heads, head_dim), g, device)
        v_new, vsn = _randn_int8((batch, num_kv_heads, head_dim), g, device)
    else:
        raise ValueError(kv_dtype)
    q = _randn_bf16((batch, num_heads, head_dim), g, device)
    slots = []
    for i, L in enumerate(lens):
        slots.append(_slot(bt[i], L - 1, block_size) if L > 0 else -1)
    # attention sinks: the key vectors at the chosen positions get 4x the norm
    if sinks:
        if kv_dtype != "bf16":
            raise ValueError("sinks are defined for the bf16 workload")
        kflat = k_cache.view(-1, num_kv_heads, head_dim)
        for i, L in enumerate(lens):
            for p in sink_pos[i]:
                if p == L - 1:
                    k_new[i] = k_new[i] * 4
                else:
                    s = _slot(bt[i], p, block_size)
                    kflat[s] = kflat[s] * 4
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return DecodeInputs(
        q=q, k_new=k_new, v_new=v_new,
        slot_mapping=torch.tensor(slots, dtype=torch.int64, device=device),
        k_cache=k_cache, v_cache=v_cache, block_tables=bt.to(device),
        context_lens=torch.tensor(lens, dtype=torch.int32, device=device), scale=float(scale),
        kv_dtype=kv_dtype, k_scale=ks, v_scale=vs, k_scale_new=ksn, v_scale_new=vsn,
        meta=dict(lens=lens, sink_positions=sink_pos, num_blocks=num_blocks, seed=seed))


def make_prefill(batch: int, num_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                 cached_lens, q_lens, *, num_blocks: int | None = None, pool_factor: float = 1.1,
                 seed: int = 0, device="cpu", scale: float | None = None) -> PrefillInputs:
    """Prefill inputs: positions 0..cached-1 of each sequence are already in the
    paged cache; the q_len new tokens (positions cached..kv_len-1) come packed,
    with their K/V and slots, to be stored before attention."""
    g_cpu = _gen(seed, "cpu")
    cached = [int(x) for x in cached_lens]
    qls = [int(x) for x in q_lens]
    kv = [c + n for c, n in zip(cached, qls)]
    need = [max(1, -(-L // block_size)) for L in kv]
    if num_blocks is None:
        num_blocks = max(1, math.ceil(sum(need) * pool_factor))
    bt = _assign_blocks(need, num_blocks, g_cpu)
    g = _gen(seed + 1000, device)
    cache_shape = (num_blocks, block_size, num_kv_heads, head_dim)
    k_cache = _randn_bf16(cache_shape, g, device)
    v_cache = _randn_bf16(cache_shape, g, device)
    total_q = sum(qls)
    q = _randn_bf16((max(total_q, 1), num_heads, head_dim), g, device)[:total_q]
    k_new = _randn_bf16((max(total_q, 1), num_kv_heads, head_dim), g, device)[:total_q]
    v_new = _randn_bf16((max(total_q, 1), num_kv_heads, head_dim), g, device)[:total_q]
    slots = []
    for i in range(batch):
        for p in range(cached[i], kv[i]):
            slots.append(_slot(bt[i], p, block_size))
    cu_q = [0]
    cu_k = [0]
    for i in range(batch):
        cu_q.append(cu_q[-1] + qls[i])
        cu_k.append(cu_k[-1] + kv[i])
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return PrefillInputs(
        q=q.contiguous(), k_new=k_new.contiguous(), v_new=v_new.contiguous(),
        slot_mapping=torch.tensor(slots, dtype=torch.int64, device=device),
        k_cache=k_cache, v_cache=v_cache, block_tables=bt.to(device),
        cu_seqlens_q=torch.tensor(cu_q, dtype=torch.int32, device=device),
        cu_seqlens_k=torch.tensor(cu_k, dtype=torch.int32, device=device), scale=float(scale),
        meta=dict(cached=cached, q_lens=qls, kv_lens=kv, num_blocks=num_blocks, seed=seed))


def workload_lengths(name: str) -> list[int]:
    """The context lengths a decode workload draws (cheap: no tensors)."""
    w = WORKLOADS[name]
    if "context_lens" in w:
        return list(w["context_lens"])
    return draw_lengths(w["lens"], w["batch"], _gen(w["seed"], "cpu"))


def prefill_lengths(name: str) -> tuple[list[int], list[int]]:
    """(cached lengths, new-token counts) a prefill workload draws (cheap: no tensors)."""
    w = WORKLOADS[name]
    g_cpu = _gen(w["seed"], "cpu")
    cached = torch.randint(w["cached"][0], w["cached"][1] + 1, (w["batch"],),
                           generator=g_cpu).tolist()
    qls = torch.randint(w["q_lens"][0], w["q_lens"][1] + 1, (w["batch"],),
                        generator=g_cpu).tolist()
    return cached, qls


def make_workload(name: str, device="cpu", variant: int = 0):
    """Inputs of one of the named workloads, at full size. `variant` > 0 draws
    another set of values (same lengths and shapes) for rotating buffers."""
    w = dict(WORKLOADS[name])
    kind = w.pop("kind")
    seed = w.pop("seed")
    g_cpu = _gen(seed, "cpu")
    if kind == "decode":
        lens = w.pop("context_lens", None)
        spec = w.pop("lens", None)
        if lens is None:
            lens = draw_lengths(spec, w["batch"], g_cpu)
        return make_decode(w.pop("batch"), w.pop("num_heads"), w.pop("num_kv_heads"),
                           w.pop("head_dim"), w.pop("block_size"), lens,
                           seed=seed + 7 + 7919 * variant, device=device, **w)
    cached, qls = prefill_lengths(name)
    return make_prefill(w["batch"], w["num_heads"], w["num_kv_heads"], w["head_dim"],
                        w["block_size"], cached, qls, pool_factor=w["pool_factor"],
                        seed=seed + 7 + 7919 * variant, device=device, scale=w["scale"])


def bf16_bits(t: torch.Tensor):
    """A bf16 tensor's raw bits as a numpy uint16 array (on the host)."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor):
    return t.detach().contiguous().cpu().numpy()
