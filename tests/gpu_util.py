"""Helpers shared by the GPU parity tests: move inputs, cut a sub-problem for
the oracle, compare with the stated tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

# Attention outputs (bf16 out, fp32 accumulation) against the fp64 oracle:
# |gpu - oracle| <= ATOL + |bf16(oracle) - oracle| element-wise, and relative
# L2 <= REL_L2. The second term is the rounding of the exact result to the
# bf16 output format, which every bf16-output implementation incurs: it is
# zero where the exact result is a bf16 value and exceeds 1e-2 only where
# |oracle| >= 4 (bf16 half-ulp there is 2^-6).
ATOL = 1e-2
REL_L2 = 5e-3


def to_device(inp, device="cuda"):
    d = {}
    for k, v in inp.__dict__.items():
        d[k] = v.to(device) if isinstance(v, torch.Tensor) else v
    return type(inp)(**d)


def host_subproblem(inp: W.DecodeInputs, seqs) -> W.DecodeInputs:
    """Host copy of sequences `seqs` of a decode input, with only their
    physical blocks, renumbered 0..n-1 (block tables and slots remapped).
    Must be taken before the GPU writes the new tokens into the cache."""
    seqs = torch.as_tensor(seqs, dtype=torch.long)
    bs = inp.k_cache.shape[1]
    bt = inp.block_tables.cpu()[seqs]
    lens = inp.context_lens.cpu()[seqs]
    used = sorted({int(x) for x in bt[bt >= 0].tolist()})
    remap = {old: new for new, old in enumerate(used)}
    idx = torch.tensor(used, dtype=torch.long, device=inp.k_cache.device)
    new_bt = torch.full_like(bt, -1)
    for i in range(bt.shape[0]):
        for j in range(bt.shape[1]):
            if int(bt[i, j]) >= 0:
                new_bt[i, j] = remap[int(bt[i, j])]
    slots = inp.slot_mapping.cpu()[seqs].clone()
    for i in range(len(slots)):
        s = int(slots[i])
        if s >= 0:
            slots[i] = remap[s // bs] * bs + s % bs
    sel = seqs.to(inp.q.device)
    opt = lambda t: None if t is None else t.index_select(0, sel).cpu()
    return W.DecodeInputs(
        q=inp.q.index_select(0, sel).cpu(), k_new=inp.k_new.index_select(0, sel).cpu(),
        v_new=inp.v_new.index_select(0, sel).cpu(), slot_mapping=slots,
        k_cache=inp.k_cache.index_select(0, idx).cpu(), v_cache=inp.v_cache.index_select(0, idx).cpu(),
        block_tables=new_bt, context_lens=lens, scale=inp.scale, kv_dtype=inp.kv_dtype,
        k_scale=None if inp.k_scale is None else inp.k_scale.index_select(0, idx).cpu(),
        v_scale=None if inp.v_scale is None else inp.v_scale.index_select(0, idx).cpu(),
        k_scale_new=opt(inp.k_scale_new), v_scale_new=opt(inp.v_scale_new))


def oracle_store_and_decode(h: W.DecodeInputs) -> np.ndarray:
    """The oracle's own append of the new tokens, then its decode (host inputs)."""
    if h.kv_dtype == "bf16":
        kc, vc = W.bf16_bits(h.k_cache).copy(), W.bf16_bits(h.v_cache).copy()
        oracle.store_kv(W.bf16_bits(h.k_new), W.bf16_bits(h.v_new), h.slot_mapping.numpy(), kc, vc)
        return oracle.decode(W.bf16_bits(h.q), kc, vc, h.block_tables.numpy(),
                             h.context_lens.numpy(), h.scale)
    kc, vc = W.u8(h.k_cache).copy(), W.u8(h.v_cache).copy()
    ks, vs = h.k_scale.numpy().copy(), h.v_scale.numpy().copy()
    oracle.store_kv(W.u8(h.k_new), W.u8(h.v_new), h.slot_mapping.numpy(), kc, vc,
                    h.k_scale_new.numpy(), h.v_scale_new.numpy(), ks, vs)
    return oracle.decode(W.bf16_bits(h.q), kc, vc, h.block_tables.numpy(), h.context_lens.numpy(),
                         h.scale, k_scale=ks, v_scale=vs)


def output_rounding(want: np.ndarray) -> np.ndarray:
    """|bf16(want) - want|: the error of rounding the exact result to bf16."""
    r = torch.from_numpy(np.ascontiguousarray(want)).float().to(torch.bfloat16).double().numpy()
    return np.abs(r - want)


def attention_errors(got: torch.Tensor, want: np.ndarray):
    g = got.detach().float().cpu().double().numpy()
    diff = g - want
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    excess = float((np.abs(diff) - output_rounding(want)).max()) if diff.size else 0.0
    denom = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, excess, rel


def assert_attention_close(got: torch.Tensor, want: np.ndarray, what: str = ""):
    assert torch.isfinite(got.float()).all(), f"{what}: non-finite output"
    max_abs, excess, rel = attention_errors(got, want)
    assert excess <= ATOL and rel <= REL_L2, \
        f"{what}: max_abs={max_abs:.3e} beyond-rounding={excess:.3e} rel_l2={rel:.3e}"
    return max_abs, rel
