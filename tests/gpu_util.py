"""Helpers shared by the GPU parity tests: move inputs, run the oracle on the
same inputs, compare with the stated tolerance."""
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


# Below this magnitude the bf16 rounding of the exact result is at most 2^-7,
# so the plain bound max|gpu - oracle| <= ATOL applies with no rounding term.
PLAIN_BELOW = 4.0


def attention_errors(got: torch.Tensor, want: np.ndarray):
    g = got.detach().float().cpu().double().numpy()
    diff = g - want
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    excess = float((np.abs(diff) - output_rounding(want)).max()) if diff.size else 0.0
    small = np.abs(want) < PLAIN_BELOW
    plain = float(np.abs(diff[small]).max()) if small.any() else 0.0
    denom = float(np.linalg.norm(want))
    rel = float(np.linalg.norm(diff) / denom) if denom > 0 else float(np.linalg.norm(diff))
    return max_abs, excess, plain, rel


def assert_attention_close(got: torch.Tensor, want: np.ndarray, what: str = ""):
    """The stated tolerance: max-abs <= 1e-2 wherever |oracle| < 4, max-abs
    <= 1e-2 beyond the output's own bf16 rounding everywhere, rel-L2 <= 5e-3."""
    assert tuple(got.shape) == tuple(want.shape), f"{what}: shape {tuple(got.shape)} vs {want.shape}"
    assert torch.isfinite(got.float()).all(), f"{what}: non-finite output"
    max_abs, excess, plain, rel = attention_errors(got, want)
    assert plain <= ATOL and excess <= ATOL and rel <= REL_L2, \
        (f"{what}: max_abs={max_abs:.3e} max_abs(|oracle|<4)={plain:.3e} "
         f"beyond-rounding={excess:.3e} rel_l2={rel:.3e}")
    return max_abs, rel


def host_copy(inp):
    """Host copy of every tensor of a workload (take it before the GPU writes
    the new tokens into the cache)."""
    return to_device(inp, "cpu")
