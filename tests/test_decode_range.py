"""Operand ranges of the 8-bit decode path against the oracle.

With an 8-bit cache (the "Decode Phase" glossary's FP8 / INT8 KV-cache
quantisation, with dequantisation in the kernel) the kernels feed the tensor
cores f16 operands: q (given in bf16) and the probabilities times the V
scales. The kernels scale both by powers of two chosen from the data, so
results stay within the decode tolerance whatever the magnitudes. These cases
multiply q, the K scales or the V scales of a random workload by 2^10 (about
10^3), 2^24, 2^-13 (about 10^-4) or 2^-20 (about 10^-6). Attention is linear in V,
so with scaled V scales both outputs are divided by the same power of two
before the comparison (exact in bf16 and fp64), which keeps the stated
tolerance in units of V.
"""
import numpy as np
import pytest
import torch

import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import assert_attention_close, oracle_store_and_decode, to_device

pytestmark = pytest.mark.gpu

LENS = [1, 31, 33, 700, 2500, 64]


def _scaled(kv, what, f, seed):
    H, Hkv, bs = (64, 8, 32) if kv != "bf16" else (32, 8, 16)
    h = W.make_decode(len(LENS), H, Hkv, 128, bs, LENS, seed=seed, kv_dtype=kv)
    if what == "q":
        h.q = (h.q.float() * f).to(torch.bfloat16)
    elif what == "k_scale":
        h.k_scale, h.k_scale_new = h.k_scale * f, h.k_scale_new * f
    elif what == "v_scale":
        h.v_scale, h.v_scale_new = h.v_scale * f, h.v_scale_new * f
    return h


CASES = [(kv, what, f) for kv in ("fp8", "int8")
         for what, f in (("q", 2.0 ** 10), ("q", 2.0 ** -13), ("k_scale", 2.0 ** 10),
                         ("k_scale", 2.0 ** -20), ("v_scale", 2.0 ** 10),
                         ("v_scale", 2.0 ** 24), ("v_scale", 2.0 ** -20))]
CASES += [("bf16", "q", 2.0 ** 10), ("bf16", "q", 2.0 ** -13)]


@pytest.mark.parametrize("kv,what,f", CASES, ids=lambda x: str(x))
def test_scaled_operands_match_oracle(kv, what, f):
    h = _scaled(kv, what, f, seed=400 + len(what))
    want = oracle_store_and_decode(h)
    g = to_device(h)
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, g.k_scale_new,
                g.v_scale_new, g.k_scale, g.v_scale)
    got = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                    k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    norm = f if what == "v_scale" else 1.0
    assert_attention_close((got.float() / norm).to(torch.bfloat16) if norm != 1.0 else got,
                           want / norm, f"{kv} {what} x {f:g}")


@pytest.mark.parametrize("kv", ["fp8", "int8"])
def test_v_scales_spanning_many_octaves_in_one_sequence(kv):
    # V scales that change by 2^12 and 2^24 from block to block within a
    # sequence: the kernel's power-of-two factor for P.V moves with them in
    # both directions. Outputs then mix terms of very different sizes, so the
    # check is relative to the largest output: every element within 1e-2 of
    # max|oracle|, and rel-L2 <= 5e-3.
    h = W.make_decode(2, 64, 8, 128, 32, [3000, 1500], seed=410, kv_dtype=kv)
    nb = h.v_scale.shape[0]
    octave = torch.tensor([2.0 ** (12 * ((i % 3) - 1)) for i in range(nb)]).view(nb, 1, 1)
    h.v_scale = h.v_scale * octave
    want = oracle_store_and_decode(h)
    g = to_device(h)
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, g.k_scale_new,
                g.v_scale_new, g.k_scale, g.v_scale)
    got = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                    k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    got = got.double().cpu().numpy()
    assert np.isfinite(got).all()
    err = np.abs(got - want)
    assert err.max() <= 1e-2 * np.abs(want).max(), (err.max(), np.abs(want).max())
    assert np.linalg.norm(got - want) <= 5e-3 * np.linalg.norm(want)
