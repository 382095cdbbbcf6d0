"""store_kv + decode captured once in a CUDA graph and replayed as a decode
loop: lengths live on the device and the persistent decode grid does not
depend on them, so one graph serves every step. Each replay is compared with
the same step run eagerly on a copy of the cache (same tolerance as decode),
and the first step also with the oracle."""
import pytest
import torch

import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import assert_attention_close, oracle_store_and_decode, to_device

pytestmark = pytest.mark.gpu


def _step_inputs(base, step, gen):
    """Inputs of decode step `step`: every sequence grows by one token."""
    B, Hkv, D = base.k_new.shape
    H = base.q.shape[1]
    bs = base.k_cache.shape[1]
    lens = base.context_lens + step
    slots = []
    for b in range(B):
        p = int(lens[b]) - 1
        slots.append(int(base.block_tables[b, p // bs]) * bs + p % bs)
    mk = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)
    return dict(q=mk(B, H, D), k_new=mk(B, Hkv, D), v_new=mk(B, Hkv, D),
                slot_mapping=torch.tensor(slots, dtype=torch.int64), context_lens=lens.clone())


def test_captured_store_and_decode_replays_over_growing_lengths():
    B, H, Hkv, D, bs = 12, 32, 8, 128, 16
    lens0 = [1, 15, 16, 300, 1024, 2047, 5, 77, 3000, 129, 640, 2500]
    steps = 4
    # room in the block table for the extra tokens
    h = W.make_decode(B, H, Hkv, D, bs, [L + steps for L in lens0], seed=120)
    h.context_lens = torch.tensor(lens0, dtype=torch.int32)
    gen = torch.Generator().manual_seed(121)
    inputs = [_step_inputs(h, s, gen) for s in range(steps)]
    # first step also against the oracle (its own store of the new token)
    first = W.DecodeInputs(**{**h.__dict__, **inputs[0]})
    want0 = oracle_store_and_decode(first)

    eager = to_device(h)
    graph = to_device(h)
    static = {k: v.cuda() for k, v in inputs[0].items()}
    out_g = torch.empty((B, H, D), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(pa.decode_workspace_size(graph.k_cache, B, H, graph.block_tables.shape[1]),
                     dtype=torch.uint8, device="cuda")

    def run(x, cache, out):
        pa.store_kv(x["k_new"], x["v_new"], x["slot_mapping"], cache.k_cache, cache.v_cache)
        return pa.decode(x["q"], cache.k_cache, cache.v_cache, cache.block_tables,
                         x["context_lens"], cache.scale, out=out, workspace=ws)

    # warm-up on a side stream does the one-time host set-up before capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        scratch = to_device(h)
        run(static, scratch, out_g)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(static, graph, out_g)

    for step, x in enumerate(inputs):
        for k, v in x.items():
            static[k].copy_(v)
        g.replay()
        ref = run({k: v.cuda() for k, v in x.items()}, eager, None)
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        diff = (out_g.float() - ref.float()).abs().max().item()
        assert diff == 0.0, f"step {step}: graph replay differs from eager by {diff}"
        if step == 0:
            assert_attention_close(out_g, want0, "graph step 0 vs oracle")
    assert torch.equal(graph.k_cache.view(torch.int16), eager.k_cache.view(torch.int16))
