"""Decode captured once in a CUDA graph and replayed as a decode loop.

The engine of "Decode Phase Attention Forward Pass" runs its decode step
under CUDA-graph capture (its warm-up pass exists for that, section 1), and
"Prefill Forward Prefix Caching Explained" notes that capture forbids
host reads of device lengths ("What comes out"). Here lengths live on the
device and the persistent decode grid depends only on the batch, so one graph
serves every step. A graph freezes the kernel parameters, the split-K
counters' call tag among them, so these tests replay each graph several
times back to back with nothing else touching its workspace, every step with
new queries and one more token per sequence, at shapes where most
(sequence, kv head) segments are split across warps and merged in-kernel.
Every replay is compared with the oracle (its own store of each step's new
token, then its decode); the same steps run eagerly on their own cache and
workspace must give bit-identical outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import assert_attention_close, to_device

pytestmark = pytest.mark.gpu


def _step_inputs(base, step, gen):
    """Inputs of decode step `step`: every sequence grows by one token."""
    B, Hkv, D = base.k_new.shape
    H = base.q.shape[1]
    bs = base.k_cache.shape[1]
    lens = base.context_lens + step
    slots = []
    for b in range(B):
        p = int(lens[b]) - 1  # -1: no token yet, nothing to store
        slots.append(int(base.block_tables[b, p // bs]) * bs + p % bs if p >= 0 else -1)
    mk = lambda *s: torch.randn(*s, generator=gen).to(torch.bfloat16)
    return dict(q=mk(B, H, D), k_new=mk(B, Hkv, D), v_new=mk(B, Hkv, D),
                slot_mapping=torch.tensor(slots, dtype=torch.int64), context_lens=lens.clone())


class OracleLoop:
    """The oracle's own decode loop over a host copy of the cache."""

    def __init__(self, h):
        self.kc = W.bf16_bits(h.k_cache).copy()
        self.vc = W.bf16_bits(h.v_cache).copy()
        self.bt = h.block_tables.numpy()
        self.scale = h.scale

    def step(self, x):
        oracle.store_kv(W.bf16_bits(x["k_new"]), W.bf16_bits(x["v_new"]),
                        x["slot_mapping"].numpy(), self.kc, self.vc)
        return oracle.decode(W.bf16_bits(x["q"]), self.kc, self.vc, self.bt,
                             x["context_lens"].numpy(), self.scale)


def _setup(B, H, Hkv, lens0, steps, seed):
    # room in the block table for the extra tokens
    h = W.make_decode(B, H, Hkv, 128, 16, [L + steps for L in lens0], seed=seed)
    h.context_lens = torch.tensor(lens0, dtype=torch.int32)
    gen = torch.Generator().manual_seed(seed + 1)
    return h, [_step_inputs(h, s, gen) for s in range(steps)]


def _workspace(g, B, H):
    n = pa.decode_workspace_size(g.k_cache, B, H, g.block_tables.shape[1])
    return torch.empty(max(n, 16), dtype=torch.uint8, device="cuda")


def _replay_loop(h, inputs, run, B, H):
    """Capture run(static inputs, cache, out, ws) once, replay it once per
    step back to back; compare each replay with the oracle and with the same
    step run eagerly (own cache copy, own workspace)."""
    graph_state, eager_state = to_device(h), to_device(h)
    ws_graph, ws_eager = _workspace(graph_state, B, H), _workspace(eager_state, B, H)
    static = {k: v.cuda() for k, v in inputs[0].items()}
    out_g = torch.empty((B, H, 128), dtype=torch.bfloat16, device="cuda")

    # warm-up on a side stream does the one-time host set-up before capture
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        scratch = to_device(h)
        run(static, scratch, out_g, _workspace(scratch, B, H))
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    del scratch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run(static, graph_state, out_g, ws_graph)

    ref = OracleLoop(h)
    eager_outs = []
    for step, x in enumerate(inputs):
        for k, v in x.items():
            static[k].copy_(v)
        g.replay()
        torch.cuda.synchronize()
        got = out_g.clone()
        assert pa.get_device_error() == 0
        assert_attention_close(got, ref.step(x), f"replay {step} vs oracle")
        eager_outs.append(got)
    # the eager loop afterwards, on its own cache and workspace
    for step, x in enumerate(inputs):
        e = run({k: v.cuda() for k, v in x.items()}, eager_state, None, ws_eager)
        torch.cuda.synchronize()
        assert torch.equal(e.view(torch.int16), eager_outs[step].view(torch.int16)), \
            f"replay {step} differs from the eager call"
    assert torch.equal(graph_state.k_cache.view(torch.int16), eager_state.k_cache.view(torch.int16))
    assert torch.equal(graph_state.v_cache.view(torch.int16), eager_state.v_cache.view(torch.int16))


def _store_then_decode(x, cache, out, ws):
    pa.store_kv(x["k_new"], x["v_new"], x["slot_mapping"], cache.k_cache, cache.v_cache)
    return pa.decode(x["q"], cache.k_cache, cache.v_cache, cache.block_tables, x["context_lens"],
                     cache.scale, out=out, workspace=ws)


def _fused_append(x, cache, out, ws):
    return pa.decode_append(x["q"], x["k_new"], x["v_new"], cache.k_cache, cache.v_cache,
                            cache.block_tables, x["context_lens"], cache.scale, out=out,
                            workspace=ws)


def _bench_shaped_lengths(seed):
    # the Llama-3-8B-shaped decode's length recipe, batch 64
    gen = torch.Generator().manual_seed(seed)
    return torch.randint(512, 4097, (64,), generator=gen).tolist()


def test_captured_store_and_decode_replays_back_to_back():
    lens0 = _bench_shaped_lengths(120)
    h, inputs = _setup(64, 32, 8, lens0, 5, seed=121)
    _replay_loop(h, inputs, _store_then_decode, 64, 32)


def test_captured_decode_append_replays_back_to_back():
    lens0 = _bench_shaped_lengths(122)
    h, inputs = _setup(64, 32, 8, lens0, 5, seed=123)
    _replay_loop(h, inputs, _fused_append, 64, 32)


def test_captured_decode_replays_with_short_and_long_sequences():
    # lengths crossing block and split boundaries as they grow, zero-length rows
    lens0 = [1, 15, 16, 300, 1024, 2047, 0, 77, 3000, 129, 640, 2500]
    h, inputs = _setup(12, 32, 8, lens0, 5, seed=124)
    _replay_loop(h, inputs, _store_then_decode, 12, 32)


def test_captured_decode_replays_grouped_merges():
    # one long sequence: every (sequence, kv head) segment is split into more
    # than 32 parts, which merge in groups of 16 (group counters) and then
    # across groups (segment counters)
    h, inputs = _setup(1, 32, 8, [70001], 4, seed=125)
    _replay_loop(h, inputs, _fused_append, 1, 32)


def test_captured_window_and_fp8_decodes_replay_back_to_back():
    # the sliding-window instantiation and the 8-bit instantiation, each
    # captured once and replayed with new queries, against the oracle
    lens = _bench_shaped_lengths(128)
    for kv, H, Hkv, bs in (("bf16", 32, 8, 16), ("fp8", 64, 8, 32)):
        h = W.make_decode(64, H, Hkv, 128, bs, lens, seed=129, kv_dtype=kv)
        g_state = to_device(h)
        n = pa.decode_workspace_size(g_state.k_cache, 64, H, g_state.block_tables.shape[1],
                                     k_scale=g_state.k_scale, v_scale=g_state.v_scale)
        assert n > 0
        ws = torch.empty(n, dtype=torch.uint8, device="cuda")
        out = torch.empty((64, H, 128), dtype=torch.bfloat16, device="cuda")
        q = g_state.q.clone()
        pa.store_kv(g_state.k_new, g_state.v_new, g_state.slot_mapping, g_state.k_cache,
                    g_state.v_cache, g_state.k_scale_new, g_state.v_scale_new, g_state.k_scale,
                    g_state.v_scale)
        window, sinks = (1024, 4) if kv == "bf16" else (0, 0)

        def run():
            return pa.decode_window(q, g_state.k_cache, g_state.v_cache, g_state.block_tables,
                                    g_state.context_lens, g_state.scale, window, sinks, out=out,
                                    workspace=ws, k_scale=g_state.k_scale, v_scale=g_state.v_scale)

        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            run()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run()
        # the oracle's cache after the one store
        if kv == "bf16":
            kc, vc = W.bf16_bits(h.k_cache).copy(), W.bf16_bits(h.v_cache).copy()
            oracle.store_kv(W.bf16_bits(h.k_new), W.bf16_bits(h.v_new), h.slot_mapping.numpy(),
                            kc, vc)
            ks = vs = None
        else:
            kc, vc = W.u8(h.k_cache).copy(), W.u8(h.v_cache).copy()
            ks, vs = h.k_scale.numpy().copy(), h.v_scale.numpy().copy()
            oracle.store_kv(W.u8(h.k_new), W.u8(h.v_new), h.slot_mapping.numpy(), kc, vc,
                            h.k_scale_new.numpy(), h.v_scale_new.numpy(), ks, vs)
        gen = torch.Generator().manual_seed(130)
        for r in range(4):
            qh = torch.randn(q.shape, generator=gen).to(torch.bfloat16)
            q.copy_(qh)
            out.fill_(float("nan"))
            graph.replay()
            torch.cuda.synchronize()
            assert pa.get_device_error() == 0
            want = oracle.decode(W.bf16_bits(qh), kc, vc, h.block_tables.numpy(),
                                 h.context_lens.numpy(), h.scale, k_scale=ks, v_scale=vs,
                                 window=window, sinks=sinks)
            assert_attention_close(out, want, f"{kv} window {window} replay {r}")


def test_replays_of_an_unchanged_step_stay_correct():
    # the same inputs every replay: the output must not change between replays
    lens0 = _bench_shaped_lengths(126)
    h, inputs = _setup(64, 32, 8, lens0, 1, seed=127)
    g_state = to_device(h)
    ws = _workspace(g_state, 64, 32)
    static = {k: v.cuda() for k, v in inputs[0].items()}
    out = torch.empty((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pa.decode(static["q"], g_state.k_cache, g_state.v_cache, g_state.block_tables,
                  static["context_lens"], g_state.scale, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pa.decode(static["q"], g_state.k_cache, g_state.v_cache, g_state.block_tables,
                  static["context_lens"], g_state.scale, out=out, workspace=ws)
    want = oracle.decode(W.bf16_bits(inputs[0]["q"]), W.bf16_bits(h.k_cache),
                         W.bf16_bits(h.v_cache), h.block_tables.numpy(),
                         inputs[0]["context_lens"].numpy(), h.scale)
    first = None
    for r in range(4):
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pa.get_device_error() == 0
        assert_attention_close(out, want, f"replay {r}")
        if first is None:
            first = out.clone()
        assert torch.equal(out.view(torch.int16), first.view(torch.int16))
    assert np.isfinite(want).all()
