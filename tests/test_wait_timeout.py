"""Failure detection on the GPU without a fault: a decode launch whose
bounded wait on a block copy runs out must record PA_DEVERR_WAIT_TIMEOUT,
let its copies in flight land and return, leaving the context usable.

The wait is made to run out on purpose with the library's test hook
(pa_debug_inject_wait_timeout): the first warp of the first CTA leaves one
block copy unissued, so nothing ever completes that stage's barrier (a flag
that nothing sets). The wait bound is shortened to 2 ms for the test. The
next normal call must match the oracle.
"""
import time

import pytest
import torch

import paged_kv_cache_186_gb300 as pa
import workloads as W
from gpu_util import assert_attention_close, oracle_store_and_decode, to_device

pytestmark = pytest.mark.gpu

LIMIT_NS = 2_000_000  # 2 ms


@pytest.fixture
def disarm():
    yield
    pa.debug_inject_wait_timeout(-1)


@pytest.mark.parametrize("skip_copy", [0, 1, 3])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_wait_that_runs_out_is_reported_and_the_next_call_is_correct(skip_copy, kv, disarm):
    lens = [700, 45, 2000, 300]
    H, Hkv, bs = (32, 8, 16) if kv == "bf16" else (64, 8, 32)
    h = W.make_decode(len(lens), H, Hkv, 128, bs, lens, seed=300 + skip_copy, kv_dtype=kv)
    want = oracle_store_and_decode(h)
    g = to_device(h)
    pa.store_kv(g.k_new, g.v_new, g.slot_mapping, g.k_cache, g.v_cache, g.k_scale_new,
                g.v_scale_new, g.k_scale, g.v_scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0

    pa.debug_inject_wait_timeout(skip_copy, LIMIT_NS)
    t0 = time.perf_counter()
    pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
              k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    err = pa.get_device_error()
    assert err & pa.PA_DEVERR_WAIT_TIMEOUT, f"error word {err:#x}"
    # the failing warp waited twice (its block, then the drain), each bounded
    assert elapsed < 1.0, f"launch with a bounded wait took {elapsed:.3f} s"

    pa.debug_inject_wait_timeout(-1)
    out = pa.decode(g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.scale,
                    k_scale=g.k_scale, v_scale=g.v_scale)
    torch.cuda.synchronize()
    assert pa.get_device_error() == 0
    assert_attention_close(out, want, "call after the timeout")
