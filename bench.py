"""Benchmark of the paged decode hot path on GB300.

One step = the append of the batch's new tokens to the cache + decode
attention over the whole batch, by default through pa_decode_append (one
persistent launch that stores each new row while attending; --step separate
times pa_store_kv + pa_decode instead), on the Llama-3-8B-shaped workload
(batch 64, 32/8 heads, head_dim 128, block_size 16, context_len ~ U[512, 4096])
unless --workload says otherwise.

Prints ONE JSON line (rank 0). Inputs are resident in HBM before timing; the
step rotates over several independently drawn KV pools so consecutive steps
never re-read KV from L2. The decode launch is also timed on its own with CUDA
events inside the timed region for the roofline figure. The default run also
measures the other workloads (the tiny decode, the long-context decode with
and without a sliding window, the FP8 and INT8 70B-shaped decodes and the
varlen prefill) in the same process and adds them to the line under
"workloads", each with its own oracle baseline and clock record
(--headline-only skips them).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_BYTES = 129 * 2 ** 20
METRIC = "Paged decode attention KV-cache GB/s (% of GB300 HBM peak), seq-steps/s"
DEFAULT_WORKLOAD = "llama3_8b_decode_b64"


def visible_keys(L: int, window: int = 0, sinks: int = 0) -> int:
    """Keys a query attends to: all L, or with a sliding window the last
    `window` plus the first `sinks` (counted once where they meet)."""
    if window <= 0 or L <= window:
        return L
    return min(sinks, L - window) + window


def kv_bytes(name: str, lens, window: int = 0, sinks: int = 0) -> int:
    w = W.WORKLOADS[name]
    q8 = w["kv_dtype"] in ("fp8", "int8")
    eb = 1 if q8 else 2
    per_tok = w["num_kv_heads"] * w["head_dim"] * eb * 2
    if q8:
        per_tok += w["num_kv_heads"] * 4 * 2  # one fp32 scale per (token, head) for K and V
    return int(sum(visible_keys(L, window, sinks) for L in lens)) * per_tok


def _measured(keys):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    for k in keys:
        v = d.get(k)
        if isinstance(v, dict):
            v = v.get("value")
        if v:
            return float(v)
    return None


def peaks():
    hbm = _measured(("hbm_gbs", "hbm_GBps", "hbm"))
    return (hbm, "measured") if hbm else (FALLBACK_HBM_GBS, "fallback")


def tensor_peak():
    tf = _measured(("bf16_tflops", "bf16_TFLOPs"))
    return (tf, "measured") if tf else (FALLBACK_BF16_TFLOPS, "fallback")


def prefill_flops(cached, q_lens, num_heads, head_dim) -> int:
    """4 * D * H * sum over query rows of the keys each row sees (Q.K^T and P.V)."""
    keys = sum(ql * c + ql * (ql + 1) // 2 for c, ql in zip(cached, q_lens))
    return 4 * head_dim * num_heads * keys


def profile_name(workload: str, window: int = 0) -> str:
    """The committed ncu summary of a workload's main kernel."""
    if W.WORKLOADS[workload]["kind"] == "prefill":
        return f"prefill_kernel_{workload}.md"
    win = f"window{window}_" if window > 0 else ""
    return f"decode_persistent_kernel_{win}{workload}.md"


def traffic_from_profile(kernel_file: str, workload: str, window: int = 0):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (the summary records the source's sha256)."""
    src = os.path.join(ROOT, "paged_kv_cache_186_gb300", "csrc", kernel_file)
    prof = os.path.join(ROOT, "profiles", profile_name(workload, window))
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        text = open(prof).read()
    except OSError:
        return None
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != sha:
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(gpu_index), "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self, t0: float, t1: float):
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0] or rows
        sm = sorted(r[1] for r in inside)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for name, v in zip(names, r[3][1:]):
                if v.strip().lower() in ("active", "0x1", "1"):
                    reasons.add(name)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "gpu" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif args.impl == "gpu":
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, x: float) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(world, x: float) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(name: str, max_seqs: int, seed: int = 0):
    """Host inputs for a bounded sample of a decode workload: the first
    `max_seqs` of its sequences (same lengths, shapes and value recipe, a pool
    just big enough for them)."""
    w = W.WORKLOADS[name]
    lens = W.workload_lengths(name)[:max_seqs]
    kw = {}
    if w.get("sinks"):
        kw["sinks"] = w["sinks"]
    h = W.make_decode(len(lens), w["num_heads"], w["num_kv_heads"], w["head_dim"],
                      w["block_size"], lens, seed=w["seed"] + 7 + seed, kv_dtype=w["kv_dtype"],
                      scale=w["scale"], **kw)
    return h, lens


def run_oracle_step(h, threads: int, window: int = 0, sinks: int = 0):
    import oracle
    if h.kv_dtype == "bf16":
        kc, vc = W.bf16_bits(h.k_cache).copy(), W.bf16_bits(h.v_cache).copy()
        t0 = time.perf_counter()
        oracle.store_kv(W.bf16_bits(h.k_new), W.bf16_bits(h.v_new), h.slot_mapping.numpy(), kc, vc)
        oracle.decode(W.bf16_bits(h.q), kc, vc, h.block_tables.numpy(), h.context_lens.numpy(),
                      h.scale, threads=threads, window=window, sinks=sinks)
        return time.perf_counter() - t0
    kc, vc = W.u8(h.k_cache).copy(), W.u8(h.v_cache).copy()
    ks, vs = h.k_scale.numpy().copy(), h.v_scale.numpy().copy()
    t0 = time.perf_counter()
    oracle.store_kv(W.u8(h.k_new), W.u8(h.v_new), h.slot_mapping.numpy(), kc, vc,
                    h.k_scale_new.numpy(), h.v_scale_new.numpy(), ks, vs)
    oracle.decode(W.bf16_bits(h.q), kc, vc, h.block_tables.numpy(), h.context_lens.numpy(),
                  h.scale, k_scale=ks, v_scale=vs, threads=threads, window=window, sinks=sinks)
    return time.perf_counter() - t0


def sample_size_for(name: str, budget_s: float, threads: int, window: int = 0,
                    sinks: int = 0) -> int:
    """Sequences per oracle step so one step takes about budget_s (estimated
    from a 1-sequence probe)."""
    h, lens = oracle_sample(name, 1)
    dt = max(run_oracle_step(h, threads, window, sinks), 1e-4)
    per_tok = dt / max(1, sum(visible_keys(L, window, sinks) for L in lens))
    all_lens = W.workload_lengths(name)
    n, acc = 0, 0.0
    for L in all_lens:
        cost = visible_keys(L, window, sinks) * per_tok
        if n > 0 and acc + cost > budget_s:
            break
        acc += cost
        n += 1
    return max(1, n)


def cpu_baseline(name: str, budget_s: float = 15.0, window: int = 0, sinks: int = 0,
                 one_core: bool = True):
    import oracle
    oracle.build()
    threads = len(os.sched_getaffinity(0))
    n = sample_size_for(name, budget_s, threads, window, sinks)
    h, lens = oracle_sample(name, n)
    dt = run_oracle_step(h, threads, window, sinks)
    keys = sum(visible_keys(L, window, sinks) for L in lens)
    total = len(W.workload_lengths(name))
    res = {"value": kv_bytes(name, lens, window, sinks) / dt / 1e9, "unit": "GB/s",
           "cores": threads, "kind": "oracle",
           "sample": f"first {n} of {total} sequences "
                     f"({keys} attended keys), one store_kv+decode, fp64 C oracle, {dt:.2f} s"}
    if one_core:
        # the same on one core, on its own bounded sample
        n1 = sample_size_for(name, budget_s / 3, 1, window, sinks)
        h1, lens1 = oracle_sample(name, n1)
        dt1 = run_oracle_step(h1, 1, window, sinks)
        res["value_1core"] = kv_bytes(name, lens1, window, sinks) / dt1 / 1e9
        res["sample_1core"] = f"first {n1} of {total} sequences, one core, {dt1:.2f} s"
    return res


def prefill_oracle_sample(name: str, max_seqs: int, seed: int = 0):
    """Host inputs of the first `max_seqs` sequences of a prefill workload
    (same cached and new lengths, shapes and value recipe)."""
    w = W.WORKLOADS[name]
    cached, qls = W.prefill_lengths(name)
    cached, qls = cached[:max_seqs], qls[:max_seqs]
    h = W.make_prefill(len(qls), w["num_heads"], w["num_kv_heads"], w["head_dim"],
                       w["block_size"], cached, qls, pool_factor=w["pool_factor"],
                       seed=w["seed"] + 7 + seed, scale=w["scale"])
    return h, cached, qls


def run_oracle_prefill_step(h, threads: int) -> float:
    import oracle
    kc, vc = W.bf16_bits(h.k_cache).copy(), W.bf16_bits(h.v_cache).copy()
    t0 = time.perf_counter()
    oracle.store_kv(W.bf16_bits(h.k_new), W.bf16_bits(h.v_new), h.slot_mapping.numpy(), kc, vc)
    oracle.prefill(W.bf16_bits(h.q), kc, vc, h.block_tables.numpy(), h.cu_seqlens_q.numpy(),
                   h.cu_seqlens_k.numpy(), h.scale, threads=threads)
    return time.perf_counter() - t0


def prefill_sample_size(name: str, budget_s: float, threads: int) -> int:
    """Sequences per oracle prefill step so one step takes about budget_s
    (estimated from a 1-sequence probe, by FLOPs)."""
    w = W.WORKLOADS[name]
    h, cached, qls = prefill_oracle_sample(name, 1)
    dt = max(run_oracle_prefill_step(h, threads), 1e-4)
    per_flop = dt / max(1, prefill_flops(cached, qls, w["num_heads"], w["head_dim"]))
    n, acc = 0, 0.0
    for c, q in zip(*W.prefill_lengths(name)):
        cost = prefill_flops([c], [q], w["num_heads"], w["head_dim"]) * per_flop
        if n > 0 and acc + cost > budget_s:
            break
        acc += cost
        n += 1
    return max(1, n)


def cpu_prefill_baseline(name: str, budget_s: float = 10.0):
    import oracle
    oracle.build()
    w = W.WORKLOADS[name]
    threads = len(os.sched_getaffinity(0))
    n = prefill_sample_size(name, budget_s, threads)
    h, cached, qls = prefill_oracle_sample(name, n)
    dt = run_oracle_prefill_step(h, threads)
    flops = prefill_flops(cached, qls, w["num_heads"], w["head_dim"])
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"first {n} of {w['batch']} sequences ({sum(qls)} query rows), one "
                      f"store_kv+prefill, fp64 C oracle, {dt:.2f} s"}


def copy_ceiling(dev) -> dict:
    """A plain device-to-device copy of 1 GiB (torch, not this library): the
    practical HBM ceiling on this machine beside the kernel's own figure. Read +
    write bytes over the median of 10 timed copies."""
    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8, device=dev)
    dst = torch.empty_like(src)
    src.fill_(1)
    for _ in range(3):
        dst.copy_(src)
    torch.cuda.synchronize()
    times = []
    for _ in range(10):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        dst.copy_(src)
        e.record()
        e.synchronize()
        times.append(s.elapsed_time(e))
    times.sort()
    gbs = 2 * n / (times[len(times) // 2] / 1e3) / 1e9
    del src, dst
    torch.cuda.empty_cache()
    return {"copy_gbs": gbs, "what": "torch device-to-device copy of 1 GiB, read+write bytes, "
                                     "median of 10"}


def run_reference(args, world, rank):
    name = args.workload
    if rank != 0:
        return
    import oracle
    oracle.build()
    threads = len(os.sched_getaffinity(0))
    budget = max(0.5, 120.0 / max(1, args.steps + args.warmup))
    win, snk = args.window, args.sinks
    n = sample_size_for(name, budget, threads, win, snk)
    h, lens = oracle_sample(name, n)
    for _ in range(args.warmup):
        run_oracle_step(h, threads, win, snk)
    t = 0.0
    for _ in range(args.steps):
        t += run_oracle_step(h, threads, win, snk)
    per_step = t / max(1, args.steps)
    bytes_step = kv_bytes(name, lens, win, snk)
    value = bytes_step / per_step / 1e9
    w = W.WORKLOADS[name]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "batch": n, "num_heads": w["num_heads"],
                   "num_kv_heads": w["num_kv_heads"], "head_dim": w["head_dim"],
                   "block_size": w["block_size"], "kv_dtype": w["kv_dtype"],
                   "sample_of_batch": f"{n}/{w['batch']}",
                   **({"window": win, "sinks": snk} if win > 0 else {})},
        "seq_steps_per_s": n / per_step,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"first {n} of {w['batch']} sequences per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_prefill(args, world, rank):
    """The oracle's prefill (fp64 C, all host cores) on a bounded sample of the
    varlen prefill workload: its first sequences."""
    name = args.workload
    if rank != 0:
        return
    import oracle
    oracle.build()
    threads = len(os.sched_getaffinity(0))
    budget = max(0.5, 120.0 / max(1, args.steps + args.warmup))
    n = prefill_sample_size(name, budget, threads)
    h, cached, qls = prefill_oracle_sample(name, n)
    for _ in range(args.warmup):
        run_oracle_prefill_step(h, threads)
    t = 0.0
    for _ in range(args.steps):
        t += run_oracle_prefill_step(h, threads)
    per_step = t / max(1, args.steps)
    w = W.WORKLOADS[name]
    flops = prefill_flops(cached, qls, w["num_heads"], w["head_dim"])
    value = flops / per_step / 1e12
    line = {
        "impl": "reference", "metric": "Varlen prefix-cached prefill attention TFLOP/s",
        "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": name, "batch": n, "num_heads": w["num_heads"],
                   "num_kv_heads": w["num_kv_heads"], "head_dim": w["head_dim"],
                   "block_size": w["block_size"], "q_lens": qls, "cached": cached,
                   "sample_of_batch": f"{n}/{w['batch']}"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"first {n} of {w['batch']} sequences per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
# The other configurations, measured in the default run beside the headline
# decode (each with its own oracle baseline and clock record): (key, workload,
# sliding window, sinks).
OTHER_WORKLOADS = (
    ("tiny_decode", "tiny_decode", 0, 0),
    ("long_context_decode_b8", "long_context_decode_b8", 0, 0),
    ("long_context_decode_b8_window4096_sinks4", "long_context_decode_b8", 4096, 4),
    ("llama3_70b_fp8_decode_b256", "llama3_70b_fp8_decode_b256", 0, 0),
    ("llama3_70b_int8_decode_b256", "llama3_70b_int8_decode_b256", 0, 0),
    ("varlen_prefill_b8", "varlen_prefill_b8", 0, 0),
)


class DecodeBench:
    """One decode workload on the device: rotating KV pools (so consecutive
    steps never find the KV in L2), the step as the library's user makes it,
    device-timed and end-to-end loops."""

    def __init__(self, pa, name, dev, rank=0, window=0, sinks=0, step_kind="append"):
        self.pa, self.name, self.dev = pa, name, dev
        self.w = w = W.WORKLOADS[name]
        self.lens = W.workload_lengths(name)
        self.B = w["batch"]
        self.window, self.sinks = window, sinks
        self.step_bytes = kv_bytes(name, self.lens, window, sinks)
        self.n_pools = max(2, min(4, math.ceil(4 * L2_BYTES / max(1, self.step_bytes)) + 1))
        self.pools = [W.make_workload(name, device=dev, variant=v + 97 * rank)
                      for v in range(self.n_pools)]
        self.q8 = w["kv_dtype"] in ("fp8", "int8")  # 8-bit codes with scales
        self.max_len = max(self.lens)
        p0 = self.pools[0]
        ws = pa.decode_workspace_size(p0.k_cache, self.B, w["num_heads"],
                                      p0.block_tables.shape[1], self.max_len,
                                      k_scale=p0.k_scale, v_scale=p0.v_scale)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
        self.out = torch.empty((self.B, w["num_heads"], w["head_dim"]), dtype=torch.bfloat16,
                               device=dev)
        self.stream = torch.cuda.current_stream()
        # the fused append (with or without a window): one persistent launch
        self.fused = step_kind == "append"
        # store_kv + decode (or the fused append: one persistent launch); the
        # grid-split path (batches above 16384) stores first and adds a merge
        self.launches_per_step = (1 if self.fused else 2) if self.B <= 16384 else 3

    def describe_step(self):
        if self.fused and self.window > 0:
            return (f"decode_window_append (store of the new tokens fused into the windowed "
                    f"decode; window {self.window}, sinks {self.sinks})")
        if self.fused:
            return "decode_append (store of the new tokens fused into decode)"
        if self.window > 0:
            return f"store_kv(new tokens) + decode_window(window {self.window}, sinks {self.sinks})"
        return "store_kv(new tokens) + decode"

    def run(self, p, inp=None, out=None, ev=None):
        """One step on pool p's cache; step inputs from `inp` (default: p)."""
        pa, x = self.pa, (p.__dict__ if inp is None else inp)
        out = self.out if out is None else out
        if self.fused:
            if ev is not None:
                ev[0].record(self.stream)
            pa.decode_window_append(x["q"], x["k_new"], x["v_new"], p.k_cache, p.v_cache,
                                    x["block_tables"], x["context_lens"], p.scale, self.window,
                                    self.sinks, max_context_len=self.max_len, out=out,
                                    workspace=self.workspace, k_scale_new=x.get("k_scale_new"),
                                    v_scale_new=x.get("v_scale_new"), k_scale=p.k_scale,
                                    v_scale=p.v_scale)
            if ev is not None:
                ev[1].record(self.stream)
            return
        pa.store_kv(x["k_new"], x["v_new"], x["slot_mapping"], p.k_cache, p.v_cache,
                    x.get("k_scale_new"), x.get("v_scale_new"), p.k_scale, p.v_scale)
        if ev is not None:
            ev[0].record(self.stream)
        pa.decode_window(x["q"], p.k_cache, p.v_cache, x["block_tables"], x["context_lens"],
                         p.scale, self.window, self.sinks, max_context_len=self.max_len, out=out,
                         workspace=self.workspace, k_scale=p.k_scale, v_scale=p.v_scale)
        if ev is not None:
            ev[1].record(self.stream)

    def warm(self, n):
        for i in range(n):
            self.run(self.pools[i % self.n_pools])
        torch.cuda.synchronize()
        if self.pa.get_device_error() != 0:
            raise RuntimeError(f"{self.name}: device error during warm-up")

    def time_device(self, steps, world=1):
        """Region events around `steps` steps (the fused step is one launch;
        otherwise the decode launch is also timed on its own). Returns
        (region ms, decode ms per step, wall start, wall end)."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.time()
        start.record(self.stream)
        for i in range(steps):
            # events between launches would add a gap to every fused step
            self.run(self.pools[i % self.n_pools], ev=None if self.fused else evs[i])
        end.record(self.stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
        ms_total = start.elapsed_time(end)
        if self.fused:
            dec_ms = ms_total / steps
        else:
            dec_ms = sum(a.elapsed_time(b) for a, b in evs) / steps
        err = self.pa.get_device_error()
        if err != 0:
            raise RuntimeError(f"{self.name}: device error word {err:#x} after the timed region")
        return ms_total, dec_ms, t0, t1

    def time_e2e(self, steps, warmup, world=1):
        """End to end through the public API with host buffers: each step
        uploads its inputs (q, new K/V rows, block tables, lengths; packed in
        one pinned staging buffer per pool: one copy) and downloads its
        output, over the same rotating pools as the device loop. Two device
        slots and an upload and a download stream let step i+1's upload and
        step i-1's download overlap step i's kernels; every step's own copies
        are inside the timed region. Returns (ms, h2d bytes, d2h bytes)."""
        dev, stream = self.dev, self.stream
        keys = ("q", "k_new", "v_new", "block_tables", "context_lens")
        if not self.fused:
            keys += ("slot_mapping",)
        if self.q8:
            keys += ("k_scale_new", "v_scale_new")
        p0 = self.pools[0]
        fields, off = [], 0
        for k in keys:
            t = getattr(p0, k)
            nbytes = t.numel() * t.element_size()
            fields.append((k, off, nbytes, t.dtype, tuple(t.shape)))
            off = (off + nbytes + 255) // 256 * 256
        h2d = off
        host = []
        for p in self.pools:
            buf = torch.empty(h2d, dtype=torch.uint8).pin_memory()
            for k, o, n, dt, shp in fields:
                buf[o:o + n].copy_(getattr(p, k).contiguous().cpu().view(-1).view(torch.uint8))
            host.append(buf)
        slots = [torch.empty(h2d, dtype=torch.uint8, device=dev) for _ in range(2)]
        views = [{k: sl[o:o + n].view(dt).view(shp) for k, o, n, dt, shp in fields}
                 for sl in slots]
        outs = [torch.empty_like(self.out) for _ in range(2)]
        out_host = [torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
                    for _ in range(2)]
        d2h = out_host[0].numel() * out_host[0].element_size()
        up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "used", "out")}

        def e2e_step(i):
            s, p = i % 2, self.pools[i % self.n_pools]
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(ev["used"][s])  # step i-2 finished reading slot s
                slots[s].copy_(host[i % self.n_pools], non_blocking=True)
                ev["in"][s].record(up)
            stream.wait_event(ev["in"][s])
            if i >= 2:
                stream.wait_event(ev["out"][s])  # step i-2's output has been downloaded
            self.run(p, inp=views[s], out=outs[s])
            ev["used"][s].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev["used"][s])
                out_host[s].copy_(outs[s], non_blocking=True)
                ev["out"][s].record(down)

        for i in range(max(3, warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e_start.record(stream)
        up.wait_event(e_start)
        for i in range(steps):
            e2e_step(i)
        e_end.record(down)  # after the last download
        torch.cuda.synchronize()
        barrier(world)
        return e_start.elapsed_time(e_end), h2d, d2h

    def time_graph(self, replays: int, steps_per_graph: int = 16):
        """Device time per step with the host out of the loop: steps_per_graph
        steps (cycling the pools) captured once in a CUDA graph, replayed
        back to back. Returns microseconds per step."""
        side = torch.cuda.Stream(device=self.dev)
        side.wait_stream(self.stream)
        with torch.cuda.stream(side):
            for i in range(self.n_pools):  # one-time host set-up before capture
                self.run(self.pools[i])
        self.stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(steps_per_graph):
                self.run(self.pools[i % self.n_pools])
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(self.stream)
        for _ in range(replays):
            g.replay()
        end.record(self.stream)
        torch.cuda.synchronize()
        if self.pa.get_device_error() != 0:
            raise RuntimeError(f"{self.name}: device error word set by the graph replays")
        return start.elapsed_time(end) * 1e3 / (replays * steps_per_graph)

    def config(self):
        w = self.w
        return {"workload": self.name, "batch": self.B, "num_heads": w["num_heads"],
                "num_kv_heads": w["num_kv_heads"], "head_dim": w["head_dim"],
                "block_size": w["block_size"], "kv_dtype": w["kv_dtype"],
                "context_len_mean": sum(self.lens) / len(self.lens),
                "context_len_max": self.max_len, "kv_bytes_per_step": self.step_bytes,
                **({"window": self.window, "sinks": self.sinks} if self.window > 0 else {}),
                "step": self.describe_step(),
                "l2": f"rotating {self.n_pools} KV pools, "
                      f"{self.n_pools * self.step_bytes / 1e9:.3f} GB of KV between reuses"
                      + (" > 129 MB L2" if self.n_pools * self.step_bytes > L2_BYTES
                         else " (fits in the 129 MB L2: launch-bound)")}

    def free(self):
        del self.pools, self.workspace, self.out
        torch.cuda.empty_cache()


def steps_for_wall(per_step_ms, target_s, lo, hi):
    """Steps that keep a timed region busy about target_s (for clock samples)."""
    n = int(target_s * 1e3 / max(per_step_ms, 1e-3))
    return max(lo, min(hi, n))


def other_decode_entry(pa, key, name, dev, args, window, sinks):
    b = DecodeBench(pa, name, dev, window=window, sinks=sinks, step_kind=args.step)
    b.warm(max(3, args.warmup))
    probe, _, _, _ = b.time_device(10)
    steps = steps_for_wall(probe / 10, 0.5, max(args.steps, 20), 20000)
    ms_total, dec_ms, t0, t1 = b.time_device(steps)
    e2e_ms, h2d, d2h = b.time_e2e(steps, args.warmup)
    peak, peak_kind = peaks()
    gbs = b.step_bytes / (ms_total / steps / 1e3) / 1e9
    achieved = b.step_bytes / (dec_ms / 1e3) / 1e9
    fits_l2 = b.n_pools * b.step_bytes <= L2_BYTES
    entry = {
        "kind": "decode", "steps": steps, "us_per_step": ms_total / steps * 1e3,
        "kv_gbs": gbs, "seq_steps_per_s": b.B * steps / (ms_total / 1e3),
        "roofline": ({"bound": "launch", "note": "KV of all pools fits in L2: launch-bound "
                      "latency, no HBM roofline fraction (graph_us_per_step: the same step "
                      "replayed from a CUDA graph)", "achieved": achieved, "unit": "GB/s"}
                     if fits_l2 else
                     {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                      "frac": achieved / peak, "peak_kind": f"of {peak_kind}",
                      "traffic": traffic_from_profile("pa_decode.cu", name, window),
                      "traffic_source": "profiles/" + profile_name(name, window),
                      "kernel": ("decode_persistent_kernel (pa_decode_append: region events / "
                                 "steps)" if b.fused else
                                 "decode_persistent_kernel (pa_decode_window: CUDA events per "
                                 "call)")}),
        "e2e": {"value": b.step_bytes * steps / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": b.launches_per_step * steps,
        "config": b.config(),
        "_wall": (t0, t1),
    }
    if fits_l2:
        # launch-bound: the same step captured in a CUDA graph and replayed
        # shows the device time without the per-call host marshalling
        entry["graph_us_per_step"] = b.time_graph(max(args.steps, 50))
    b.free()
    if not args.no_cpu_baseline:
        entry["cpu_baseline"] = cpu_baseline(name, budget_s=4.0, window=window, sinks=sinks,
                                             one_core=False)
    del key
    return entry


def run_gpu(args, world, rank, local):
    import paged_kv_cache_186_gb300 as pa
    from paged_kv_cache_186_gb300 import build as pabuild
    if rank == 0 or world == 1:
        pabuild.build()
    barrier(world)
    name = args.workload
    dev = torch.device("cuda", torch.cuda.current_device())
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        time.sleep(0.3)
    b = DecodeBench(pa, name, dev, rank=rank, window=args.window, sinks=args.sinks,
                    step_kind=args.step)
    b.warm(args.warmup)
    ms_total, dec_avg_ms, t_wall0, t_wall1 = b.time_device(args.steps, world)
    e2e_ms, h2d, d2h = b.time_e2e(args.steps, args.warmup, world)

    ms_total = max_over_ranks(world, ms_total)
    e2e_ms = max_over_ranks(world, e2e_ms)
    dec_avg_ms = max_over_ranks(world, dec_avg_ms)
    total_bytes = sum_over_ranks(world, float(b.step_bytes)) * args.steps
    value = total_bytes / (ms_total / 1e3) / 1e9
    e2e_value = total_bytes / (e2e_ms / 1e3) / 1e9
    step_bytes, B, w, fused = b.step_bytes, b.B, b.w, b.fused
    config = b.config()
    launches = b.launches_per_step * args.steps
    graph_us = (b.time_graph(max(args.steps, 50))
                if world == 1 and b.n_pools * b.step_bytes <= L2_BYTES else None)
    b.free()

    if rank != 0:
        return
    peak, peak_kind = peaks()
    achieved = step_bytes / (dec_avg_ms / 1e3) / 1e9
    traffic = traffic_from_profile("pa_decode.cu", name, args.window)
    config["parallelism"] = f"replicas x{world} (sequences sharded, no collective)"
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp8": "fp8_e4m3", "int8": "int8"}.get(w["kv_dtype"], "bf16"),
        "data": "synthetic",
        "config": config,
        "seq_steps_per_s": B * world * args.steps / (ms_total / 1e3),
        "us_per_step": ms_total / args.steps * 1e3,
        "hbm_frac_of_peak": value / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": ("pa_decode_append (decode_persistent_kernel, the only launch "
                                "of the timed region: region events / steps)" if fused else
                                "pa_decode (decode_persistent_kernel, CUDA events per call)"),
                     "traffic_source": "profiles/" + profile_name(name, args.window),
                     "peak_kind": f"of {peak_kind}"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": None,
    }
    if graph_us is not None:  # launch-bound: device time per step from a replayed graph
        line["graph_us_per_step"] = graph_us
    if world == 1:
        ceil = copy_ceiling(dev)
        ceil["kernel_frac_of_copy"] = achieved / ceil["copy_gbs"]
        line["ceiling"] = ceil
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(name, window=args.window, sinks=args.sinks)
    if world == 1 and not args.headline_only and name == DEFAULT_WORKLOAD and args.window <= 0:
        others = {}
        for key, wname, win, snk in OTHER_WORKLOADS:
            if W.WORKLOADS[wname]["kind"] == "prefill":
                others[key] = prefill_entry(pa, wname, dev, args)
            else:
                others[key] = other_decode_entry(pa, key, wname, dev, args, win, snk)
        line["workloads"] = others
    if sampler:
        time.sleep(0.3)
        sampler.stop()
        line["clocks"] = sampler.summary(t_wall0, t_wall1)
    for e in line.get("workloads", {}).values():
        wall = e.pop("_wall")
        e["clocks"] = sampler.summary(*wall) if sampler else None
    print(json.dumps(line), flush=True)


class PrefillBench:
    """The varlen prefill step: store_kv of the new tokens + pa_prefill_varlen,
    over rotating pools with an L2 flush between steps (the ~52 MB of K/V
    read per step fits in L2)."""

    def __init__(self, pa, name, dev, rank=0):
        self.pa, self.name, self.dev = pa, name, dev
        self.w = w = W.WORKLOADS[name]
        self.pools = [W.make_workload(name, device=dev, variant=v + 97 * rank) for v in range(3)]
        m = self.pools[0].meta
        self.m = m
        self.flops = prefill_flops(m["cached"], m["q_lens"], w["num_heads"], w["head_dim"])
        self.max_q = max(m["q_lens"])
        self.total_q = sum(m["q_lens"])
        self.out = torch.empty((self.total_q, w["num_heads"], w["head_dim"]),
                               dtype=torch.bfloat16, device=dev)
        self.flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
        self.stream = torch.cuda.current_stream()

    def run(self, p, ev=None):
        pa = self.pa
        pa.store_kv(p.k_new, p.v_new, p.slot_mapping, p.k_cache, p.v_cache)
        if ev is not None:
            ev[0].record(self.stream)
        pa.prefill_varlen(p.q, p.k_cache, p.v_cache, p.block_tables, p.cu_seqlens_q,
                          p.cu_seqlens_k, p.scale, max_q_len=self.max_q, out=self.out)
        if ev is not None:
            ev[1].record(self.stream)

    def time(self, steps, warmup, world=1):
        for i in range(warmup):
            self.run(self.pools[i % 3])
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.time()
        for i in range(steps):
            self.flush.zero_()  # outside the timed events: write > L2 between steps
            evs[i][0].record(self.stream)
            self.run(self.pools[i % 3], ev=pev[i])
            evs[i][1].record(self.stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
        if self.pa.get_device_error() != 0:
            raise RuntimeError("device error word set after the timed region")
        step_ms = sum(a.elapsed_time(b) for a, b in evs) / steps
        pre_ms = sum(a.elapsed_time(b) for a, b in pev) / steps
        return step_ms, pre_ms, t0, t1

    def config(self):
        w, m = self.w, self.m
        return {"workload": self.name, "batch": w["batch"], "num_heads": w["num_heads"],
                "num_kv_heads": w["num_kv_heads"], "head_dim": w["head_dim"],
                "block_size": w["block_size"], "q_lens": m["q_lens"], "cached": m["cached"],
                "total_q": self.total_q, "flops_per_step": self.flops,
                "step": "store_kv(new tokens) + prefill_varlen",
                "l2": "256 MB buffer written between timed steps (outside the events)"}

    def free(self):
        del self.pools, self.out, self.flush
        torch.cuda.empty_cache()


def prefill_entry(pa, name, dev, args):
    b = PrefillBench(pa, name, dev)
    steps = max(args.steps, 50)
    step_ms, pre_ms, t0, t1 = b.time(steps, max(3, args.warmup))
    peak, kind = tensor_peak()
    achieved = b.flops / (pre_ms / 1e3) / 1e12
    entry = {
        "kind": "prefill", "steps": steps, "us_per_step": step_ms * 1e3,
        "prefill_us": pre_ms * 1e3, "tflops": b.flops / (step_ms / 1e3) / 1e12,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "peak_kind": f"of {kind} (bf16 dense, burst)",
                     "traffic": traffic_from_profile("pa_prefill.cu", name),
                     "traffic_source": "profiles/" + profile_name(name),
                     "kernel": "prefill_kernel (CUDA events per call)"},
        "gpu_launches": 2 * steps,
        "config": b.config(),
        "_wall": (t0, t1),
    }
    b.free()
    if not args.no_cpu_baseline:
        entry["cpu_baseline"] = cpu_prefill_baseline(name, budget_s=4.0)
    return entry


def run_prefill(args, world, rank, local):
    """Varlen prefill step: store_kv of the new tokens + pa_prefill_varlen."""
    import paged_kv_cache_186_gb300 as pa
    from paged_kv_cache_186_gb300 import build as pabuild
    if rank == 0 or world == 1:
        pabuild.build()
    barrier(world)
    dev = torch.device("cuda", torch.cuda.current_device())
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        time.sleep(0.3)
    b = PrefillBench(pa, args.workload, dev, rank=rank)
    step_ms, pre_ms, t_wall0, t_wall1 = b.time(args.steps, args.warmup, world)
    step_ms = max_over_ranks(world, step_ms)
    pre_ms = max_over_ranks(world, pre_ms)
    total_flops = sum_over_ranks(world, float(b.flops))
    flops, config = b.flops, b.config()
    b.free()
    if sampler:
        time.sleep(0.3)
        sampler.stop()
    if rank != 0:
        return
    peak, kind = tensor_peak()
    achieved = flops / (pre_ms / 1e3) / 1e12
    line = {
        "metric": "Varlen prefix-cached prefill attention TFLOP/s", "value":
            total_flops / (step_ms / 1e3) / 1e12, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "traffic": traffic_from_profile("pa_prefill.cu", args.workload),
                     "traffic_source": "profiles/" + profile_name(args.workload),
                     "kernel": "prefill_kernel (CUDA events per call)",
                     "peak_kind": f"of {kind} (bf16 dense)"},
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(t_wall0, t_wall1) if sampler else None,
    }
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_prefill_baseline(args.workload)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other workloads measured beside the headline decode")
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window in keys (pa_decode_window); 0 = all keys")
    ap.add_argument("--sinks", type=int, default=0, help="leading keys kept with --window")
    ap.add_argument("--step", choices=["append", "separate"], default="append",
                    help="decode step: fused pa_decode_append, or pa_store_kv + pa_decode")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup(args)
    try:
        if W.WORKLOADS[args.workload]["kind"] == "prefill":
            if args.impl == "reference":
                run_reference_prefill(args, world, rank)
            else:
                run_prefill(args, world, rank, local)
        elif args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_gpu(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
