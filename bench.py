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
events inside the timed region for the roofline figure.

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


def traffic_from_profile(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (the summary records the source's sha256)."""
    src = os.path.join(ROOT, "paged_kv_cache_186_gb300", "csrc", kernel_file)
    prof = os.path.join(ROOT, "profiles", f"decode_persistent_kernel_{workload}.md")
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


def cpu_baseline(name: str, budget_s: float = 15.0, window: int = 0, sinks: int = 0):
    import oracle
    oracle.build()
    threads = len(os.sched_getaffinity(0))
    n = sample_size_for(name, budget_s, threads, window, sinks)
    h, lens = oracle_sample(name, n)
    dt = run_oracle_step(h, threads, window, sinks)
    keys = sum(visible_keys(L, window, sinks) for L in lens)
    # the same on one core, on its own bounded sample
    n1 = sample_size_for(name, budget_s / 3, 1, window, sinks)
    h1, lens1 = oracle_sample(name, n1)
    dt1 = run_oracle_step(h1, 1, window, sinks)
    total = len(W.workload_lengths(name))
    return {"value": kv_bytes(name, lens, window, sinks) / dt / 1e9, "unit": "GB/s",
            "cores": threads, "kind": "oracle",
            "sample": f"first {n} of {total} sequences "
                      f"({keys} attended keys), one store_kv+decode, fp64 C oracle, {dt:.2f} s",
            "value_1core": kv_bytes(name, lens1, window, sinks) / dt1 / 1e9,
            "sample_1core": f"first {n1} of {total} sequences, one core, {dt1:.2f} s"}


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


# ------------------------------------------------------------------ GPU arm
def run_gpu(args, world, rank, local):
    import paged_kv_cache_186_gb300 as pa
    from paged_kv_cache_186_gb300 import build as pabuild
    if rank == 0 or world == 1:
        pabuild.build()
    barrier(world)
    name = args.workload
    w = W.WORKLOADS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    lens = W.workload_lengths(name)
    B = w["batch"]
    win, snk = args.window, args.sinks
    step_bytes = kv_bytes(name, lens, win, snk)
    pool_bytes = step_bytes
    n_pools = max(2, min(4, math.ceil(4 * L2_BYTES / max(1, pool_bytes)) + 1))
    pools = [W.make_workload(name, device=dev, variant=v + 97 * rank) for v in range(n_pools)]
    q8 = w["kv_dtype"] in ("fp8", "int8")  # 8-bit codes with scales
    max_len = max(lens)
    ws_bytes = pa.decode_workspace_size(pools[0].k_cache, B, w["num_heads"],
                                        pools[0].block_tables.shape[1], max_len,
                                        k_scale=pools[0].k_scale, v_scale=pools[0].v_scale)
    workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    out = torch.empty((B, w["num_heads"], w["head_dim"]), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    fused = args.step == "append" and win <= 0  # the fused append has no window variant

    def step(p, ev=None):
        if fused:
            if ev is not None:
                ev[0].record(stream)
            pa.decode_append(p.q, p.k_new, p.v_new, p.k_cache, p.v_cache, p.block_tables,
                             p.context_lens, p.scale, max_context_len=max_len, out=out,
                             workspace=workspace, k_scale_new=p.k_scale_new,
                             v_scale_new=p.v_scale_new, k_scale=p.k_scale, v_scale=p.v_scale)
            if ev is not None:
                ev[1].record(stream)
            return
        pa.store_kv(p.k_new, p.v_new, p.slot_mapping, p.k_cache, p.v_cache, p.k_scale_new,
                    p.v_scale_new, p.k_scale, p.v_scale)
        if ev is not None:
            ev[0].record(stream)
        pa.decode_window(p.q, p.k_cache, p.v_cache, p.block_tables, p.context_lens, p.scale,
                         win, snk, max_context_len=max_len, out=out, workspace=workspace,
                         k_scale=p.k_scale, v_scale=p.v_scale)
        if ev is not None:
            ev[1].record(stream)

    for i in range(args.warmup):
        step(pools[i % n_pools])
    torch.cuda.synchronize()
    if pa.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        # the fused step is a single launch: the region's own events time it
        # (events between launches would add a gap to every step)
        step(pools[i % n_pools], None if fused else evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    if sampler:
        time.sleep(0.3)
        sampler.stop()
    ms_total = start.elapsed_time(end)
    if fused:
        dec_avg_ms = ms_total / args.steps
    else:
        dec_ms = [a.elapsed_time(b) for a, b in evs]
        dec_avg_ms = sum(dec_ms) / len(dec_ms)
    err = pa.get_device_error()
    if err != 0:
        raise RuntimeError(f"device error word {err:#x} after the timed region")

    # ---------------- end to end through the public API with host buffers
    # Each step uploads its inputs from pinned host memory (packed into one
    # staging buffer: one copy) and downloads its output. Two device slots and
    # an upload and a download stream let step i+1's upload and step i-1's
    # download overlap step i's kernel; every step's own copies are inside the
    # timed region.
    p0 = pools[0]
    host_keys = ("q", "k_new", "v_new", "block_tables", "context_lens")
    if not fused:
        host_keys += ("slot_mapping",)
    if q8:
        host_keys += ("k_scale_new", "v_scale_new")
    fields, off = [], 0
    for k in host_keys:
        t = getattr(p0, k).contiguous()
        nbytes = t.numel() * t.element_size()
        fields.append((k, off, nbytes, t.dtype, tuple(t.shape)))
        off = (off + nbytes + 255) // 256 * 256
    h2d = off
    host_buf = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    for k, o, n, dt, shp in fields:
        host_buf[o:o + n].copy_(getattr(p0, k).contiguous().cpu().view(-1).view(torch.uint8))
    slots = [torch.empty(h2d, dtype=torch.uint8, device=dev) for _ in range(2)]
    views = [{k: sl[o:o + n].view(dt).view(shp) for k, o, n, dt, shp in fields} for sl in slots]
    outs = [torch.empty_like(out) for _ in range(2)]
    out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    d2h = out_host[0].numel() * out_host[0].element_size()
    up_stream, down_stream = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "used", "done", "out")}

    def e2e_step(i, p):
        s, v = i % 2, views[i % 2]
        with torch.cuda.stream(up_stream):
            if i >= 2:
                up_stream.wait_event(ev["used"][s])  # step i-2 finished reading slot s
            slots[s].copy_(host_buf, non_blocking=True)
            ev["in"][s].record(up_stream)
        stream.wait_event(ev["in"][s])
        if i >= 2:
            stream.wait_event(ev["out"][s])  # step i-2's output has been downloaded
        if fused:
            pa.decode_append(v["q"], v["k_new"], v["v_new"], p.k_cache, p.v_cache,
                             v["block_tables"], v["context_lens"], p.scale,
                             max_context_len=max_len, out=outs[s], workspace=workspace,
                             k_scale_new=v.get("k_scale_new"), v_scale_new=v.get("v_scale_new"),
                             k_scale=p.k_scale, v_scale=p.v_scale)
        else:
            pa.store_kv(v["k_new"], v["v_new"], v["slot_mapping"], p.k_cache, p.v_cache,
                        v.get("k_scale_new"), v.get("v_scale_new"), p.k_scale, p.v_scale)
            pa.decode_window(v["q"], p.k_cache, p.v_cache, v["block_tables"], v["context_lens"],
                             p.scale, win, snk, max_context_len=max_len, out=outs[s],
                             workspace=workspace, k_scale=p.k_scale, v_scale=p.v_scale)
        ev["used"][s].record(stream)
        ev["done"][s].record(stream)
        with torch.cuda.stream(down_stream):
            down_stream.wait_event(ev["done"][s])
            out_host[s].copy_(outs[s], non_blocking=True)
            ev["out"][s].record(down_stream)

    for i in range(max(3, args.warmup)):
        e2e_step(i, p0)
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e_start.record(stream)
    up_stream.wait_event(e_start)
    for i in range(args.steps):
        e2e_step(i, p0)  # same pool: the KV cache is resident state, only step inputs move
    e_end.record(down_stream)  # after the last download
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = e_start.elapsed_time(e_end)

    ms_total = max_over_ranks(world, ms_total)
    e2e_ms = max_over_ranks(world, e2e_ms)
    dec_avg_ms = max_over_ranks(world, dec_avg_ms)
    total_bytes = sum_over_ranks(world, float(step_bytes)) * args.steps
    value = total_bytes / (ms_total / 1e3) / 1e9
    e2e_value = total_bytes / (e2e_ms / 1e3) / 1e9

    if rank != 0:
        return
    peak, peak_kind = peaks()
    achieved = step_bytes / (dec_avg_ms / 1e3) / 1e9
    traffic = traffic_from_profile("pa_decode.cu", name) if win <= 0 else None
    # store_kv + decode (or the fused append: one persistent launch); the
    # grid-split path (batches above 2048) adds a merge
    n_launch = (1 if fused else 2) if B <= 2048 else 3
    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp8": "fp8_e4m3", "int8": "int8"}.get(w["kv_dtype"], "bf16"),
        "data": "synthetic",
        "config": {"workload": name, "batch": B, "num_heads": w["num_heads"],
                   "num_kv_heads": w["num_kv_heads"], "head_dim": w["head_dim"],
                   "block_size": w["block_size"], "kv_dtype": w["kv_dtype"],
                   "context_len_mean": sum(lens) / len(lens), "context_len_max": max_len,
                   "kv_bytes_per_step": step_bytes,
                   **({"window": win, "sinks": snk} if win > 0 else {}),
                   "step": ("decode_append (store of the new tokens fused into decode)"
                            if fused else "store_kv(new tokens) + decode"),
                   "l2": f"rotating {n_pools} KV pools, {n_pools * step_bytes / 1e9:.2f} GB of KV "
                         f"between reuses > 129 MB L2",
                   "parallelism": f"replicas x{world} (sequences sharded, no collective)"},
        "seq_steps_per_s": B * world * args.steps / (ms_total / 1e3),
        "us_per_step": ms_total / args.steps * 1e3,
        "hbm_frac_of_peak": value / peak,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": ("pa_decode_append (decode_persistent_kernel, the only launch "
                                "of the timed region: region events / steps)" if fused else
                                "pa_decode (decode_persistent_kernel, CUDA events per call)"),
                     "traffic_source": "profiles/decode_persistent_kernel_" + name + ".md",
                     "peak_kind": f"of {peak_kind}"},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": n_launch * args.steps,
        "clocks": clocks,
    }
    if world == 1:
        ceil = copy_ceiling(dev)
        ceil["kernel_frac_of_copy"] = achieved / ceil["copy_gbs"]
        line["ceiling"] = ceil
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(name, window=win, sinks=snk)
    print(json.dumps(line), flush=True)


def run_prefill(args, world, rank, local):
    """Varlen prefill step: store_kv of the new tokens + pa_prefill_varlen."""
    import paged_kv_cache_186_gb300 as pa
    from paged_kv_cache_186_gb300 import build as pabuild
    if rank == 0 or world == 1:
        pabuild.build()
    barrier(world)
    name = args.workload
    w = W.WORKLOADS[name]
    dev = torch.device("cuda", torch.cuda.current_device())
    pools = [W.make_workload(name, device=dev, variant=v + 97 * rank) for v in range(3)]
    m = pools[0].meta
    flops = prefill_flops(m["cached"], m["q_lens"], w["num_heads"], w["head_dim"])
    max_q = max(m["q_lens"])
    total_q = sum(m["q_lens"])
    out = torch.empty((total_q, w["num_heads"], w["head_dim"]), dtype=torch.bfloat16, device=dev)
    # L2 flush buffer: the K/V of one step (~52 MB) fits in L2, so flush between steps
    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step(p):
        pa.store_kv(p.k_new, p.v_new, p.slot_mapping, p.k_cache, p.v_cache)
        pa.prefill_varlen(p.q, p.k_cache, p.v_cache, p.block_tables, p.cu_seqlens_q,
                          p.cu_seqlens_k, p.scale, max_q_len=max_q, out=out)

    for i in range(args.warmup):
        step(pools[i % 3])
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(args.steps):
        flush.zero_()  # outside the timed events: write > L2 between steps
        p = pools[i % 3]
        evs[i][0].record(stream)
        pa.store_kv(p.k_new, p.v_new, p.slot_mapping, p.k_cache, p.v_cache)
        pev[i][0].record(stream)
        pa.prefill_varlen(p.q, p.k_cache, p.v_cache, p.block_tables, p.cu_seqlens_q,
                          p.cu_seqlens_k, p.scale, max_q_len=max_q, out=out)
        pev[i][1].record(stream)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    barrier(world)
    if sampler:
        time.sleep(0.3)
        sampler.stop()
    if pa.get_device_error() != 0:
        raise RuntimeError("device error word set after the timed region")
    step_ms = sum(a.elapsed_time(b) for a, b in evs) / args.steps
    pre_ms = sum(a.elapsed_time(b) for a, b in pev) / args.steps
    step_ms = max_over_ranks(world, step_ms)
    pre_ms = max_over_ranks(world, pre_ms)
    total_flops = sum_over_ranks(world, float(flops))
    if rank != 0:
        return
    peak, kind = tensor_peak()
    achieved = flops / (pre_ms / 1e3) / 1e12
    line = {
        "metric": "Varlen prefix-cached prefill attention TFLOP/s", "value":
            total_flops / (step_ms / 1e3) / 1e12, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": name, "batch": w["batch"], "num_heads": w["num_heads"],
                   "num_kv_heads": w["num_kv_heads"], "head_dim": w["head_dim"],
                   "block_size": w["block_size"], "q_lens": m["q_lens"], "cached": m["cached"],
                   "total_q": total_q, "flops_per_step": flops,
                   "step": "store_kv(new tokens) + prefill_varlen",
                   "l2": "256 MB buffer written between timed steps (outside the events)"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "prefill_kernel (CUDA events per call)",
                     "peak_kind": f"of {kind} (bf16 dense)"},
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(t_wall0, t_wall1) if sampler else None,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
                print(json.dumps({"impl": "reference", "unavailable":
                                  "the reference arm times the decode workloads only"}))
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
