"""Benchmark of the attention forward on GB300: one JSON line on stdout (rank 0).

Default workload: LLM prefill, B=4, H=32, N=4096, d=128, causal, fp16 (the headline
metric: attention-forward TFLOP/s against the dense fp16 tensor peak). A step is one
forward over the whole batch with inputs resident in HBM. The same line carries:
  e2e          the same metric through the public API with host tensors (pinned host ->
               device copies of Q, K, V and the device -> host copy of O inside the timing)
  short_n      the reranking workload (B=50, H=12, N=256, d=32, key padding) in GB/s of
               minimum traffic, inputs rotated over buffer sets larger than L2
  split_kv     one long causal head, the tiled kernel alone and with split-KV
  variants     the long (N=32768) and stress (d=64, peaked rows) workloads, grouped-query
               prefill (32 query heads over 8 key/value heads), a block of 1024 queries over
               16384 cached keys and the prefill shape in bf16 in TFLOP/s; decoding, a block of
               draft queries and fp32 reranking in GB/s
  roofline     the dominant kernel's achieved FLOP/s against the measured peak
  cpu_baseline the fp64 oracle timed on the host cores on a bounded sample (rank 0, N=1)
  clocks       SM clocks and throttle reasons sampled during the timed region

--impl reference times the oracle itself (the reference arm: a CPU program) on the same
workload, metric and unit.

Multi-GPU (torchrun, one rank per GPU): every rank runs its own copy of the workload
(independent (batch, head) problems, no collective on the data path); the time is the
max over ranks and the value counts the work of all ranks (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_scaled_dot_attn_gb300 import synth  # noqa: E402

METRIC = "attn fwd TFLOPS & % of GB300 fp16 dense peak (N=4096,d=128,causal); GB/s short-N"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--path", default="auto", choices=["auto", "warp_mma", "tcgen05", "short", "naive", "splitkv"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-short-n", action="store_true")
    ap.add_argument("--no-split-kv", action="store_true")
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-naive", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(value: float, device=None) -> float:
    """The largest of `value` over all ranks (the value itself in a single process).

    With one process per GPU the slowest rank sets the time of a step; the collective is
    only for timing, never on the data path.
    """
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(world: int, work_per_rank: float, seconds: float, unit_scale: float = 1e12):
    """Whole-job throughput: every rank processes its own copy of the workload, so the
    work of all ranks is divided by the slowest rank's time."""
    return world * work_per_rank / seconds / unit_scale


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling (every 200 ms) of SM clocks and throttle reasons."""

    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 10:
                continue
            if self.uuid and self.uuid not in parts[1] and parts[1] not in self.uuid:
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- CPU arm
def oracle_sample(w, q, k, v, kl, heads):
    """Times the oracle on every row of the given flat (batch*head) heads; returns
    (flops, seconds, threads used)."""
    import numpy as np

    import oracle
    rows = np.concatenate([np.arange(h * w.N, (h + 1) * w.N) for h in heads]).astype(np.int64)
    t0 = time.perf_counter()
    oracle.attn(q, k, v, sm_scale=w.sm_scale, causal=w.causal, key_lengths=kl, rows=rows,
                dtype=w.dtype)
    dt = time.perf_counter() - t0
    flops = synth.attention_flops_ex(1, len(heads), w.N, w.N_k, w.d, w.causal)
    return flops, dt, oracle.default_threads()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = synth.WORKLOADS[args.workload]
    q, k, v, kl = synth.draw_workload(w)
    oracle.build()
    steps, warmup = max(1, args.steps), max(3, args.warmup)
    # Each step: every row of one (batch 0) head, sized so the whole run stays within minutes.
    n_heads = 1
    per_step = []
    for s in range(warmup + steps):
        h = s % w.H
        flops, dt, cores = oracle_sample(w, q, k, v, kl, [h])
        if s >= warmup:
            per_step.append((flops, dt))
        if s >= warmup + 1 and sum(t for _, t in per_step) > 120:
            break  # the oracle is slow by design; keep the arm bounded
    total_f = sum(f for f, _ in per_step)
    total_t = sum(t for _, t in per_step)
    value = total_f / total_t / 1e12
    sample = (f"{len(per_step)} steps x {n_heads} head(s) of batch 0, all {w.N} rows each "
              f"({w.describe()})")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": len(per_step), "warmup": warmup, "ms_per_step": total_t / len(per_step) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w):
    cfg = {"workload": w.describe(), "B": w.B, "H": w.H, "N": w.N, "d": w.d,
           "causal": w.causal, "sm_scale": w.sm_scale,
           "key_lengths": list(w.key_len_range) if w.key_len_range else None,
           "l2": "inputs larger than L2"
           if synth.min_bytes_ex(w.B, w.H, w.H_kv, w.N, w.N_k, w.d) > 2 * 129e6
           else "L2 flushed between timed launches"}
    if (w.H_kv, w.N_k) != (w.H, w.N):
        cfg.update(H_kv=w.H_kv, N_k=w.N_k)
    return cfg


# ----------------------------------------------------------------------------- GPU arm
def source_digest(files):
    """First 16 hex digits of the sha256 of the listed source files, concatenated."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profile(kernel_name: str, workload: str):
    """Per-launch DRAM bytes from the committed ncu summary, if it still matches the source.

    profiles/<kernel>_<workload>_traffic.txt records the DRAM read + write bytes of one launch
    and a digest of the kernel's source files; a kernel changed since the capture gives None.
    """
    path = os.path.join(ROOT, "profiles", f"{kernel_name}_{workload}_traffic.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and not line.startswith("#"):
            key, val = line.split(":", 1)
            vals[key.strip()] = val.strip()
    files = [f.strip() for f in vals.get("source_files", "").split(",") if f.strip()]
    if not files or not all(os.path.exists(os.path.join(ROOT, f)) for f in files):
        return None
    if source_digest(files) != vals.get("source_sha256_16"):
        return None  # the kernel changed since the counters were taken
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def l2_flush_buffer(torch):
    return torch.empty(512 * 1024 * 1024 // 4, dtype=torch.int32, device="cuda")


def time_launches(torch, fn, n, flush=None):
    """Per-launch CUDA-event durations (ms) on the current stream."""
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a, b in evs:
        if flush is not None:
            flush.fill_(1)
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    import numpy as np
    import torch
    import torch.distributed as dist

    from exact_scaled_dot_attn_gb300 import api, build

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    build.build()
    peaks, peak_src = load_peaks()
    w = synth.WORKLOADS[args.workload]
    steps, warmup = max(1, args.steps), max(3, args.warmup)

    q, k, v, kl = synth.draw_workload(w)
    qd, kd, vd = (to_device(torch, x, w.dtype) for x in (q, k, v))
    kld = torch.from_numpy(kl).cuda() if kl is not None else None
    od = torch.empty_like(qd)
    flops = synth.attention_flops_ex(w.B, w.H, w.N, w.N_k, w.d, w.causal)

    naive_ws = None
    if args.path == "naive":
        naive_ws = torch.empty(api.naive_workspace_bytes(w.B, w.H, w.N), dtype=torch.uint8,
                               device="cuda")

    def step():
        if naive_ws is not None:
            api.fwd_naive(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, key_lengths=kld,
                          out=od, workspace=naive_ws)
            return
        if args.path == "splitkv":
            # split-KV with the automatic split count (the kernel plus the merge kernel)
            api.fwd_splitkv(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, key_lengths=kld, out=od)
            return
        api.fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, key_lengths=kld, out=od,
                path=args.path)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(local_rank).uuid)
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)  # let the sampler take its first reading under load
    for _ in range(max(3, warmup)):
        step()
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for a, b in evs:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    region_ms = evs[0][0].elapsed_time(evs[-1][1])
    launch_ms = [a.elapsed_time(b) for a, b in evs]
    region_ms = max_over_ranks(region_ms, device="cuda")
    ms_per_step = region_ms / steps
    value = weak_scaling_value(world, flops, ms_per_step * 1e-3)

    del naive_ws
    # End to end through the public API with host tensors.
    e2e_steps = max(1, min(args.e2e_steps, steps))
    tq, tk, tv = (to_host(torch, x, w.dtype).pin_memory() for x in (q, k, v))
    tkl = torch.from_numpy(kl) if kl is not None else None
    o_host = torch.empty(q.shape, dtype=tq.dtype, pin_memory=True)
    e2e_path = "auto" if args.path in ("naive", "splitkv") else args.path  # (the host-tensor API is fused only)
    for _ in range(2):
        api.fwd(tq, tk, tv, causal=w.causal, sm_scale=w.sm_scale, key_lengths=tkl, out=o_host,
                path=e2e_path)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        api.fwd(tq, tk, tv, causal=w.causal, sm_scale=w.sm_scale, key_lengths=tkl, out=o_host,
                path=e2e_path)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, device="cuda")
    h2d = sum(x.nbytes for x in (q, k, v)) + (kl.nbytes if kl is not None else 0)
    d2h = q.nbytes

    # Roofline of the dominant (only) kernel.
    kernel_name = "tcgen05" if args.path == "splitkv" else args.path
    if args.path == "auto":
        kernel_name = api.auto_path_ex(w.H, w.H_kv, w.N, w.N_k, w.d, w.dtype, w.causal)
    avg_launch_ms = statistics.mean(launch_ms)
    achieved = flops / (avg_launch_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic_from_profile(kernel_name, w.name),
                "kernel": kernel_name, "peak_source": f"{peak_src} bf16 dense burst (fp16 rate = bf16 rate)",
                "avg_launch_ms": avg_launch_ms}
    if args.path == "naive":
        # the three passes are bound by the traffic of the materialised S and P
        gbs = naive_model_bytes(w) / (avg_launch_ms * 1e-3) / 1e9
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                    "traffic": traffic_from_profile("naive", w.name), "kernel": "naive (three passes)",
                    "peak_source": f"{peak_src} copy bandwidth", "avg_launch_ms": avg_launch_ms}
    if args.path == "splitkv" or kernel_name == "decode":
        # few query rows over many keys: bound by reading K and V
        min_bytes = sum(x.nbytes for x in (q, k, v)) + q.nbytes
        gbs = min_bytes / (avg_launch_ms * 1e-3) / 1e9
        hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        split = args.path == "splitkv"
        roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                    "traffic": traffic_from_profile("tcgen05_splitkv" if split else "decode", w.name),
                    "kernel": "tcgen05 split-KV and merge" if split else "decode",
                    "peak_source": f"{peak_src} copy bandwidth", "avg_launch_ms": avg_launch_ms}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
        "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": dict(workload_config(w), path=args.path, kernel=kernel_name),
        "e2e": {"value": weak_scaling_value(world, flops, e2e_s), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": steps * {"naive": 3, "splitkv": 2}.get(args.path, 1),
        "roofline": roofline,
        "clocks": clocks,
    }

    if not args.no_short_n:
        line["short_n"] = short_n(torch, api, peaks, peak_src)
    if not args.no_split_kv:
        line["split_kv"] = split_kv(torch, api, peaks, peak_src)
    if not args.no_variants:
        line["variants"] = variants(torch, api, peaks, peak_src)
    if not args.no_naive:
        line["naive"] = naive_lines(torch, api, peaks, peak_src)

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # Bounded sample of the same workload: the first heads (flat batch*head order), all
        # rows each, as many as take about 10-20 s of host time.
        n_heads = max(1, min(w.B * w.H, int(os.environ.get("ATTN_CPU_BASELINE_HEADS", w.B * w.H))))
        f, dt, cores = oracle_sample(w, q, k, v, kl, list(range(n_heads)))
        line["cpu_baseline"] = {"value": f / dt / 1e12, "unit": UNIT, "cores": cores,
                                "kind": "oracle",
                                "sample": f"heads 0..{n_heads - 1} of {w.B * w.H} (flat batch*head),"
                                          f" all {w.N} rows each, {dt:.1f} s of host time"}
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def short_n(torch, api, peaks, peak_src):
    """Reranking workload in GB/s of minimum traffic (Q, K, V, O once at full padded size).

    Inputs larger than L2: the launches rotate over buffer sets whose total is more than
    twice the L2 size, so every launch reads its inputs from HBM. The launches run back to
    back from a CUDA graph (as a serving loop would issue them), timed with CUDA events
    around the replays; the per-launch time is the total over the launch count. A single
    launch right after a 512 MiB write (L2 flushed, launch latency included) is reported
    beside it.
    """
    import math
    w = synth.WORKLOADS["rerank"]
    q, k, v, kl = synth.draw_workload(w)
    nbytes = synth.min_bytes(w.B, w.H, w.N, w.d) + kl.nbytes
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    nsets = max(2, math.ceil(2 * l2 / nbytes) + 1)
    sets = []
    for _ in range(nsets):
        qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, v))
        sets.append((qd, kd, vd, torch.from_numpy(kl).cuda(), torch.empty_like(qd)))

    def fn(i):
        qd, kd, vd, kld, od = sets[i % nsets]
        api.fwd(qd, kd, vd, causal=False, sm_scale=w.sm_scale, key_lengths=kld, out=od)

    for i in range(2 * nsets):
        fn(i)
    torch.cuda.synchronize()
    per_graph = 4 * nsets
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(per_graph):
                fn(i)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    reps = 10
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    launch_ms = a.elapsed_time(b) / (reps * per_graph)
    gbs = nbytes / (launch_ms * 1e-3) / 1e9
    flush = l2_flush_buffer(torch)
    time_launches(torch, lambda: fn(0), 3, flush)
    flushed_ms = statistics.median(time_launches(torch, lambda: fn(0), 30, flush))
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    valid_bytes = int(sum(int(L) for L in kl) * w.H * w.d * 2 * 2 + q.nbytes * 2)
    kernel = api.auto_path(w.N, w.d)
    return {"workload": w.describe(), "value": gbs, "unit": "GB/s", "launch_ms": launch_ms,
            "bytes": nbytes, "valid_only_bytes": valid_bytes, "kernel": kernel,
            "gpu_launches": reps * per_graph,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                         "frac": gbs / peak, "peak_source": f"{peak_src} copy bandwidth",
                         "traffic": traffic_from_profile(kernel, "rerank")},
            "l2": f"inputs larger than L2: {nsets} rotating buffer sets ({nsets * nbytes / 1e6:.0f} MB)",
            "flushed_single_launch": {"ms": flushed_ms,
                                      "value": nbytes / (flushed_ms * 1e-3) / 1e9, "unit": "GB/s",
                                      "l2": "flushed (512 MiB write) before the launch"}}


def split_kv(torch, api, peaks, peak_src):
    """One long causal head (B=1, H=1, N=32768, d=128): fewer query tile pairs than SMs. The
    tiled kernel alone against split-KV with the automatic split count, TFLOP/s of the contract
    count; L2 flushed before every timed launch (the inputs are smaller than L2)."""
    w = synth.WORKLOADS["one_head"]
    q, k, v, _ = synth.draw_workload(w)
    qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, v))
    od = torch.empty_like(qd)
    flops = synth.attention_flops(w.B, w.H, w.N, w.d, w.causal)
    n_splits = int(api._lib.lib().attn_splitkv_auto_splits(w.B, w.H, w.N, w.d, int(w.causal)))
    ws = torch.empty(api.splitkv_workspace_bytes(w.B, w.H, w.N, w.d, n_splits), dtype=torch.uint8,
                     device="cuda")
    flush = l2_flush_buffer(torch)

    def unsplit():
        api.fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, out=od, path="tcgen05")

    def split():
        api.fwd_splitkv(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, out=od,
                        n_splits=n_splits, workspace=ws)

    res = {}
    for name, fn in (("unsplit", unsplit), ("split", split)):
        time_launches(torch, fn, 3, flush)
        res[name] = statistics.median(time_launches(torch, fn, 20, flush))
    tf = {k2: flops / (ms * 1e-3) / 1e12 for k2, ms in res.items()}
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    return {"workload": w.describe(), "value": tf["split"], "unit": "TFLOP/s", "n_splits": n_splits,
            "launch_ms": res["split"], "unsplit_value": tf["unsplit"], "unsplit_launch_ms": res["unsplit"],
            "roofline": {"bound": "tensor", "achieved": tf["split"], "peak": peak, "unit": "TFLOP/s",
                         "frac": tf["split"] / peak, "peak_source": f"{peak_src} bf16 dense burst"},
            "l2": "flushed (512 MiB write) before every timed launch; the split launch includes the merge kernel"}


def to_host(torch, x, dtype):
    """numpy -> CPU tensor (uint16 bit patterns become torch.bfloat16 for bf16; float16 and
    float32 arrays keep their type)."""
    import numpy as np
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(x)


def to_device(torch, x, dtype):
    """numpy -> CUDA tensor (uint16 bit patterns become torch.bfloat16 for bf16)."""
    return to_host(torch, x, dtype).cuda()


def variants(torch, api, peaks, peak_src):
    """Grouped-query and cross-attention shapes and bf16 inputs on the tiled kernel, TFLOP/s of
    the contract count (allowed query/key pairs as the area under the causal diagonal); L2
    flushed before every timed launch."""
    flush = l2_flush_buffer(torch)
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    out = {}
    for name in ("long", "stress", "gqa_prefill", "chunk_prefill", "prefill_bf16"):
        w = synth.WORKLOADS[name]
        q, k, v, _ = synth.draw_workload(w)
        qd, kd, vd = (to_device(torch, x, w.dtype) for x in (q, k, v))
        od = torch.empty_like(qd)
        flops = synth.attention_flops_ex(w.B, w.H, w.N, w.N_k, w.d, w.causal)

        def fn():
            api.fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, out=od)

        time_launches(torch, fn, 3, flush)
        ms = statistics.median(time_launches(torch, fn, 10 if name == "long" else 30, flush))
        tf = flops / (ms * 1e-3) / 1e12
        out[name] = {"workload": w.describe(), "value": tf, "unit": "TFLOP/s", "launch_ms": ms,
                     "kernel": "tcgen05", "dtype": w.dtype,
                     "roofline": {"bound": "tensor", "achieved": tf, "peak": peak,
                                  "unit": "TFLOP/s", "frac": tf / peak,
                                  "traffic": traffic_from_profile("tcgen05", name),
                                  "peak_source": f"{peak_src} bf16 dense burst"}}
        del qd, kd, vd, od
    # decoding (one query, or a block of draft queries, per sequence, grouped heads): HBM-bound,
    # GB/s of Q, K, V read and O written once; the tiled kernel alone and split-KV with the
    # automatic split count
    for dname in ("decode_gqa", "spec_decode"):
        out[dname] = decode_line(torch, api, peaks, peak_src, flush, synth.WORKLOADS[dname])

    # fp32 inputs at the reranking shape: HBM-bound, GB/s of Q, K, V read and O written once
    w = synth.WORKLOADS["rerank_f32"]
    q, k, v, kl = synth.draw_workload(w)
    qd, kd, vd = (to_device(torch, x, w.dtype) for x in (q, k, v))
    kld = torch.from_numpy(kl).cuda()
    od = torch.empty_like(qd)

    def fn32(path):
        api.fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, key_lengths=kld, out=od, path=path)

    res32 = {}
    for path in ("auto", "tcgen05"):
        time_launches(torch, lambda: fn32(path), 3, flush)
        res32[path] = statistics.median(time_launches(torch, lambda: fn32(path), 30, flush))
    nbytes = 2 * synth.min_bytes(w.B, w.H, w.N, w.d) + kl.nbytes  # fp32: twice the fp16 bytes
    gbs = nbytes / (res32["auto"] * 1e-3) / 1e9
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    out["rerank_f32"] = {"workload": w.describe(), "value": gbs, "unit": "GB/s",
                         "launch_ms": res32["auto"], "bytes": nbytes,
                         "kernel": "warp-level split-TF32 (fp32 accuracy)",
                         "dtype": "f32 (split-TF32 products, fp32 accuracy)",
                         "tf32_value": nbytes / (res32["tcgen05"] * 1e-3) / 1e9,
                         "tf32_launch_ms": res32["tcgen05"], "tf32_kernel": "tcgen05 (TF32 products)",
                         "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                      "frac": gbs / hbm, "peak_source": f"{peak_src} copy bandwidth"},
                         "timing": "single launches, each after the L2 flush (launch latency included)"}
    out["l2"] = "flushed (512 MiB write) before every timed launch"
    return out


def naive_model_bytes(w):
    """Algorithmic bytes of one naive forward as the three passes run it: S (fp32) written
    once and read once, P (fp16) written once and read once, over the padded [B*H, N, Np]
    matrices, plus Q and K read by pass 1, V read by pass 3, O written and the lse (fp32)
    written once."""
    np_cols = (w.N + 127) // 128 * 128
    elems = w.B * w.H * w.N * np_cols
    return 12 * elems + 8 * w.B * w.H * w.N * w.d + 4 * w.B * w.H * w.N


def pages_model_bytes(w):
    """The naive page's count of the five-step pipeline's traffic per head, 7 S^2 + 4 S d
    fp16 elements ("Naive Attention Kernel", section "2. HBM Traffic Analysis"), in bytes
    over every head."""
    return w.B * w.H * (7 * w.N * w.N + 4 * w.N * w.d) * 2


def naive_lines(torch, api, peaks, peak_src):
    """The naive three-pass forward (S and P through HBM) against the fused kernel on the
    workloads it serves: per-launch time (median, L2 flushed before each launch), the
    algorithmic bytes of its three passes and the achieved rate of them against the measured
    copy bandwidth, the page's traffic model, the measured DRAM bytes of one launch (the three
    kernels, from the committed ncu summary while the source matches), and its time over the
    fused kernel's."""
    flush = l2_flush_buffer(torch)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    names = ("tiny", "rerank", "prefill", "stress")
    ws = torch.empty(max(api.naive_workspace_bytes(synth.WORKLOADS[n].B, synth.WORKLOADS[n].H,
                                                   synth.WORKLOADS[n].N) for n in names),
                     dtype=torch.uint8, device="cuda")
    out = {}
    for name in names:
        w = synth.WORKLOADS[name]
        q, k, v, kl = synth.draw_workload(w)
        qd, kd, vd = (torch.from_numpy(x).cuda() for x in (q, k, v))
        kld = torch.from_numpy(kl).cuda() if kl is not None else None
        od = torch.empty_like(qd)

        def naive():
            api.fwd_naive(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, key_lengths=kld,
                          out=od, workspace=ws)

        def fused():
            api.fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, key_lengths=kld, out=od)

        res = {}
        for label, fn in (("naive", naive), ("fused", fused)):
            time_launches(torch, fn, 3, flush)
            res[label] = statistics.median(time_launches(torch, fn, 10, flush))
        nbytes = naive_model_bytes(w)
        gbs = nbytes / (res["naive"] * 1e-3) / 1e9
        flops = synth.attention_flops(w.B, w.H, w.N, w.d, w.causal)
        out[name] = {"workload": w.describe(), "launch_ms": res["naive"],
                     "fused_launch_ms": res["fused"], "naive_over_fused": res["naive"] / res["fused"],
                     "value": flops / (res["naive"] * 1e-3) / 1e12, "unit": "TFLOP/s",
                     "model_bytes": nbytes, "pages_model_bytes": pages_model_bytes(w),
                     "fused_min_bytes": synth.min_bytes(w.B, w.H, w.N, w.d),
                     "dram_bytes_measured": traffic_from_profile("naive", name),
                     "gpu_launches": 3,
                     "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                                  "frac": gbs / hbm, "peak_source": f"{peak_src} copy bandwidth"}}
        del qd, kd, vd, od
    del ws
    out["timing"] = "single forwards (three kernels) after the L2 flush; median of 10"
    return out


def decode_line(torch, api, peaks, peak_src, flush, w):
    """One decoding workload: the automatic path, the tiled kernel alone and split-KV (automatic
    count), GB/s of Q, K, V read and O written once, single launches after the L2 flush."""
    q, k, v, _ = synth.draw_workload(w)
    qd, kd, vd = (to_device(torch, x, w.dtype) for x in (q, k, v))
    od = torch.empty_like(qd)
    nbytes = synth.min_bytes_ex(w.B, w.H, w.H_kv, w.N, w.N_k, w.d)
    n_splits = int(api._lib.lib().attn_splitkv_auto_splits_ex(w.B, w.H, w.H_kv, w.N, w.N_k, w.d,
                                                               int(w.causal)))
    ws = torch.empty(api.splitkv_workspace_bytes(w.B, w.H, w.N, w.d, n_splits), dtype=torch.uint8,
                     device="cuda")

    def auto():
        api.fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, out=od)

    def plain():
        api.fwd(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, out=od, path="tcgen05")

    def split():
        api.fwd_splitkv(qd, kd, vd, causal=w.causal, sm_scale=w.sm_scale, out=od, n_splits=n_splits,
                        workspace=ws)

    kernel = api.auto_path_ex(w.H, w.H_kv, w.N, w.N_k, w.d, w.dtype, w.causal)
    res = {}
    for name, fn in (("auto", auto), ("plain", plain), ("split", split)):
        time_launches(torch, fn, 3, flush)
        res[name] = statistics.median(time_launches(torch, fn, 30, flush))
    gbs = {name: nbytes / (ms * 1e-3) / 1e9 for name, ms in res.items()}
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    return {"workload": w.describe(), "value": gbs["auto"], "unit": "GB/s", "launch_ms": res["auto"],
            "kernel": kernel, "bytes": nbytes,
            "tcgen05_value": gbs["plain"], "tcgen05_launch_ms": res["plain"],
            "splitkv_value": gbs["split"], "splitkv_launch_ms": res["split"], "n_splits": n_splits,
            "roofline": {"bound": "hbm", "achieved": gbs["auto"], "peak": hbm, "unit": "GB/s",
                         "frac": gbs["auto"] / hbm, "peak_source": f"{peak_src} copy bandwidth"},
            "timing": "single launches after the L2 flush; split-KV includes the merge kernel; "
                      "tcgen05: query heads of a group packed into one tile"}

if __name__ == "__main__":
    sys.exit(main())
