"""Benchmark of the attention forward pass (libosattn) on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step = one osattn_fwd call over the whole workload (every (b, h, query
tile)).  The default workload is the largest bf16 one: causal B=1, H=32,
N=16384, d=128, Q ~ N(0, 9), K, V ~ N(0, 1).  FLOPs per step are the nominal
4*B*H*Nq*Nkv*d, halved for causal.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events
on the launching stream with an L2 flush (a 256 MiB write) between steps
outside the events; a barrier and a device synchronisation on both sides of
the timed loop; the max over ranks.  nvidia-smi samples SM clocks and
throttle reasons during the timed loop.  `e2e` repeats the measurement
with the inputs in pinned host memory: every step copies Q, K, V
host->device and O, LSE device->host inside the events, through
osattn_fwd_offload (the library's host-memory entry point, which pipelines
the copies with the compute over chunks of heads); split-KV workloads copy,
call and copy back in sequence.

other_configs: with the default workload, the other two large forward
workloads (causal B=4 H=16 N=4096 d=64 and B=8 H=40 N=2048 d=128) are timed
the same way, kernel only, each with its own clock record and the max-abs
error of 256 sampled rows against the oracle.

cpu_baseline: the fp64 oracle as it stands, timed on this host's cores on a
bounded random sample of query rows of the same workload (about 10-20 s of
CPU work) and scaled to TFLOPS by the sample's own FLOPs; the GPU's outputs
on those rows give the max-abs error reported beside the throughput.

--impl reference: times that oracle alone (rank 0; other ranks exit 0), each
step a bounded row sample, and prints the same JSON line with
"impl": "reference".

N > 1 (torchrun): replicas only - every rank runs its own copy of the
workload (no collective on the data path); value = total FLOPs of all ranks
over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOPS on 1 GB300 and % of dense BF16 tensor peak; max-abs err vs oracle"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNEL_SOURCES = ("fwd_bf16_tcgen05.cu", "sm100_ptx.cuh", "tc_attn_mma.cuh")


def fwd_config(w, world):
    """The forward line's `config`, shared by both arms."""
    return {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nkv": w.Nkv, "d": w.d,
            "causal": w.causal, "key_len": w.key_len, "splits": w.splits, "flops_per_step": w.flops,
            "l2": "flushed between timed steps (256 MiB write)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "attention_forward_online_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per launch of the bf16 kernel from the committed ncu summary,
    if it was taken on the kernel source as it is now (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(workload)
    if not ent or ent.get("kernel_source_sha") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    # Raw nvidia-smi samples of the timed region go to this directory (under
    # the repository, git-ignored); OSATTN_CLOCKS_DIR overrides it.
    LOG_DIR = os.environ.get("OSATTN_CLOCKS_DIR", os.path.join(ROOT, "bench_logs"))

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = os.path.join(self.LOG_DIR, f"clocks_bench_gpu{gpu_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            return summarize_clocks(f)


def summarize_clocks(lines):
    """Median SM clock, maximum clock and the throttle reasons seen, from
    nvidia-smi CSV lines in ClockSampler.FIELDS order; None without samples."""
    sm, mx, reasons = [], 0.0, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx = max(mx, float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
            "samples": len(sm)}


REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(info):
    """Why a timed region's clock record voids its number, or None: a
    hardware or thermal slowdown, or a median SM clock below 80 % of the
    maximum with no reason active (a leftover clock lock).  sw_power_cap
    alone is kept (and shows in the record)."""
    if not info:
        return None
    bad = [r for r in info["reasons"] if r in REJECT_REASONS]
    if bad:
        return ",".join(bad)
    if not info["reasons"] and info["sm_max_mhz"] > 0 and info["sm_mhz"] < 0.8 * info["sm_max_mhz"]:
        return f"sm clock {info['sm_mhz']:.0f} of {info['sm_max_mhz']:.0f} MHz with no reason"
    return None


def timed_steps(torch, dev, stream, step, flush, steps, world, gpu_index):
    """Times `steps` calls of step() on `stream`, each after a write of
    `flush` (larger than L2), with CUDA events on that stream, a barrier and
    a device synchronise on both sides and the SM clocks sampled throughout.
    When the clock record voids the number (clocks_rejected) on any rank,
    every rank runs the loop once more and the second run is kept, its
    record noting why.  Returns (per-step milliseconds, clock record)."""
    first_why = None
    for attempt in range(2):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        clocks = ClockSampler(gpu_index)
        barrier(world)
        torch.cuda.synchronize(dev)
        clocks.start()
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            for i in range(steps):
                flush.fill_(i & 0xFF)  # evict the previous step's lines from L2
                starts[i].record(stream)
                step()
                ends[i].record(stream)
        torch.cuda.synchronize(dev)
        info = clocks.stop()
        barrier(world)
        ms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
        why = clocks_rejected(info)
        if attempt == 0 and reduce_max(1.0 if why else 0.0, world) > 0:
            first_why = why or "another rank's clock record"
            continue
        if first_why and info is not None:
            info["remeasured_after"] = first_why
        return ms, info


# ------------------------------------------------------------------ distributed
def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group(backend=os.environ.get("OSATTN_DIST_BACKEND", "nccl"))
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def reduce_max(value: float, world: int) -> float:
    """Max of a per-rank float over all ranks (rank-local value if world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ oracle leg
def row_flops(w, rows):
    """FLOPs the definition spends on the given flat rows: 4*d per visible key."""
    total = 0
    for r in rows:
        i = r % w.Nq
        vis = w.Nkv if not w.causal else min(w.Nkv, i + 1)
        total += 4 * w.d * vis
    return total


def oracle_sample(w, q, k, v, n_rows, seed):
    import numpy as np

    import oracle

    rng = np.random.default_rng(seed)
    rows = sorted(set(rng.integers(0, w.B * w.H * w.Nq, size=n_rows).tolist()))
    t0 = time.perf_counter()
    O, L = oracle.attention_fwd(q, k, v, w.scale, w.causal, w.key_len, rows=rows)
    dt = time.perf_counter() - t0
    return rows, O, L, dt


def calibrate_rows(w, q, k, v, target_s: float, seed: int):
    """Number of sampled rows whose oracle time is about target_s: one small
    warm-up call (thread start-up, page faults), then a timed call whose row
    count grows until it takes at least a quarter of a second."""
    oracle_sample(w, q, k, v, 32, seed)
    n = 256
    while True:
        rows, _, _, dt = oracle_sample(w, q, k, v, n, seed + 1)
        if dt >= 0.25 or n >= 1 << 20:
            break
        n *= 4
    per_row = dt / max(len(rows), 1)
    return max(64, int(target_s / max(per_row, 1e-9)))


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args, w):
    rank, _, world = int(os.environ.get("RANK", "0")), 0, int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    from attention_forward_online_gb300.inputs import make_inputs

    q, k, v, _ = make_inputs(w)
    # Each step is a bounded row sample: about two minutes for the whole run
    # (K + W steps), at most 4 s a step.
    per_step = max(0.05, min(4.0, 120.0 / max(1, args.steps + args.warmup)))
    n_rows = calibrate_rows(w, q, k, v, target_s=per_step, seed=1)
    for s in range(args.warmup):
        oracle_sample(w, q, k, v, n_rows, seed=100 + s)
    flops, secs = 0, 0.0
    for s in range(args.steps):
        rows, _, _, dt = oracle_sample(w, q, k, v, n_rows, seed=1000 + s)
        flops += row_flops(w, rows)
        secs += dt
    tflops = flops / secs / 1e12
    sample = (f"{args.steps} steps x {n_rows} random query rows of {w.name} "
              f"(of {w.B * w.H * w.Nq}), fp64, {secs:.1f} s total")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(tflops, 6), "unit": "TFLOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": fwd_config(w, world),
        "cpu_baseline": {"value": round(tflops, 6), "unit": "TFLOPS", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(tflops, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ other configs
# The other two large forward workloads, timed kernel-only beside the
# headline one (the line's `other_configs`).
OTHER_CONFIGS = ("bf16_causal_b4_h16_n4096_d64", "bf16_b8_h40_n2048_d128")


def measure_other_configs(torch, dev, stream, flush, args, world, local, rank, peak):
    """Kernel-only CUDA-event timing of each OTHER_CONFIGS workload (3
    warm-up calls, then min(steps, 20) timed calls with the L2 flushed
    between them and the clocks sampled), and on rank 0 the max-abs error
    of 256 sampled rows against the oracle."""
    import numpy as np

    from attention_forward_online_gb300 import osattn
    from attention_forward_online_gb300.inputs import WORKLOADS, make_inputs, sample_rows

    out = []
    for name in OTHER_CONFIGS:
        w = WORKLOADS[name]
        q, k, v, _ = make_inputs(w)
        qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
        O = torch.empty_like(qd)
        L = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)

        def step():
            osattn.fwd(qd, kd, vd, scale=w.scale, causal=w.causal, out=O, lse=L, stream=stream)

        with torch.cuda.stream(stream):
            for _ in range(3):
                step()
        stream.synchronize()
        steps = max(3, min(args.steps, 20))
        ms, clocks = timed_steps(torch, dev, stream, step, flush, steps, world, local)
        if osattn.get_device_status(stream) != osattn.OK:
            raise RuntimeError(f"device-side wait timed out on {name}")
        avg = reduce_max(sum(ms), world) / steps
        tflops = w.flops / (avg * 1e-3) / 1e12
        rec = {"workload": name, "steps": steps, "ms_per_launch": round(avg, 4),
               "tflops": round(tflops, 2), "pct_of_bf16_peak": round(100 * tflops / peak, 2),
               "traffic": committed_traffic(name), "clocks": clocks}
        if rank == 0:
            import oracle

            rows = sample_rows(w.B, w.H, w.Nq, 256, seed=11)
            Oref, Lref = oracle.attention_fwd(q, k, v, w.scale, w.causal, rows=rows)
            idx = torch.tensor(rows, device=dev)
            Og = O.reshape(-1, w.d)[idx].double().cpu().numpy()
            Lg = L.reshape(-1)[idx].double().cpu().numpy()
            rec["max_abs_err"] = {"O": float(np.abs(Og - Oref).max()),
                                  "LSE": float(np.abs(Lg - Lref).max()), "rows_checked": len(rows)}
        out.append(rec)
        del qd, kd, vd, O, L
    return out


# ------------------------------------------------------------------ our arm
def run_ours(args, w):
    import torch

    from attention_forward_online_gb300 import osattn
    from attention_forward_online_gb300.inputs import make_inputs

    rank, local, world = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()

    q, k, v, kl = make_inputs(w)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    kld = None if kl is None else kl.to(dev)
    O = torch.empty_like(qd)
    L = torch.empty((w.B, w.H, w.Nq), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    ws = None
    if w.splits:
        ws = torch.empty(osattn.splitkv_workspace_bytes(w.B, w.H, w.Nq, w.d, w.splits),
                         dtype=torch.uint8, device=dev)

    def step():
        if w.splits:  # split-KV entry point: split kernel + combine kernel
            osattn.fwd_splitkv(qd, kd, vd, w.splits, scale=w.scale, causal=w.causal,
                               key_len=kld, out=O, lse=L, workspace=ws, stream=stream)
        else:
            osattn.fwd(qd, kd, vd, scale=w.scale, causal=w.causal, key_len=kld, out=O,
                       lse=L, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.synchronize()
    if osattn.get_device_status(stream) != osattn.OK:
        raise RuntimeError("device-side wait timed out during warm-up")

    # ---- device-resident timing
    per_launch_ms, clock_info = timed_steps(torch, dev, stream, step, flush, args.steps, world,
                                            local)
    if osattn.get_device_status(stream) != osattn.OK:
        raise RuntimeError("device-side wait timed out in the timed region")
    local_ms = sum(per_launch_ms)
    total_ms = reduce_max(local_ms, world)
    ms_per_step = total_ms / args.steps
    value = world * w.flops * args.steps / (total_ms * 1e-3) / 1e12
    avg_launch_ms = local_ms / args.steps
    achieved = w.flops / (avg_launch_ms * 1e-3) / 1e12

    # ---- end to end through the C ABI from pinned host buffers
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    Oh = torch.empty(O.shape, dtype=O.dtype).pin_memory()
    Lh = torch.empty(L.shape, dtype=L.dtype).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    es = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            flush.fill_(i & 0xFF)
            es[i].record(stream)
            if w.splits:
                qd.copy_(qh, non_blocking=True)
                kd.copy_(kh, non_blocking=True)
                vd.copy_(vh, non_blocking=True)
                step()
                Oh.copy_(O, non_blocking=True)
                Lh.copy_(L, non_blocking=True)
            else:
                osattn.fwd_offload(qh, kh, vh, Oh, Lh, qd, kd, vd, O, L, scale=w.scale,
                                   causal=w.causal, key_len=kld, stream=stream)
            ee[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = reduce_max(sum(s.elapsed_time(e) for s, e in zip(es, ee)), world) / e2e_steps
    e2e_value = world * w.flops / (e2e_ms * 1e-3) / 1e12
    h2d = sum(t.numel() * t.element_size() for t in (qh, kh, vh))
    d2h = Oh.numel() * Oh.element_size() + Lh.numel() * Lh.element_size()
    others = []
    if args.other_configs:
        others = measure_other_configs(torch, dev, stream, flush, args, world, local, rank,
                                       float(peaks["bf16_tflops"]))

    line = None
    if rank == 0:
        # ---- oracle leg: CPU baseline on a bounded row sample + max-abs error
        n_rows = calibrate_rows(w, q, k, v, target_s=args.cpu_seconds, seed=7)
        rows, Oref, Lref, secs = oracle_sample(w, q, k, v, n_rows, seed=8)
        cpu_tflops = row_flops(w, rows) / secs / 1e12
        idx = torch.tensor(rows, device=dev)
        Og = O.reshape(-1, w.d)[idx].double().cpu().numpy()
        Lg = L.reshape(-1)[idx].double().cpu().numpy()
        import numpy as np

        fin = np.isfinite(Lref)
        err_o = float(np.abs(Og - Oref).max())
        err_l = float(np.abs(Lg[fin] - Lref[fin]).max()) if fin.any() else 0.0

        peak = float(peaks["bf16_tflops"])
        traffic = committed_traffic(w.name)
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": fwd_config(w, world),
            "pct_of_bf16_peak": round(100 * value / world / peak, 2),
            "pct_of_bf16_peak_sustained": round(
                100 * value / world / float(peaks["bf16_tflops_sustained"]), 2),
            "max_abs_err": {"O": err_o, "LSE": err_l, "rows_checked": len(rows)},
            "roofline": {"bound": "tensor", "achieved": round(achieved, 3),
                         "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4), "traffic": traffic,
                         "kernel": ("fwd_bf16_kernel (split) + splitkv_combine_kernel, timed together"
                                    if w.splits else
                                    "fwd_bf16_kernel" if w.dtype == "bf16" else "fwd_fp32_kernel"),
                         "peak_source": f"bf16_tflops (burst) of {peak_src}"},
            "cpu_baseline": {"value": round(cpu_tflops, 6), "unit": "TFLOPS",
                             "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{len(rows)} random query rows of {w.name}, fp64, "
                                       f"{secs:.1f} s"},
            "e2e": {"value": round(e2e_value, 3), "unit": "TFLOPS",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms, 4),
                    "api": "osattn_fwd" if w.splits else "osattn_fwd_offload"},
            "gpu_launches": args.steps * (2 if w.splits else 1),
            "clocks": clock_info,
            "kernel_source_sha": kernel_source_hash(),
        }
        if others:
            line["other_configs"] = others
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ backward
BWD_METRIC = "attention backward TFLOPS on 1 GB300 (2.5x forward FLOPs) and % of dense BF16 peak"


def bwd_oracle_sample(w, q, k, v, do, target_s: float):
    """The oracle's gradients on a bounded sample of the workload: batch 0,
    its first `heads` heads, and for a causal workload only the first n
    query rows and keys (n grown until the call takes about a quarter of
    target_s; a causal prefix is itself a causal problem with the same dQ
    rows).  Returns (heads, n, dQ, dK, dV, secs, flops)."""
    import oracle

    cores = cpu_cores()
    # A causal prefix is the same problem for its dQ rows; without the mask
    # every row sees every key, so only whole heads are comparable.
    heads, n = min(w.H, cores), (min(w.Nq, w.Nkv, 256) if w.causal else w.Nq)
    while True:
        sl = (slice(0, 1), slice(0, heads), slice(0, n))
        t0 = time.perf_counter()
        dQ, dK, dV = oracle.attention_bwd(q[sl], k[sl], v[sl], do[sl], w.scale, w.causal, None)
        secs = time.perf_counter() - t0
        flops = 10.0 * heads * n * n * w.d / (2 if w.causal else 1)
        if secs >= target_s / 4 or n >= min(w.Nq, w.Nkv):
            break
        n = min(n * 2, w.Nq, w.Nkv)
    return heads, n, dQ, dK, dV, secs, flops


def run_bwd(args, w):
    import numpy as np
    import torch

    from attention_forward_online_gb300 import osattn
    from attention_forward_online_gb300.inputs import make_grad_out, make_inputs

    rank, local, world = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    q, k, v, kl = make_inputs(w)
    do = make_grad_out(w)
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        O, L = osattn.fwd(qd, kd, vd, scale=w.scale, causal=w.causal, stream=stream)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(osattn.bwd_workspace_bytes(w.B, w.H, w.Nq), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step():
        osattn.bwd(qd, kd, vd, O, L, dod, scale=w.scale, causal=w.causal, dq=dq, dk=dk, dv=dv,
                   workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.synchronize()
    if osattn.get_device_status(stream) != osattn.OK:
        raise RuntimeError("device-side wait timed out during warm-up")
    step_ms, clock_info = timed_steps(torch, dev, stream, step, flush, args.steps, world, local)
    if osattn.get_device_status(stream) != osattn.OK:
        raise RuntimeError("device-side wait timed out in the timed region")
    local_ms = sum(step_ms)
    total_ms = reduce_max(local_ms, world)
    value = world * w.bwd_flops * args.steps / (total_ms * 1e-3) / 1e12
    achieved = w.bwd_flops / (local_ms / args.steps * 1e-3) / 1e12

    # end to end: inputs (q, k, v, O, LSE, dO) in, gradients out
    hin = [t.pin_memory() for t in (q, k, v, O.cpu(), L.cpu(), do)]
    hout = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)]
    e2e_steps = max(3, min(args.steps, 20))
    es = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(e2e_steps):
            flush.fill_(i & 0xFF)
            es[i].record(stream)
            osattn.bwd_offload(*hin, scale=w.scale, causal=w.causal, dq_host=hout[0],
                               dk_host=hout[1], dv_host=hout[2],
                               device_buffers=(qd, kd, vd, O, dod, dq, dk, dv, L), workspace=ws,
                               stream=stream)
            ee[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = reduce_max(sum(s.elapsed_time(e) for s, e in zip(es, ee)), world) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in hin)
    d2h = sum(t.numel() * t.element_size() for t in hout)

    if rank == 0:
        heads, n, rQ, rK, rV, secs, cflops = bwd_oracle_sample(w, q, k, v, do, args.cpu_seconds)
        gq = dq[0:1, :heads, :n].double().cpu().numpy()
        err = {"dQ": float(np.abs(gq - rQ).max())}
        if n == w.Nq and n == w.Nkv:  # the sample is whole heads: dK and dV comparable too
            err["dK"] = float(np.abs(dk[0:1, :heads].double().cpu().numpy() - rK).max())
            err["dV"] = float(np.abs(dv[0:1, :heads].double().cpu().numpy() - rV).max())
        err["sample"] = f"batch 0, heads 0-{heads - 1}, first {n} rows"
        peak = float(peaks["bf16_tflops"])
        line = {
            "metric": BWD_METRIC, "value": round(value, 3), "unit": "TFLOPS", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Nq": w.Nq, "Nkv": w.Nkv,
                       "d": w.d, "causal": w.causal, "flops_per_step": w.bwd_flops,
                       "l2": "flushed between timed steps (256 MiB write)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "pct_of_bf16_peak": round(100 * value / world / peak, 2),
            "max_abs_err": err,
            "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": None,
                         "kernel": "bwd_dq + bwd_dkdv kernels (D formed in the dQ kernel), timed together",
                         "peak_source": f"bf16_tflops (burst) of {peak_src}"},
            "cpu_baseline": {"value": round(cflops / secs / 1e12, 6), "unit": "TFLOPS",
                             "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"gradients of batch 0, {heads} heads, first {n} query "
                                       f"rows and keys of {w.name}, fp64, {secs:.1f} s"},
            "e2e": {"value": round(world * w.bwd_flops / (e2e_ms * 1e-3) / 1e12, 3),
                    "unit": "TFLOPS", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": round(e2e_ms, 4), "api": "osattn_bwd_offload"},
            "gpu_launches": args.steps * 3,
            "clocks": clock_info,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ row softmax
def run_softmax_rows(args, w):
    """The standalone online row softmax: HBM-bound, one read and one write
    per element; value = bytes moved / kernel time."""
    import numpy as np
    import torch

    from attention_forward_online_gb300 import osattn
    from attention_forward_online_gb300.inputs import make_rows

    rank, local, world = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    x = make_rows(w)
    xd = x.to(dev)
    yd = torch.empty_like(xd)
    ld = torch.empty(w.rows, dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        osattn.softmax_rows(xd, out=yd, lse=ld, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            step()
    stream.synchronize()
    step_ms, clock_info = timed_steps(torch, dev, stream, step, flush, args.steps, world, local)
    local_ms = sum(step_ms)
    total_ms = reduce_max(local_ms, world)
    gbs = world * w.bytes_moved * args.steps / (total_ms * 1e-3) / 1e9
    achieved = w.bytes_moved / (local_ms / args.steps * 1e-3) / 1e9

    xh = x.pin_memory()
    yh = torch.empty(x.shape, dtype=x.dtype).pin_memory()
    lh = torch.empty(w.rows, dtype=torch.float32).pin_memory()
    n_e2e = max(3, min(args.steps, 20))
    es = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(n_e2e)]
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        for i in range(n_e2e):
            es[i].record(stream)
            osattn.softmax_rows_offload(xh, yh, lh, xd, yd, ld, stream=stream)
            ee[i].record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(sum(s_.elapsed_time(e_) for s_, e_ in zip(es, ee)), world) / n_e2e
    if rank == 0:
        import oracle

        rng = np.random.default_rng(9)
        n_rows = 64
        while True:  # bounded sample: grow until the oracle takes ~args.cpu_seconds
            rows = np.sort(rng.choice(w.rows, size=min(n_rows, w.rows), replace=False))
            t0 = time.perf_counter()
            Yr, Lr = oracle.softmax_rows(x[torch.from_numpy(rows)])
            secs = time.perf_counter() - t0
            if secs >= args.cpu_seconds / 4 or n_rows >= w.rows:
                break
            n_rows = min(w.rows, int(n_rows * max(2.0, args.cpu_seconds / 4 / max(secs, 1e-3))))
        cpu_gbs = len(rows) * (w.N * w.elem_bytes * 2 + 4) / secs / 1e9
        Yg = yd[torch.from_numpy(rows).to(dev)].double().cpu().numpy()
        Lg = ld[torch.from_numpy(rows).to(dev)].double().cpu().numpy()
        fin = np.isfinite(Lr)
        peak = float(peaks["hbm_gbs"])
        line = {
            "metric": "online row softmax HBM GB/s (one read + one write per element)",
            "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "rows": w.rows, "N": w.N,
                       "bytes_per_step": w.bytes_moved,
                       "l2": "flushed between timed steps (256 MiB write)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "max_abs_err": {"y": float(np.abs(Yg - Yr).max()),
                            "LSE": float(np.abs(Lg[fin] - Lr[fin]).max()),
                            "rows_checked": int(len(rows))},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": None,
                         "kernel": "softmax_rows_regs",
                         "peak_source": f"hbm_gbs (copy) of {peak_src}"},
            "cpu_baseline": {"value": round(cpu_gbs, 4), "unit": "GB/s", "cores": cpu_cores(),
                             "kind": "oracle",
                             "sample": f"{len(rows)} random rows of {w.name}, fp64, {secs:.1f} s"},
            "e2e": {"value": round(world * w.bytes_moved / (e2e_ms * 1e-3) / 1e9, 2),
                    "unit": "GB/s", "h2d_bytes_per_step": xh.numel() * xh.element_size(),
                    "d2h_bytes_per_step": yh.numel() * yh.element_size() + lh.numel() * 4,
                    "ms_per_step": round(e2e_ms, 4), "api": "osattn_softmax_rows_offload"},
            "gpu_launches": args.steps, "clocks": clock_info,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    from attention_forward_online_gb300.inputs import (BENCH_WORKLOAD, BWD_WORKLOADS,
                                                       ROW_WORKLOADS, SPLITKV_WORKLOADS,
                                                       WORKLOADS)

    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    allw = dict(WORKLOADS, **SPLITKV_WORKLOADS)
    ap.add_argument("--workload", default=BENCH_WORKLOAD,
                    choices=sorted(allw) + sorted(ROW_WORKLOADS) + sorted(BWD_WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--other-configs", dest="other_configs", action="store_true", default=None,
                    help="also time the other large forward workloads (default: with the "
                         "default workload only)")
    ap.add_argument("--no-other-configs", dest="other_configs", action="store_false")
    args = ap.parse_args(argv)
    if args.other_configs is None:
        args.other_configs = args.workload == BENCH_WORKLOAD
    if args.workload in ROW_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the reference arm is defined for the attention workloads"}))
            return 0
        return run_softmax_rows(args, ROW_WORKLOADS[args.workload])
    if args.workload in BWD_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the reference arm is defined for the forward attention workloads"}))
            return 0
        return run_bwd(args, BWD_WORKLOADS[args.workload])
    w = allw[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
