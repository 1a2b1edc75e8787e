"""Benchmark: causal ring-attention forward on one B300 (or N replicas).

One step = one ``ring_attn_fwd`` call over the whole workload (every shard,
every ring step, online-softmax accumulation, normalised output and lse).
Default workload: B=1, H=32, Hkv=8, S=131072, D=128, P=16 virtual shards,
zig-zag layout, causal, bf16 inputs drawn from N(0, 1).

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead
(bounded row samples of the same workload on the host cores).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from ring_attention_02_b300.inputs import HEADLINE, Workload, by_name, make_for  # noqa: E402

METRIC = "causal ring-attn fwd TFLOP/s (bf16, S=128k, 1 B300) and % of BF16 tensor peak"
UNIT = "TFLOP/s"
L2_NOTE = "inputs larger than L2 (1.5 GiB of q/k/v, 126 MB L2); no flush"


def _dist():
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        torch.distributed.init_process_group(backend)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        return torch.distributed.get_rank(), torch.distributed.get_world_size()
    return 0, 1


def _barrier():
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def max_over_ranks(x: float) -> float:
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())
    return x


def config_of(w: Workload) -> dict:
    return {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "S": w.S, "D": w.D, "P": w.P,
            "layout": w.layout, "causal": w.causal, "l2": L2_NOTE}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples during the timed region (read-only queries)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.lines = []
        self.proc = None
        sel = []
        try:
            bus = torch.cuda.get_device_properties(device_index).pci_bus_id
            sel = ["-i", str(bus)]
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            if vis:
                sel = ["-i", vis.split(",")[device_index]]
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "200", *sel]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- peaks
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bf16_tflops"), d.get("bf16_tflops_sustained"), "of measured"
    return 1800.0, 1400.0, "of fallback"


def traffic_from_profiles():
    """Per-launch DRAM bytes of the forward kernel from the committed ncu summary."""
    path = os.path.join(ROOT, "profiles", "attn_fwd_headline_dram.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("bytes_per_launch")
    return None


# ---------------------------------------------------------------- CPU oracle leg
def oracle_sample(w: Workload, q, k, v, rows_per_step: int, seed: int):
    """Times the fp64 oracle on `rows_per_step` query rows (all heads)."""
    import oracle  # test infrastructure: the CPU-baseline leg only

    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(w.S, size=rows_per_step, replace=False)).astype(np.int64)
    qr = q[:, torch.from_numpy(rows).to(q.device)].float().cpu().numpy().astype(np.float64)
    flops = float(sum(4.0 * w.D * ((r + 1) if w.causal else w.S) for r in rows)) * w.B * w.H
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(qr, rows, k, v, w.causal, w.scale)
    dt = time.perf_counter() - t0
    return flops, dt


def host_kv(k, v):
    return (k.float().cpu().numpy().astype(np.float64), v.float().cpu().numpy().astype(np.float64))


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------- arms
def run_reference(args, w: Workload, rank: int):
    if rank != 0:
        return
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    q, k, v = make_for(w, seed=args.seed, device=dev)
    kh, vh = host_kv(k, v)
    rows = args.ref_rows
    for i in range(args.warmup):
        oracle_sample(w, q, kh, vh, rows, seed=1000 + i)
    tot_f, tot_t = 0.0, 0.0
    for i in range(args.steps):
        f, t = oracle_sample(w, q, kh, vh, rows, seed=i)
        tot_f += f
        tot_t += t
    val = tot_f / tot_t / 1e12
    sample = f"{rows} query rows x {w.B * w.H} (b,h) per step, uniform positions, fp64 C oracle"
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_e2e(w, api, q, k, v, out, lse, stream, dev, flops, world, steps):
    """Same metric through the public call with host buffers: each step copies
    q/k/v from pinned host memory, runs ring_attn_fwd and copies out and lse
    back, all inside the timed region."""
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    outh = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lseh = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    qd, kd, vd = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def e2e_step():
        qd.copy_(qh, non_blocking=True)
        kd.copy_(kh, non_blocking=True)
        vd.copy_(vh, non_blocking=True)
        api.fwd(qd, kd, vd, w.P, w.layout, w.causal, out=out, lse=lse, stream=stream)
        outh.copy_(out, non_blocking=True)
        lseh.copy_(lse, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize(dev)
    n = max(1, min(steps, 3))
    _barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    api.check_status(stream)
    ms = max_over_ranks(e0.elapsed_time(e1)) / n
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = out.numel() * out.element_size() + lse.numel() * lse.element_size()
    return {"value": world * flops / (ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms}


def run_ours(args, w: Workload, rank: int, world: int):
    from ring_attention_02_b300 import api

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    q, k, v = make_for(w, seed=args.seed + 17 * rank, device=dev)
    out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)

    def step():
        api.fwd(q, k, v, w.P, w.layout, w.causal, out=out, lse=lse, stream=stream)

    for _ in range(args.warmup):
        step()
    api.check_status(stream)

    # ---- device-resident timed region
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    _barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_all0 = torch.cuda.Event(enable_timing=True)
        t_all1 = torch.cuda.Event(enable_timing=True)
        t_all0.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t_all1.record(stream)
        torch.cuda.synchronize(dev)
    _barrier()
    api.check_status(stream)
    total_ms = t_all0.elapsed_time(t_all1)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(total_ms)
    ms_per_step = total_ms / args.steps
    flops = w.counted_flops()
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12

    # ---- end to end through host buffers (pinned), one C-ABI call per step
    e2e = None
    if not args.skip_e2e:
        e2e = measure_e2e(w, api, q, k, v, out, lse, stream, dev, flops, world, args.steps)
    if rank != 0:
        return
    peak, peak_sus, peak_src = measured_peaks()
    avg_launch = sum(launch_ms) / len(launch_ms)
    achieved = flops / (avg_launch * 1e-3) / 1e12
    pairs, tiles = api.census(w.S, w.P, w.layout, w.causal)
    tiles = tiles.double()
    imbalance = float(tiles.max() / tiles.mean() - 1.0)

    # CPU oracle on a bounded sample (rank 0, N=1 only)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        kh, vh = host_kv(k, v)
        f_s, t_s = 0.0, 0.0
        while t_s < args.cpu_seconds:
            f, t = oracle_sample(w, q, kh, vh, 64, seed=int(t_s * 1000) + 7)
            f_s += f
            t_s += t
        cpu = {"value": f_s / t_s / 1e12, "unit": UNIT, "cores": cores(), "kind": "oracle",
               "sample": f"uniform query rows x {w.B * w.H} (b,h), {t_s:.1f} s of fp64 C oracle, "
                         f"{f_s:.3g} counted flop"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(w),
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "traffic": traffic_from_profiles(),
                     "peak_source": f"bf16 burst {peak_src}", "peak_sustained": peak_sus,
                     "kernel": "attn_fwd_kernel<128>"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "shard_imbalance": imbalance,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--workload", default=HEADLINE.name,
                    help="registered workload name (default: the 128k GQA zig-zag forward)")
    ap.add_argument("--layout", default=None, help="override the workload's layout")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=48)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = by_name(args.workload)
    if args.layout is not None and args.layout != w.layout:
        w = w.with_layout(args.layout)
    rank, world = _dist()
    if args.impl == "reference":
        run_reference(args, w, rank)
    else:
        run_ours(args, w, rank, world)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
