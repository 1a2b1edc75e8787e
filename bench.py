"""Benchmark: causal ring-attention forward on one B300 (or N replicas).

One step = one ``ring_attn_fwd`` call over the whole workload (every shard,
every ring step, online-softmax accumulation, normalised output and lse).
Default workload: B=1, H=32, Hkv=8, S=131072, D=128, P=16 virtual shards,
zig-zag layout, causal, bf16 inputs drawn from N(0, 1).

With a training workload (``--workload train-B2H16S32768D128P8``) one step
is ``ring_attn_fwd`` followed by ``ring_attn_bwd`` (dq, dk, dv from a seeded
dO), counted as 3.5x the forward's flops.

``--op`` times one of the other calls on the workload's shapes instead:
``permute`` (token rows of q into shard-major order, HBM bound), ``merge``
(LSE fold of one shard's fp32 partials, HBM bound), ``step_merge`` (the
per-hop form of the whole ring: P*P ``ring_attn_step`` calls and the
``ring_attn_merge`` folds, on shard-major inputs permuted beforehand) or
``decode`` (``--decode-tokens`` new tokens against the workload's key/value
cache, HBM bound) or ``varlen`` (the forward over a pack of 16 documents with
a seeded log-uniform length mix of 2k..32k tokens, on the workload's heads).

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead
(bounded samples of the same workload on the host cores).
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from ring_attention_02_b300.inputs import (HEADLINE, Workload, by_name, make_dout,  # noqa: E402
                                           make_for, make_qkv)

METRIC = "causal ring-attn fwd TFLOP/s (bf16, S=128k, 1 B300) and % of BF16 tensor peak"
METRIC_TRAIN = "causal ring-attn fwd+bwd TFLOP/s (bf16, 1 B300; bwd counted as 2.5x fwd)"
UNIT = "TFLOP/s"
NOMINAL_BF16_TFLOPS = 2250.0   # dense bf16 tensor rate of a B300, vendor figure (context)


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
    qkv = w.B * w.S * (w.H + 2 * w.Hkv) * w.D * 2
    l2 = (f"inputs larger than L2 ({qkv / 2**30:.2f} GiB of q/k/v, 126 MB L2); no flush"
          if qkv > 126e6 else "inputs smaller than L2: repeated steps may hit in L2")
    return {"workload": w.name, "B": w.B, "H": w.H, "Hkv": w.Hkv, "S": w.S, "D": w.D, "P": w.P,
            "layout": w.layout, "causal": w.causal, "backward": w.backward, "l2": l2}


def metric_of(w: Workload) -> str:
    return METRIC_TRAIN if w.backward else METRIC


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


def measured_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f).get("hbm_gbs"), "of measured"
    return 6400.0, "of fallback"


FWD_SOURCES = ["attn_fwd.cuh", "geometry.cuh", "sm103_ptx.cuh"]


def fwd_source_digest() -> str:
    import hashlib

    h = hashlib.sha256()
    for name in FWD_SOURCES:
        with open(os.path.join(ROOT, "ring_attention_02_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def traffic_from_profiles(w: Workload):
    """DRAM bytes per launch of the forward kernel on this workload, from the
    committed ncu summary, or None when there is none or the kernel sources
    changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"attn_fwd_traffic_{w.name}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for ln in f:
            if ":" in ln and not ln.startswith("#"):
                key, val = ln.split(":", 1)
                vals[key.strip()] = val.strip()
    if vals.get("kernel_sources_sha256") != fwd_source_digest():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- CPU oracle leg
def oracle_sample(w: Workload, q, k, v, rows_per_step: int, seed: int, nthreads=None):
    """Times the fp64 oracle on `rows_per_step` query rows (all heads), on
    `nthreads` host threads (all cores when None)."""
    import oracle  # test infrastructure: the CPU-baseline leg only

    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(w.S, size=rows_per_step, replace=False)).astype(np.int64)
    qr = q[:, torch.from_numpy(rows).to(q.device)].float().cpu().numpy().astype(np.float64)
    flops = float(sum(4.0 * w.D * ((r + 1) if w.causal else w.S) for r in rows)) * w.B * w.H
    t0 = time.perf_counter()
    oracle.attn_fwd_rows(qr, rows, k, v, w.causal, w.scale, nthreads=nthreads)
    dt = time.perf_counter() - t0
    return flops, dt


def oracle_train_sample(w: Workload, q, k, v, do, prefix: int, nthreads=None):
    """Times the fp64 oracle's forward+backward on one (b, kv head) pair over
    the first `prefix` tokens (a causal prefix is a whole problem of its own)."""
    import oracle  # test infrastructure: the CPU-baseline leg only

    G = w.H // w.Hkv
    sl = slice(0, prefix)
    f64 = lambda t: t[:1, sl].float().cpu().numpy().astype(np.float64)
    qs = f64(q[:, :, :G])
    ks, vs = f64(k[:, :, :1]), f64(v[:, :, :1])
    dos = f64(do[:, :, :G])
    flops = 3.5 * 4.0 * G * prefix * prefix * w.D / (2 if w.causal else 1)
    t0 = time.perf_counter()
    oracle.attn_fwd(qs, ks, vs, w.causal, w.scale, nthreads=nthreads)
    oracle.attn_bwd(qs, ks, vs, dos, w.causal, w.scale, [(0, 0)], nthreads=nthreads)
    return flops, time.perf_counter() - t0


def host_kv(k, v):
    return (k.float().cpu().numpy().astype(np.float64), v.float().cpu().numpy().astype(np.float64))


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or "unknown"


def one_core_baseline(w: Workload, q, k, v, do, kh, vh, prefix: int, seconds: float = 2.0):
    """The same oracle on one host thread, over a short sample, for scale."""
    f1, t1 = 0.0, 0.0
    if w.backward:
        pre = min(prefix, 1024)
        f1, t1 = oracle_train_sample(w, q, k, v, do, pre, nthreads=1)
        what = f"fwd+bwd of (b=0, kv head 0) over the first {pre} tokens"
    else:
        while t1 < seconds:
            f, t = oracle_sample(w, q, kh, vh, 1, seed=int(t1 * 1000) + 11, nthreads=1)
            f1 += f
            t1 += t
        what = f"uniform query rows x {w.B * w.H} (b,h)"
    return {"value": f1 / t1 / 1e12, "unit": UNIT, "cores": 1,
            "sample": f"{what}, {t1:.1f} s of fp64 C oracle on 1 thread"}


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
    tot_f, tot_t = 0.0, 0.0
    if w.backward:
        do = make_dout(w.B, w.H, w.S, w.D, seed=args.seed, device=dev)
        prefix = args.ref_prefix
        for i in range(args.warmup):
            oracle_train_sample(w, q, k, v, do, min(prefix, 512))
        for i in range(args.steps):
            f, t = oracle_train_sample(w, q, k, v, do, prefix)
            tot_f += f
            tot_t += t
        sample = (f"fwd+bwd of (b=0, kv head 0) over the first {prefix} tokens per step, "
                  f"fp64 C oracle")
    else:
        kh, vh = host_kv(k, v)
        rows = args.ref_rows
        for i in range(args.warmup):
            oracle_sample(w, q, kh, vh, rows, seed=1000 + i)
        for i in range(args.steps):
            f, t = oracle_sample(w, q, kh, vh, rows, seed=i)
            tot_f += f
            tot_t += t
        sample = f"{rows} query rows x {w.B * w.H} (b,h) per step, uniform positions, fp64 C oracle"
    val = tot_f / tot_t / 1e12
    line = {"impl": "reference", "metric": metric_of(w), "value": val, "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_of(w),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores(), "kind": "oracle",
                             "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def measure_e2e(w, api, make_step, dev_in, dev_out, dev_scratch, dev, flops, world, steps):
    """Same metric through the public calls with host buffers: every step
    copies its inputs from pinned host memory to the device, runs the step and
    copies its results back to pinned host memory, all inside the timed region.
    Steps are pipelined the way a serving or training loop runs them: two
    device buffer sets, and separate streams for host-to-device copies, compute
    and device-to-host copies, so step i's copies overlap step i-1's compute.
    make_step(ins, outs, scratch, stream) runs one step on one buffer set."""
    host_in = [t.cpu().pin_memory() for t in dev_in]
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in dev_out]
    sets = [(dev_in, dev_out, dev_scratch),
            ([torch.empty_like(t) for t in dev_in], [torch.empty_like(t) for t in dev_out],
             [torch.empty_like(t) for t in dev_scratch])]
    s_h2d, s_cmp, s_d2h = (torch.cuda.Stream(dev) for _ in range(3))

    def run(n, start_evt=None, end_evt=None):
        ev = lambda: torch.cuda.Event()
        in_ready, comp_done, out_done = [ev() for _ in range(n)], [ev() for _ in range(n)], \
            [ev() for _ in range(n)]
        if start_evt is not None:
            start_evt.record(s_h2d)
        for i in range(n):
            ins, outs, scratch = sets[i % 2]
            with torch.cuda.stream(s_h2d):
                if i >= 2:
                    s_h2d.wait_event(comp_done[i - 2])      # this set's inputs are free again
                for d, h in zip(ins, host_in):
                    d.copy_(h, non_blocking=True)
                in_ready[i].record(s_h2d)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_ready[i])
                if i >= 2:
                    s_cmp.wait_event(out_done[i - 2])       # this set's results were copied out
                make_step(ins, outs, scratch, s_cmp)
                comp_done[i].record(s_cmp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(comp_done[i])
                for h, d in zip(host_out, outs):
                    h.copy_(d, non_blocking=True)
                out_done[i].record(s_d2h)
        if end_evt is not None:
            end_evt.record(s_d2h)

    run(2)
    torch.cuda.synchronize(dev)
    n = max(2, steps)
    _barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run(n, e0, e1)
    torch.cuda.synchronize(dev)
    api.check_status(s_cmp)
    ms = max_over_ranks(e0.elapsed_time(e1)) / n
    h2d = sum(t.numel() * t.element_size() for t in dev_in)
    d2h = sum(t.numel() * t.element_size() for t in dev_out)
    return {"value": world * flops / (ms * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": n,
            "pipelined": "double-buffered; H2D, compute and D2H on separate streams"}


def other_configs(api, dev, seed: int) -> dict:
    """The other problem configurations, timed on the device after the headline's
    timed region (default single-GPU run only): CUDA events on the launching
    stream around `steps` calls after `warmup`, inputs resident, clocks sampled."""
    from ring_attention_02_b300.inputs import TINY, CAUSAL_8K, GQA_128K, MILLION, TRAIN_32K
    peak, _, _ = measured_peaks()
    stream = torch.cuda.current_stream(dev)
    out = {}
    for w, steps, warmup in ((TINY, 200, 5), (CAUSAL_8K, 20, 3), (GQA_128K, 3, 3),
                             (MILLION, 2, 3), (TRAIN_32K, 3, 3)):
        q, k, v = make_for(w, seed=seed, device=dev)
        o = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.float32 if w.out_f32 else torch.bfloat16,
                        device=dev)
        lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
        if w.backward:
            do = make_dout(w.B, w.H, w.S, w.D, seed=seed, device=dev)
            dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]

        def step(i=None):
            if i is not None and w.backward:
                ev[i][0].record(stream)
            api.fwd(q, k, v, w.P, w.layout, w.causal, out=o, lse=lse, stream=stream)
            if w.backward:
                if i is not None:
                    ev[i][1].record(stream)
                api.bwd(q, k, v, o, lse, do, w.P, w.layout, w.causal, dq=dq, dk=dk, dv=dv,
                        stream=stream)
                if i is not None:
                    ev[i][2].record(stream)

        for _ in range(warmup):
            step()
        api.check_status(stream)
        torch.cuda.synchronize(dev)
        with ClockSampler(dev.index or 0) as clk:
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for i in range(steps):
                step(i)
            t1.record(stream)
            torch.cuda.synchronize(dev)
        api.check_status(stream)
        ms = t0.elapsed_time(t1) / steps
        value = w.step_flops() / (ms * 1e-3) / 1e12
        rec = {"layout": w.layout, "causal": w.causal, "steps": steps, "warmup": warmup,
               "ms_per_step": ms, "value": value, "unit": UNIT, "frac": value / peak,
               "clocks": clk.summary()}
        if w.backward:
            f_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / steps
            b_ms = sum(e[1].elapsed_time(e[2]) for e in ev) / steps
            b_tf = 2.5 * w.counted_flops() / (b_ms * 1e-3) / 1e12
            rec.update({"fwd_ms": f_ms, "bwd_ms": b_ms, "bwd_value": b_tf, "bwd_frac": b_tf / peak})
        out[w.name] = rec
        del q, k, v, o, lse
        if w.backward:
            del do, dq, dk, dv
        torch.cuda.empty_cache()
    return out


def run_ours(args, w: Workload, rank: int, world: int):
    from ring_attention_02_b300 import api

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    q, k, v = make_for(w, seed=args.seed + 17 * rank, device=dev)
    out = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    if w.backward:
        do = make_dout(w.B, w.H, w.S, w.D, seed=args.seed + 17 * rank, device=dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    # events: [fwd start, fwd end (= bwd start), bwd end] per timed step of a
    # training workload; a forward-only step is its one launch, timed by the
    # events around the whole region (per-step event records would add host
    # work between the calls of a short one)
    marks = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]

    def step(i=None):
        if i is not None and w.backward:
            marks[i][0].record(stream)
        api.fwd(q, k, v, w.P, w.layout, w.causal, out=out, lse=lse, stream=stream)
        if w.backward:
            if i is not None:
                marks[i][1].record(stream)
            api.bwd(q, k, v, out, lse, do, w.P, w.layout, w.causal, dq=dq, dk=dk, dv=dv,
                    stream=stream)
            if i is not None:
                marks[i][2].record(stream)

    for _ in range(args.warmup):
        step()
    api.check_status(stream)

    # ---- device-resident timed region
    _barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_all0 = torch.cuda.Event(enable_timing=True)
        t_all1 = torch.cuda.Event(enable_timing=True)
        t_all0.record(stream)
        for i in range(args.steps):
            step(i)
        t_all1.record(stream)
        torch.cuda.synchronize(dev)
    _barrier()
    api.check_status(stream)
    total_ms = max_over_ranks(t_all0.elapsed_time(t_all1))
    ms_per_step = total_ms / args.steps
    flops = w.step_flops()
    value = world * flops * args.steps / (total_ms * 1e-3) / 1e12
    fwd_ms = [m[0].elapsed_time(m[1]) for m in marks] if w.backward else [ms_per_step]
    bwd_ms = [m[1].elapsed_time(m[2]) for m in marks] if w.backward else []

    # ---- end to end through host buffers (pinned), C-ABI calls per step
    e2e = None
    if not args.skip_e2e:
        if w.backward:
            def make_step(ins, outs, scratch, st):
                o, l = scratch
                api.fwd(ins[0], ins[1], ins[2], w.P, w.layout, w.causal, out=o, lse=l, stream=st)
                api.bwd(ins[0], ins[1], ins[2], o, l, ins[3], w.P, w.layout, w.causal,
                        dq=outs[0], dk=outs[1], dv=outs[2], stream=st)
            e2e = measure_e2e(w, api, make_step, [q, k, v, do], [dq, dk, dv], [out, lse], dev,
                              flops, world, args.steps)
        else:
            def make_step(ins, outs, scratch, st):
                api.fwd(ins[0], ins[1], ins[2], w.P, w.layout, w.causal, out=outs[0],
                        lse=outs[1], stream=st)
            e2e = measure_e2e(w, api, make_step, [q, k, v], [out, lse], [], dev, flops, world,
                              args.steps)
    if rank != 0:
        return
    peak, peak_sus, peak_src = measured_peaks()
    if w.backward:
        # dominant call: the backward (prep + dK/dV pass + dQ pass)
        dom_ms = sum(bwd_ms) / len(bwd_ms)
        achieved = 2.5 * w.counted_flops() / (dom_ms * 1e-3) / 1e12
        kernel = "ring_attn_bwd: bwd_prep_kernel + attn_bwd_dkdv_kernel + attn_bwd_dq_kernel"
        traffic = None
        launches = 4 * args.steps
    else:
        dom_ms = sum(fwd_ms) / len(fwd_ms)
        achieved = w.counted_flops() / (dom_ms * 1e-3) / 1e12
        kernel = f"attn_fwd_kernel<{w.D}>"
        traffic = traffic_from_profiles(w)
        launches = args.steps
    pairs, tiles = api.census(w.S, w.P, w.layout, w.causal)
    tiles = tiles.double()
    imbalance = float(tiles.max() / tiles.mean() - 1.0)

    # CPU oracle on a bounded sample (rank 0, N=1 only)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        f_s, t_s = 0.0, 0.0
        if w.backward:
            f_s, t_s = oracle_train_sample(w, q, k, v, do, args.ref_prefix)
            sample = (f"fwd+bwd of (b=0, kv head 0) over the first {args.ref_prefix} tokens, "
                      f"{t_s:.1f} s of fp64 C oracle, {f_s:.3g} counted flop")
        else:
            kh, vh = host_kv(k, v)
            while t_s < args.cpu_seconds:
                f, t = oracle_sample(w, q, kh, vh, 64, seed=int(t_s * 1000) + 7)
                f_s += f
                t_s += t
            sample = (f"uniform query rows x {w.B * w.H} (b,h), {t_s:.1f} s of fp64 C oracle, "
                      f"{f_s:.3g} counted flop")
        cpu = {"value": f_s / t_s / 1e12, "unit": UNIT, "cores": cores(), "kind": "oracle",
               "sample": sample, "cpu_model": cpu_model()}
        if w.backward:
            cpu["one_core"] = one_core_baseline(w, q, k, v, do, None, None, args.ref_prefix)
        else:
            cpu["one_core"] = one_core_baseline(w, q, k, v, None, kh, vh, args.ref_prefix)

    line = {
        "metric": metric_of(w), "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_of(w),
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT,
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"bf16 burst {peak_src}", "peak_sustained": peak_sus,
                     "frac_of_sustained": achieved / peak_sus,
                     "frac_of_nominal": achieved / NOMINAL_BF16_TFLOPS,
                     "nominal_peak": NOMINAL_BF16_TFLOPS, "kernel": kernel},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "shard_imbalance": imbalance,
    }
    if w.backward:
        line["fwd_ms"] = sum(fwd_ms) / len(fwd_ms)
        line["bwd_ms"] = sum(bwd_ms) / len(bwd_ms)
    if world == 1 and w.name == HEADLINE.name and not args.headline_only:
        # outside the headline's timed region; the headline's value does not include them
        del q, k, v, out, lse
        torch.cuda.empty_cache()
        line["other_configs"] = other_configs(api, dev, args.seed)
    print(json.dumps(line), flush=True)


def run_op(args, w: Workload, rank: int, world: int):
    """Times ring_attn_permute, ring_attn_merge or the step+merge ring on the
    workload's shapes (device-resident inputs; CUDA events on the stream)."""
    from ring_attention_02_b300 import api

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    n = w.S // w.P
    q, k, v = make_for(w, seed=args.seed + 17 * rank, device=dev)
    hbm_peak, hbm_src = measured_hbm()
    launches_per_step = 1
    if args.op == "permute":
        dst = torch.empty_like(q)
        step = lambda: api.permute(q, w.S, w.P, w.layout, out=dst, stream=stream)
        work = 2.0 * q.numel() * q.element_size()          # bytes read + written
        unit, bound, peak, peak_src = "GB/s", "hbm", hbm_peak, hbm_src
        metric = "ring_attn_permute HBM GB/s (q rows to shard-major order)"
        dtype = "u8"
    elif args.op == "merge":
        g = torch.Generator(device=dev).manual_seed(args.seed + 5)
        oa = torch.randn((w.B, n, w.H, w.D), device=dev, generator=g)
        op = torch.randn((w.B, n, w.H, w.D), device=dev, generator=g)
        la = torch.randn((w.B, w.H, n), device=dev, generator=g)
        lp = torch.randn((w.B, w.H, n), device=dev, generator=g)
        step = lambda: api.merge(oa, la, op, lp, stream=stream)
        rows = w.B * n * w.H
        work = 3.0 * rows * (4 * w.D + 4)                   # read both partials, write one
        unit, bound, peak, peak_src = "GB/s", "hbm", hbm_peak, hbm_src
        metric = "ring_attn_merge HBM GB/s (LSE fold of one shard's fp32 partials)"
        dtype = "f32"
    elif args.op == "decode":
        T = args.decode_tokens
        qd = q[:, w.S - T:].contiguous()
        out_d = torch.empty_like(qd)
        lse_d = torch.empty((w.B, w.H, T), dtype=torch.float32, device=dev)
        step = lambda: api.decode(qd, k, v, w.P, w.layout, out=out_d, lse=lse_d, stream=stream)
        work = 2.0 * k.numel() * k.element_size()             # the cache is read once per step
        unit, bound, peak, peak_src = "GB/s", "hbm", hbm_peak, hbm_src
        metric = f"ring_attn_decode HBM GB/s ({T} new token(s) against the sharded cache)"
        dtype = "bf16"
        launches_per_step = 2
    elif args.op == "varlen":
        # a pack of documents with a seeded length mix, on the workload's heads,
        # head dim, ranks and layout; counted flops per sequence
        from ring_attention_02_b300.inputs import pack_lengths
        mult = 2 * w.P * 128 if w.layout == "zigzag" else w.P * 128
        lengths = pack_lengths(16, 2048, 32768, mult, seed=args.seed)
        total = sum(lengths)
        cu = torch.tensor([0] + np.cumsum(lengths).tolist(), dtype=torch.int64)
        qv, kv_, vv = (t[0] for t in make_qkv(1, w.H, w.Hkv, total, w.D, seed=args.seed,
                                              device=dev))
        out_v = torch.empty_like(qv)
        lse_v = torch.empty((w.H, total), dtype=torch.float32, device=dev)
        step = lambda: api.fwd_varlen(qv, kv_, vv, cu, w.P, w.layout, w.causal, out=out_v,
                                      lse=lse_v, stream=stream)
        work = sum(4.0 * w.H * L * L * w.D / (2 if w.causal else 1) for L in lengths)
        unit, bound = UNIT, "tensor"
        peak, _, peak_src = measured_peaks()
        metric = (f"causal ring-attn fwd over a pack of 16 documents TFLOP/s "
                  f"({total} tokens, lengths {min(lengths)}..{max(lengths)})")
        dtype = "bf16"
    elif args.op == "sp_rank":
        # one rank's forward compute under the two sequence-parallel schemes
        # at R ranks (R = --sp-ranks, default min(P, Hkv): the head-sharded
        # scheme needs Hkv % R == 0), the exchanges left out (one GPU):
        #   ring:    R hops of ring_attn_step on shard 0 plus R-1 merges
        #   Ulysses: the packing kernels around its two all-to-alls and the
        #            fused forward over the whole sequence of H/R heads
        R = args.sp_ranks or min(w.P, w.Hkv)
        if w.S % (2 * R) or w.H % R or w.Hkv % R:
            raise SystemExit(f"--sp-ranks {R} does not divide the workload")
        nr = w.S // R
        sh = lambda t: api.permute(t, w.S, R, w.layout).view(w.B, R, nr, *t.shape[2:])
        q0 = sh(q)[:, 0].contiguous()
        kvs = [(sh(k)[:, s_].contiguous(), sh(v)[:, s_].contiguous()) for s_ in range(R)]
        acc_o = torch.empty((w.B, nr, w.H, w.D), dtype=torch.float32, device=dev)
        acc_l = torch.empty((w.B, w.H, nr), dtype=torch.float32, device=dev)
        part_o, part_l = torch.empty_like(acc_o), torch.empty_like(acc_l)
        Hg, Hkg = w.H // R, w.Hkv // R
        qf = torch.empty((w.B, w.S, Hg, w.D), dtype=torch.bfloat16, device=dev)
        kf = torch.empty((w.B, w.S, Hkg, w.D), dtype=torch.bfloat16, device=dev)
        vf = torch.empty_like(kf)
        of = torch.empty_like(qf)
        lf = torch.empty((w.B, Hg, w.S), dtype=torch.float32, device=dev)
        k0, v0 = kvs[0]
        blk_q, blk_k, blk_v = torch.empty_like(q0), torch.empty_like(k0), torch.empty_like(k0)
        blk_o = torch.empty_like(qf)
        out_s = torch.empty_like(q0)

        def ring_rank():
            api.step(q0, kvs[0][0], kvs[0][1], w.S, R, w.layout, 0, 0, w.causal, out=acc_o,
                     lse=acc_l, stream=stream)
            for t in range(1, R):
                s_ = (-t) % R
                api.step(q0, kvs[s_][0], kvs[s_][1], w.S, R, w.layout, 0, s_, w.causal,
                         out=part_o, lse=part_l, stream=stream)
                api.merge(acc_o, acc_l, part_o, part_l, stream=stream)

        def ulysses_rank():
            # send side: head groups of the local shard; receive side: the
            # whole sequence of one head group (the all-to-all in between is
            # the exchange, not timed here)
            api.head_split(q0, w.B * nr, R, out=blk_q, stream=stream)
            api.head_split(k0, w.B * nr, R, out=blk_k, stream=stream)
            api.head_split(v0, w.B * nr, R, out=blk_v, stream=stream)
            api.permute_shards(blk_q.view(R, w.B, nr, Hg, w.D), w.S, R, w.layout, inverse=True,
                               out=qf, stream=stream)
            api.permute_shards(blk_k.view(R, w.B, nr, Hkg, w.D), w.S, R, w.layout, inverse=True,
                               out=kf, stream=stream)
            api.permute_shards(blk_v.view(R, w.B, nr, Hkg, w.D), w.S, R, w.layout, inverse=True,
                               out=vf, stream=stream)
            api.fwd(qf, kf, vf, 1, "contiguous", w.causal, out=of, lse=lf, stream=stream)
            api.permute_shards(of, w.S, R, w.layout, out=blk_o, stream=stream)
            api.head_split(blk_o.view(R, w.B * nr, Hg * w.D), w.B * nr, R, inverse=True,
                           out=out_s, stream=stream)

        def timed(fn, reps):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize(dev)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(reps):
                fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            return a.elapsed_time(b) / reps

        with ClockSampler(local) as clk:
            ring_ms = timed(ring_rank, args.steps)
            uly_ms = timed(ulysses_rank, args.steps)
        api.check_status(stream)
        if rank != 0:
            return
        rank_flops = w.counted_flops() / R
        kv_bytes = 2 * w.B * nr * w.Hkv * w.D * 2
        line = {
            "metric": "per-rank forward compute, ring vs head-sharded (Ulysses), ms",
            "value": ring_ms, "unit": "ms", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ring_ms, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {**config_of(w), "op": args.op, "ranks": R},
            "ring": {"ms": ring_ms, "tflops": rank_flops / (ring_ms * 1e-3) / 1e12,
                     "calls": f"{R} ring_attn_step + {R - 1} ring_attn_merge on shard 0",
                     "bytes_sent_per_rank": (R - 1) * kv_bytes},
            "ulysses": {"ms": uly_ms, "tflops": rank_flops / (uly_ms * 1e-3) / 1e12,
                        "calls": "head_split x4, permute_shards x4, ring_attn_fwd (P=1)",
                        "bytes_sent_per_rank": (R - 1) * (w.B * nr * (2 * w.H + 2 * w.Hkv)
                                                          * w.D * 2) // R},
            "roofline": None, "cpu_baseline": None, "e2e": None,
            "gpu_launches": args.steps * (2 * R - 1 + 9), "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
        return
    else:
        qs = api.permute(q, w.S, w.P, w.layout).view(w.B, w.P, n, w.H, w.D)
        ks = api.permute(k, w.S, w.P, w.layout).view(w.B, w.P, n, w.Hkv, w.D)
        vs = api.permute(v, w.S, w.P, w.layout).view(w.B, w.P, n, w.Hkv, w.D)
        qs = [qs[:, r].contiguous() for r in range(w.P)]
        ks = [ks[:, r].contiguous() for r in range(w.P)]
        vs = [vs[:, r].contiguous() for r in range(w.P)]
        acc_o = torch.empty((w.B, n, w.H, w.D), dtype=torch.float32, device=dev)
        acc_l = torch.empty((w.B, w.H, n), dtype=torch.float32, device=dev)
        part_o, part_l = torch.empty_like(acc_o), torch.empty_like(acc_l)

        def step():
            for r in range(w.P):
                api.step(qs[r], ks[r], vs[r], w.S, w.P, w.layout, r, r, w.causal, out=acc_o,
                         lse=acc_l, stream=stream)
                for t in range(1, w.P):
                    s_blk = (r - t) % w.P
                    api.step(qs[r], ks[s_blk], vs[s_blk], w.S, w.P, w.layout, r, s_blk,
                             w.causal, out=part_o, lse=part_l, stream=stream)
                    api.merge(acc_o, acc_l, part_o, part_l, stream=stream)
        work = w.counted_flops()
        unit, bound = UNIT, "tensor"
        peak, _, peak_src = measured_peaks()
        metric = "causal ring-attn step+merge ring TFLOP/s (bf16, per-hop calls, 1 B300)"
        dtype = "bf16"
        launches_per_step = w.P * w.P + w.P * (w.P - 1)
    for _ in range(args.warmup):
        step()
    api.check_status(stream)
    _barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    _barrier()
    api.check_status(stream)
    ms = max_over_ranks(e0.elapsed_time(e1)) / args.steps
    scale = 1e9 if unit == "GB/s" else 1e12
    value = world * work / (ms * 1e-3) / scale
    if rank != 0:
        return
    achieved = work / (ms * 1e-3) / scale
    line = {
        "metric": metric, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": {**config_of(w), "op": args.op},
        "roofline": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": None, "peak_source": peak_src,
                     "work_per_launch": work},
        "cpu_baseline": None,
        "e2e": None,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
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
    ap.add_argument("--ref-prefix", type=int, default=12288,
                    help="training workloads: tokens of the oracle's fwd+bwd sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the other configurations the default single-GPU run adds")
    ap.add_argument("--decode-tokens", type=int, default=1, help="--op decode: new tokens T")
    ap.add_argument("--sp-ranks", type=int, default=0,
                    help="--op sp_rank: ranks of the two schemes (default min(P, Hkv))")
    ap.add_argument("--op", choices=["fwd", "permute", "merge", "step_merge", "decode", "varlen",
                                     "sp_rank"],
                    default="fwd",
                    help="fwd: the workload's step (default); the others time one call")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = by_name(args.workload)
    if args.layout is not None and args.layout != w.layout:
        w = w.with_layout(args.layout)
    rank, world = _dist()
    if args.impl == "reference":
        run_reference(args, w, rank)
    elif args.op != "fwd":
        run_op(args, w, rank, world)
    else:
        run_ours(args, w, rank, world)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
