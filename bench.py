#!/usr/bin/env python3
"""Benchmark of the attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step = one pass of the hot path over one batch of the workload: every
mask mode the workload is run with (s4096: non-causal and causal), each one
call of the C-ABI entry point fa_fwd_splitkv (which splits the keys of each
query block over several CTAs when the shape would leave SMs idle, and then
launches the merge kernel as a second launch).  Metric: attention forward TFLOP/s, counting
4*B*H*S^2*D FLOPs per call (half when causal), and its fraction of the
measured dense bf16/fp16 tensor peak.

value      device time: CUDA events on the launching stream around each
           step, L2 flushed (256 MB write) before every timed step, inputs
           resident in HBM.
e2e        the same metric through the C-ABI with host buffers: per step the
           pinned-host -> device copies of Q, K, V, the calls, and the
           device -> pinned-host copies of O and LSE, timed with events.
roofline   the dominant kernel (the only kernel of the path) against the
           measured tensor peak; traffic is read from the committed ncu
           summary when it was taken on the current kernel sources.
cpu_baseline  the fp64 oracle as it stands on the host cores, on a bounded
           sample of the same workload.

--impl reference times the oracle alone (the reference arm) on the same
workload, metric and unit.  With N > 1 (torchrun) every rank runs an
independent replica (the path has no exchange step); value is the sum over
ranks of the FLOPs divided by the slowest rank's time.
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

import numpy as np  # noqa: E402

import fa_inputs  # noqa: E402

DEFAULT_WORKLOAD = "s4096"
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    return 1900.0, 1700.0, "fallback"


def _kernel_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_fwd_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def _traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources and this workload; else None."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    entry = d.get(workload)
    if not entry or entry.get("kernel_sha") != _kernel_sha():
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]),
                                 hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------- oracle
def cpu_baseline(w: fa_inputs.Workload, budget_s: float = 15.0, inputs=None):
    """Time the fp64 oracle on a bounded sample of the workload: whole heads
    (all rows, every mask mode of the workload) one after another, cycling
    over the workload's heads, until ``budget_s`` seconds are spent (at least
    one head)."""
    from oracle import attention_rows
    qb, kb, vb = inputs if inputs is not None else fa_inputs.make_qkv_for(w)
    flops = 0.0
    heads = 0
    rows = np.arange(w.S)
    order = [(b, h) for b in range(w.B) for h in range(w.H)]
    t0 = time.perf_counter()
    while True:
        b, h = order[heads % len(order)]
        for causal in w.modes:
            attention_rows(qb, kb, vb, w.dtype, causal, w.scale, b, h, rows)
            flops += fa_inputs.attention_flops(1, 1, w.S, w.D, causal)
        heads += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{heads} (b,h) heads of {w.name} ({w.B * w.H} in the workload), all "
                      f"{w.S} rows, modes {['causal' if c else 'non-causal' for c in w.modes]}; "
                      f"fp64 numpy, BLAS threads = cores; {dt:.1f} s"}


def run_reference(args, w):
    world, rank, _ = _dist_env()
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        pass  # the oracle has no warm state; warm-up steps are not needed
    times = []
    cb = None
    inputs = fa_inputs.make_qkv_for(w)
    # keep the whole run within a couple of minutes whatever --steps is
    per_step = max(0.5, min(args.ref_budget, 120.0 / max(1, args.steps)))
    for _ in range(args.steps):
        cb = cpu_baseline(w, budget_s=per_step, inputs=inputs)
        times.append(cb["value"])
    value = statistics.median(times)
    cb["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D,
                       "modes": ["causal" if c else "non-causal" for c in w.modes]},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


METRIC = "attention fwd TFLOP/s and % of GB300 dense FP16/BF16 tensor peak, 1 GPU"


# ----------------------------------------------------------------------- ours
def run_ours(args, w):
    import torch
    import attention_forward_fwd_gb300 as fa

    world, rank, local = _dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    fa.build()
    lib = fa.library()

    qb, kb, vb = fa_inputs.make_qkv_for(w)
    tq, tk, tv = (fa_inputs.to_torch(x, w.dtype) for x in (qb, kb, vb))
    q, k, v = (t.to(dev) for t in (tq, tk, tv))
    modes = list(w.modes)
    outs = [torch.empty_like(q) for _ in modes]
    lses = [torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev) for _ in modes]
    dtype_code = fa.FA_F16 if w.dtype == "f16" else fa.FA_BF16
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    # split-over-keys workspace (0 bytes when the shape fills the GPU)
    ws_bytes = max(fa.fa_splitkv_workspace_size(w.B, w.H, w.S, w.D, c) for c in modes)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def call(qp, kp, vp, o, lse, causal):
        rc = lib.fa_fwd_splitkv(qp, kp, vp, o.data_ptr(), lse.data_ptr(), w.B, w.H, w.S, w.D,
                                int(causal), w.scale, dtype_code, ws.data_ptr(), ws.numel(), sp)
        if rc != 0:
            raise fa.FaError(rc, "fa_fwd_splitkv")

    def step():
        for causal, o, lse in zip(modes, outs, lses):
            call(q.data_ptr(), k.data_ptr(), v.data_ptr(), o, lse, causal)

    flops_step = sum(fa_inputs.attention_flops(w.B, w.H, w.S, w.D, c) for c in modes)
    launches_per_step = sum(fa.fa_splitkv_launches(w.B, w.H, w.S, w.D, c) for c in modes)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.fill_(1.0)
            step()
    torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                flush.fill_(float(i))          # evict Q, K, V, O from L2
                starts[i].record(stream)
                step()
                ends[i].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = sum(step_ms)
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / args.steps
    value = world * flops_step * args.steps / (total_ms * 1e-3) / 1e12
    status = fa.fa_device_status(clear=False)
    if status != 0:
        raise RuntimeError(f"device status {status}: {fa.fa_status_string(status)}")

    # ------------------------------------------------ end to end (host buffers)
    e2e = None
    if not args.no_e2e:
        hq, hk, hv = (t.pin_memory() for t in (tq, tk, tv))
        ho = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in modes]
        hl = [torch.empty((w.B, w.H, w.S), dtype=torch.float32).pin_memory() for _ in modes]
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        h2d = 3 * q.numel() * q.element_size()
        d2h = len(modes) * (q.numel() * q.element_size() + w.B * w.H * w.S * 4)

        def e2e_step():
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            for causal, o, lse, h_o, h_l in zip(modes, outs, lses, ho, hl):
                call(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o, lse, causal)
                h_o.copy_(o, non_blocking=True)
                h_l.copy_(lse, non_blocking=True)

        e2e_steps = max(3, min(args.steps, 50))
        with torch.cuda.stream(stream):
            for _ in range(3):
                e2e_step()
            torch.cuda.synchronize(dev)
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(e2e_steps):
                e2e_step()
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = ev0.elapsed_time(ev1) / e2e_steps
        e2e = {"value": world * flops_step / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "steps": e2e_steps}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    peak, peak_sust, peak_kind = _peaks()
    achieved = flops_step / (ms_per_step * 1e-3) / 1e12     # one GPU, kernel time
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": _traffic(w.name),
                "peak_kind": f"{peak_kind} bf16 burst (fp16 has the same dense rate)",
                "kernel": "fa::fa_fwd_kernel (+ fa::fa_combine_kernel when split; timed together)",
                "algorithmic_flops_per_step": flops_step,
                "launches_per_step": launches_per_step}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "D": w.D,
                       "modes": ["causal" if c else "non-causal" for c in modes],
                       "scale": w.scale, "layout": "[B,S,H,D]",
                       "l2": "flushed (256 MB write) before every timed step",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "pct_of_peak": 100.0 * achieved / peak,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
            "roofline": roofline,
            "e2e": e2e,
            "wall_s_timed_region": t_wall}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
    if args.all_workloads:
        line["other_workloads"] = other_workloads(lib, fa, dev, stream, flush, w.name, peak)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def other_workloads(lib, fa, dev, stream, flush, skip, peak):
    """Kernel-timed TFLOP/s of every other workload and mode (informational)."""
    import torch
    res = {}
    for name, w in fa_inputs.WORKLOADS.items():
        if name == skip:
            continue
        qb, kb, vb = fa_inputs.make_qkv_for(w)
        q, k, v = (fa_inputs.to_torch(x, w.dtype).to(dev) for x in (qb, kb, vb))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
        code = fa.FA_F16 if w.dtype == "f16" else fa.FA_BF16
        nws = max(fa.fa_splitkv_workspace_size(w.B, w.H, w.S, w.D, c) for c in w.modes)
        ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
        for causal in w.modes:
            ms = []
            with torch.cuda.stream(stream):
                for i in range(13):
                    flush.fill_(float(i))
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    rc = lib.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                            o.data_ptr(), lse.data_ptr(), w.B, w.H, w.S, w.D,
                                            int(causal), w.scale, code, ws.data_ptr(),
                                            ws.numel(), stream.cuda_stream)
                    e1.record(stream)
                    assert rc == 0
                    if i >= 3:
                        ms.append((e0, e1))
            torch.cuda.synchronize(dev)
            t = statistics.median(a.elapsed_time(b) for a, b in ms)
            tf = fa_inputs.attention_flops(w.B, w.H, w.S, w.D, causal) / (t * 1e-3) / 1e12
            res[f"{name}/{'causal' if causal else 'non-causal'}"] = {
                "ms": t, "tflops": tf, "pct_of_peak": 100.0 * tf / peak,
                "launches": fa.fa_splitkv_launches(w.B, w.H, w.S, w.D, causal)}
        del q, k, v, o, lse, ws
    return res


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[1])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(fa_inputs.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--all-workloads", action="store_true",
                    help="also time every other workload (informational)")
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=10.0,
                    help="seconds of oracle work per reference-arm step")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    w = fa_inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
