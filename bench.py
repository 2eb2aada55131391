#!/usr/bin/env python3
"""Benchmark of the attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

One step = one pass of the hot path over one batch of the workload: every
mask mode the workload is run with (the default b2h16d128 -- B2 H16 S8192
D128 bf16, the largest single-GPU configuration -- non-causal and causal),
each one call of the C-ABI entry point fa_fwd_gqa_splitkv (which splits the
keys of each query block over several CTAs when the shape would leave SMs
idle, and then merges the partial results).  Metric: attention forward TFLOP/s, counting
4*B*H*S^2*D FLOPs per call (half when causal), and its fraction of the
measured dense bf16/fp16 tensor peak.

value      device time: CUDA events on the launching stream around each
           step, L2 flushed (256 MB write) before every timed step, inputs
           resident in HBM.
e2e        the same metric through the C-ABI with host buffers: per step one
           pinned-host -> device copy of Q, K, V, the calls, and one
           device -> pinned-host copy of O and LSE, timed with events; the
           copies run on streams of their own and overlap the neighbouring
           steps' kernels (the one-stream figure is reported as serial_value).
roofline   the dominant kernel (the only kernel of the path) against the
           measured tensor peak; traffic is read from the committed ncu
           summary when it was taken on the current kernel sources.
cpu_baseline  the fp64 oracle as it stands on the host cores, on a bounded
           sample of the same workload; with the host's CPU model and the
           oracle on one thread over the S = 256 workload.

configs    kernel-timed TFLOP/s of the other four target configurations (s256,
           s4096, b4h16, stress; every mask mode), L2 flushed before each
           call; --all-workloads adds grouped K/V heads, packed batches,
           windows, dropout and other head dimensions.

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

DEFAULT_WORKLOAD = "b2h16d128"
# the five target configurations (the headline is one of them)
TARGET_WORKLOADS = ("s256", "s4096", "b4h16", "b2h16d128", "stress")
L2_FLUSH_BYTES = 256 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    return 1900.0, 1700.0, "fallback"


# the sources of fa_fwd_kernel / fa_combine_kernel and their launch (the
# profiled kernels); the wide kernel for D > 128 has a file of its own
KERNEL_SOURCES = ("fa_api.cu", "fa_fwd_kernel.cuh", "sm103_ptx.cuh")


def _kernel_sha():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_forward_fwd_gb300", "csrc")
    for name in KERNEL_SOURCES:
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
    """SM clock / clock-event-reason sampling while the timed region runs.

    A thread reads NVML (libnvidia-ml through ctypes, read-only queries)
    about every millisecond for the GPU with the CUDA device's UUID, so even a
    region of a few milliseconds gets samples; nvidia-smi is the fallback.
    """

    # NVML clock-event reason bits
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.rows = []
        self.source = None
        self._nvml = self._open_nvml()

    def _open_nvml(self):
        import ctypes
        try:
            import torch
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.gpu).uuid)
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return None
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
                return None
            get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) != 0:   # NVML_CLOCK_SM
                return None
            return dict(lib=lib, h=h, reasons=get_reasons, max=mx.value, c=ctypes)
        except Exception:
            return None

    def _poll(self):
        n = self._nvml
        c, lib, h = n["c"], n["lib"], n["h"]
        clk, pw, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        while not self._stop.is_set():
            if (lib.nvmlDeviceGetClockInfo(h, 1, c.byref(clk)) == 0 and
                    n["reasons"](h, c.byref(rs)) == 0):
                lib.nvmlDeviceGetPowerUsage(h, c.byref(pw))
                self.rows.append(dict(sm=float(clk.value), smax=float(n["max"]),
                                      reasons=int(rs.value), power_w=pw.value / 1000.0))
            time.sleep(0.001)

    def __enter__(self):
        import threading
        if self._nvml is not None:
            self.source = "nvml"
            self._stop = threading.Event()
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
            time.sleep(0.005)       # a first sample before the region starts
            return self
        self.source = "nvidia-smi"
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.source == "nvml":
            self._stop.set()
            self._thread.join(timeout=5)
            return
        out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in (out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                bits = 0
                for name, flag in zip(names, parts[5:9]):
                    if flag.lower() == "active":
                        bits |= next(b for b, nm in self.REASONS.items() if nm == name)
                self.rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), reasons=bits,
                                      power_w=float(parts[3]) if parts[3] else 0.0))
            except ValueError:
                continue

    def summary(self):
        rows = self.rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "source": self.source}
        reasons = set()
        for r in rows:
            for bit, name in self.REASONS.items():
                if r["reasons"] & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power_w"] for r in rows), "source": self.source}


def _dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# --------------------------------------------------------------------- oracle
class _Driver:
    """The few CUDA driver calls the end-to-end loop issues per step."""

    def __init__(self):
        import ctypes
        self._c = ctypes
        lib = ctypes.CDLL("libcuda.so.1")
        u64, vp, sz, u32 = ctypes.c_uint64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint
        self._h2d = lib.cuMemcpyHtoDAsync_v2
        self._h2d.argtypes = [u64, vp, sz, vp]
        self._d2h = lib.cuMemcpyDtoHAsync_v2
        self._d2h.argtypes = [vp, u64, sz, vp]
        self._rec = lib.cuEventRecord
        self._rec.argtypes = [vp, vp]
        self._wait = lib.cuStreamWaitEvent
        self._wait.argtypes = [vp, vp, u32]
        self._create = lib.cuEventCreate
        self._create.argtypes = [ctypes.POINTER(vp), u32]
        self._events = []

    @staticmethod
    def _check(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} failed with CUDA driver error {rc}")

    def event(self):
        e = self._c.c_void_p()
        self._check(self._create(self._c.byref(e), 2), "cuEventCreate")   # no timing
        self._events.append(e)
        return e

    def h2d(self, dst, src, n, stream):
        self._check(self._h2d(dst, src, n, stream), "cuMemcpyHtoDAsync")

    def d2h(self, dst, src, n, stream):
        self._check(self._d2h(dst, src, n, stream), "cuMemcpyDtoHAsync")

    def record(self, ev, stream):
        self._check(self._rec(ev, stream), "cuEventRecord")

    def wait(self, stream, ev):
        self._check(self._wait(stream, ev, 0), "cuStreamWaitEvent")


# A head's query rows are taken in blocks of two mirrored chunks (chunk k and
# chunk n-1-k of n = CPU_CHUNKS), so that under the causal mask every block
# holds about the same work.
CPU_CHUNKS = 16


def _row_flops(rows: np.ndarray, S: int, D: int, causal: bool) -> float:
    """Counted FLOPs of query rows `rows` of one head: the workload's
    convention (4 S^2 D, half when causal) shared out over the rows, in
    proportion to the keys each row sees; all S rows sum to it exactly."""
    if causal:
        return 4.0 * D * S / (S + 1) * float(np.sum(rows + 1))
    return 4.0 * D * S * len(rows)


def _row_blocks(S: int):
    c = -(-S // CPU_CHUNKS)
    chunks = [np.arange(a, min(S, a + c)) for a in range(0, S, c)]
    n = len(chunks)
    return [np.concatenate([chunks[k], chunks[n - 1 - k]]) if k != n - 1 - k else chunks[k]
            for k in range((n + 1) // 2)], c


def cpu_baseline(w: fa_inputs.Workload, budget_s: float = 15.0, inputs=None):
    """Time the fp64 oracle on a bounded sample of the workload: blocks of
    query rows (two mirrored chunks of S / CPU_CHUNKS rows of one head, every
    mask mode of the workload) one after another, cycling over the blocks of
    every head, until ``budget_s`` seconds are spent (at least one block)."""
    from oracle import attention_rows
    qb, kb, vb = inputs if inputs is not None else fa_inputs.make_qkv_for(w)
    blocks, chunk = _row_blocks(w.S)
    order = [(b, h, rows) for b in range(w.B) for h in range(w.H) for rows in blocks]
    flops = 0.0
    done = 0
    t0 = time.perf_counter()
    while True:
        b, h, rows = order[done % len(order)]
        for causal in w.modes:
            attention_rows(qb, kb, vb, w.dtype, causal, w.scale, b, h, rows)
            flops += _row_flops(rows, w.S, w.D, causal)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    heads = len({(b, h) for b, h, _ in order[:min(done, len(order))]})
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} row blocks of {w.name} (rows of two mirrored {chunk}-row chunks of one "
                      f"(b,h) head, {len(blocks)} blocks per head; {heads} of the workload's "
                      f"{w.B * w.H} heads touched), modes "
                      f"{['causal' if c else 'non-causal' for c in w.modes]}; "
                      f"fp64 numpy, BLAS threads = cores; {dt:.1f} s"}


def _cpu_model() -> str:
    """The host CPU's model name, as the kernel reports it (x86 and Arm)."""
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "CPU part"):
        for line in text.splitlines():
            if line.split(":")[0].strip() == key:
                return f"{key}: {line.split(':', 1)[1].strip()}"
    return "unknown"


def cpu_baseline_one_thread(workload: str = "s256", budget_s: float = 1.0):
    """The oracle on one host thread: a child process with the BLAS thread
    pools set to one before numpy loads, on a bounded sample of `workload`."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench, fa_inputs; "
            "print(json.dumps(bench.cpu_baseline(fa_inputs.WORKLOADS[%r], budget_s=%r)))"
            % (ROOT, workload, float(budget_s)))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=300)
    if r.returncode != 0:
        return {"error": (r.stderr.strip().splitlines() or ["exit %d" % r.returncode])[-1]}
    out = json.loads(r.stdout.strip().splitlines()[-1])
    out["cores"] = 1
    out["sample"] = out["sample"].replace("BLAS threads = cores", "BLAS threads = 1")
    return out


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x (the slowest rank sets the job's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_rank: float, max_ms: float) -> float:
    """TFLOP/s of all ranks together: every rank did flops_per_rank in at
    most max_ms (replicas: the work grows with the ranks, weak scaling)."""
    return world * flops_per_rank / (max_ms * 1e-3) / 1e12


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
        rc = lib.fa_fwd_gqa_splitkv(qp, kp, vp, o.data_ptr(), lse.data_ptr(), w.B, w.H, w.kv_heads,
                                    w.S, w.D,
                                int(causal), w.scale, dtype_code, ws.data_ptr(), ws.numel(), sp)
        if rc != 0:
            raise fa.FaError(rc, "fa_fwd_gqa_splitkv")

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
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps
    value = whole_job_tflops(world, flops_step * args.steps, total_ms)
    status = fa.fa_device_status(clear=False)
    if status != 0:
        raise RuntimeError(f"device status {status}: {fa.fa_status_string(status)}")

    # ------------------------------------------------ end to end (host buffers)
    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(args, w, lib, fa, dev, stream, tq, tk, tv, modes, dtype_code, ws, world,
                         flops_step)

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    peak, peak_sust, peak_kind = _peaks()
    clk_summary = clk.summary()
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
            "pct_of_theoretical": _theoretical(achieved, clk_summary, dev),
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk_summary,
            "roofline": roofline,
            "e2e": e2e,
            "wall_s_timed_region": t_wall}
    line["pages_protocol"] = pages_protocol(step, stream, dev, flops_step)
    # which kernel sources produced the line (the hash the traffic table is keyed on)
    line["kernel_sha"] = _kernel_sha()
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
        line["cpu_baseline"]["cpu_model"] = _cpu_model()
        line["cpu_baseline"]["one_thread_s256"] = cpu_baseline_one_thread("s256")
    if not args.no_configs:
        line["configs"] = other_workloads(lib, fa, dev, stream, flush, w.name, peak,
                                          names=TARGET_WORKLOADS, extras=False)
    if args.all_workloads:
        line["other_workloads"] = other_workloads(
            lib, fa, dev, stream, flush, w.name, peak,
            names=[n for n in fa_inputs.WORKLOADS if n not in TARGET_WORKLOADS], extras=True)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


# dense fp16 / bf16 tensor work per SM and clock on sm_10x: one M128 N128 K16
# MMA (2 * 128 * 128 * 16 FLOPs) every 64 cycles
FLOP_PER_CLK_PER_SM = 8192


def _theoretical(achieved, clocks, dev):
    """achieved as a % of SMs x clock x 8192 FLOP/clk, at the maximum SM clock
    and at the median clock sampled during the timed region."""
    import torch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    out = {"flop_per_clk_per_sm": FLOP_PER_CLK_PER_SM, "sms": sms}
    for key, mhz in (("at_max_clock", clocks.get("sm_max_mhz")), ("at_sampled_clock", clocks.get("sm_mhz"))):
        if mhz:
            tf = sms * mhz * 1e6 * FLOP_PER_CLK_PER_SM / 1e12
            out[key] = {"sm_mhz": mhz, "tflops": tf, "pct": 100.0 * achieved / tf}
        else:
            out[key] = None
    return out


def pages_protocol(step, stream, dev, flops_step, forwards=100, rounds=9):
    """The timing protocol of the pages (section 正确性、编译与计时方法 of
    page "CuTe 详解：以 FlashAttention-2 拆解 Layout、TiledCopy 与 TiledMMA"):
    a CUDA graph of `forwards` steps replayed `rounds` times, median with min
    and max.  The inputs stay in L2 between forwards here, unlike the main
    timing, so this is context for the pages' own table, not the metric."""
    import torch
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(forwards):
                step()
        ms = []
        with torch.cuda.stream(stream):   # the replays run on the current stream
            g.replay()
            torch.cuda.synchronize(dev)
            for _ in range(rounds):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                g.replay()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                ms.append(e0.elapsed_time(e1) / forwards)
        del g
    except Exception as exc:   # capture is optional context: report, do not fail the run
        return {"error": f"{type(exc).__name__}: {exc}"[:300]}
    tf = [flops_step / (m * 1e-3) / 1e12 for m in ms]
    return {"what": f"CUDA graph of {forwards} steps, {rounds} replays, L2 warm",
            "us_per_step_median": statistics.median(ms) * 1000, "tflops_median": statistics.median(tf),
            "tflops_min": min(tf), "tflops_max": max(tf)}


def end_to_end(args, w, lib, fa, dev, stream, tq, tk, tv, modes, dtype_code, ws, world, flops_step):
    """The metric through the C-ABI with host buffers, as a serving loop runs it.

    Per step: one pinned-host -> device copy of the step's Q, K, V (packed in
    one buffer), the calls (every mode), and one device -> pinned-host copy
    of the step's O and LSE (packed likewise).  The uploads and downloads
    run on streams of their own with two device buffer slots, so that step
    i+1's upload and step i's download overlap step i's kernels; events
    order the slots.  The same loop with every operation on one stream is
    reported beside it as `serial_*`.
    """
    import torch
    n_in = tq.numel()
    n_kv = tk.numel()       # K and V (fewer heads than Q when grouped)
    elt = tq.element_size()
    n_all = n_in + 2 * n_kv
    h_in = torch.empty(n_all, dtype=tq.dtype).pin_memory()
    for off, t in ((0, tq), (n_in, tk), (n_in + n_kv, tv)):
        h_in[off:off + t.numel()].copy_(t.reshape(-1))
    o_bytes = n_in * elt
    l_bytes = (w.B * w.H * w.S * 4 + 255) // 256 * 256   # keeps the next O 16-byte aligned
    out_bytes = len(modes) * (o_bytes + l_bytes)
    d_in = [torch.empty(n_all, dtype=tq.dtype, device=dev) for _ in range(2)]
    d_out = [torch.empty(out_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    h_out = [torch.empty(out_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]

    def run_calls(slot, st):
        base_in = d_in[slot].data_ptr()
        base_out = d_out[slot].data_ptr()
        for m, causal in enumerate(modes):
            o_ptr = base_out + m * (o_bytes + l_bytes)
            rc = lib.fa_fwd_gqa_splitkv(base_in, base_in + n_in * elt, base_in + (n_in + n_kv) * elt,
                                        o_ptr, o_ptr + o_bytes, w.B, w.H, w.kv_heads, w.S, w.D,
                                        int(causal), w.scale,
                                    dtype_code, ws.data_ptr(), ws.numel(), st.cuda_stream)
            if rc != 0:
                raise fa.FaError(rc, "fa_fwd_gqa_splitkv")

    # copies, event records and stream waits go straight to the CUDA driver
    # (a few hundred ns each; the torch wrappers cost microseconds per call)
    drv = _Driver()
    up = torch.cuda.Stream(device=dev)
    down = torch.cuda.Stream(device=dev)
    s_up, s_down, s_comp = up.cuda_stream, down.cuda_stream, stream.cuda_stream
    uploaded = [drv.event() for _ in range(2)]
    computed = [drv.event() for _ in range(2)]
    downloaded = [drv.event() for _ in range(2)]
    in_bytes = n_all * elt

    def pipelined_step(i):
        sl = i % 2
        drv.wait(s_up, computed[sl])             # the slot's previous inputs are consumed
        drv.h2d(d_in[sl].data_ptr(), h_in.data_ptr(), in_bytes, s_up)
        drv.record(uploaded[sl], s_up)
        drv.wait(s_comp, uploaded[sl])
        drv.wait(s_comp, downloaded[sl])         # the slot's previous outputs are read
        run_calls(sl, stream)
        drv.record(computed[sl], s_comp)
        drv.wait(s_down, computed[sl])
        drv.d2h(h_out[sl].data_ptr(), d_out[sl].data_ptr(), out_bytes, s_down)
        drv.record(downloaded[sl], s_down)

    def serial_step(i):
        drv.h2d(d_in[0].data_ptr(), h_in.data_ptr(), in_bytes, s_comp)
        run_calls(0, stream)
        drv.d2h(h_out[0].data_ptr(), d_out[0].data_ptr(), out_bytes, s_comp)

    def timed(step_fn, n):
        for i in range(3):
            step_fn(i)
        torch.cuda.synchronize(dev)
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        up.wait_event(ev0)
        down.wait_event(ev0)
        for i in range(n):
            step_fn(i)
        stream.wait_stream(down)                 # the last download is inside the region
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        return ev0.elapsed_time(ev1) / n

    n = max(3, min(args.steps, 50))
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(timed(pipelined_step, n), world, dev)
    serial_ms = max_over_ranks(timed(serial_step, n), world, dev)
    # the downloaded result is the kernels' output
    got = h_out[(n - 1) % 2][:o_bytes].view(tq.dtype)
    if not torch.isfinite(got.float()).all():
        raise RuntimeError("end-to-end output is not finite")
    return {"value": whole_job_tflops(world, flops_step, ms), "unit": "TFLOP/s",
            "h2d_bytes_per_step": n_all * elt, "d2h_bytes_per_step": out_bytes,
            "ms_per_step": ms, "steps": n,
            "copies": "one packed upload and one packed download per step on their own "
                      "streams, two buffer slots (overlapping the neighbouring steps' kernels)",
            "serial_value": whole_job_tflops(world, flops_step, serial_ms),
            "serial_ms_per_step": serial_ms}


def other_workloads(lib, fa, dev, stream, flush, skip, peak, names, extras):
    """Kernel-timed TFLOP/s of the workloads `names` but `skip`, every mask
    mode, L2 flushed before each call (median of 10 after 3 warm-ups); with
    `extras`, also the packed, windowed, dropout and head-dimension shapes."""
    import torch
    res = {}
    for name in names:
        w = fa_inputs.WORKLOADS[name]
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
                    rc = lib.fa_fwd_gqa_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                o.data_ptr(), lse.data_ptr(), w.B, w.H, w.kv_heads,
                                                w.S, w.D, int(causal), w.scale, code, ws.data_ptr(),
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
    if not extras:
        return res
    res.update(varlen_workload(lib, fa, dev, stream, flush, peak))
    res.update(window_workload(lib, fa, dev, stream, flush, peak))
    res.update(dropout_workloads(lib, fa, dev, stream, flush, peak))
    res.update(head_dim_workloads(lib, fa, dev, stream, flush, peak))
    return res


# Head dimensions other than 64 / 128 (they run on the next kernel up, the
# extra columns read as zeros): B4 H16 S4096 causal at D = 32 (fp16) and
# D = 96 and D = 256 (bf16); FLOPs counted with the caller's D.
HEAD_DIMS = ((32, "f16", 1010), (96, "bf16", 1011), (256, "bf16", 1012))


def head_dim_workloads(lib, fa, dev, stream, flush, peak):
    """Kernel-timed TFLOP/s at other head dimensions (informational)."""
    import torch
    res = {}
    B, H, S = 4, 16, 4096
    for D, dt, seed in HEAD_DIMS:
        qb, kb, vb = fa_inputs.make_qkv(B, H, S, D, dt, "normal", seed)
        q, k, v = (fa_inputs.to_torch(x, dt).to(dev) for x in (qb, kb, vb))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
        code = fa.FA_F16 if dt == "f16" else fa.FA_BF16
        t = _median_kernel_ms(stream, flush, lambda: lib.fa_fwd_gqa(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, H, S, D, 1,
            D ** -0.5, code, stream.cuda_stream))
        tf = fa_inputs.attention_flops(B, H, S, D, True) / (t * 1e-3) / 1e12
        res[f"headdim{D}_b{B}h{H}s{S}/causal"] = {
            "ms": t, "tflops": tf, "pct_of_peak": 100.0 * tf / peak, "launches": 1}
        del q, k, v, o, lse
    return res


def _median_kernel_ms(stream, flush, call):
    """Median CUDA-event time of call() over 10 runs after 3 warm-ups, L2
    flushed before each."""
    import torch
    ms = []
    with torch.cuda.stream(stream):
        for i in range(13):
            flush.fill_(float(i))
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            rc = call()
            e1.record(stream)
            assert rc == 0, rc
            if i >= 3:
                ms.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in ms)


# Attention dropout, p = 0.1: the b4h16 (D = 64 fp16) and b2h16d128 (D = 128
# bf16) shapes, causal; FLOPs as the plain forward (the mask is extra work).
DROPOUT = dict(p=0.1, seed=1009, workloads=("b4h16", "b2h16d128"))


def dropout_workloads(lib, fa, dev, stream, flush, peak):
    """Kernel-timed TFLOP/s of the dropout variant (informational)."""
    import torch
    res = {}
    for name in DROPOUT["workloads"]:
        w = fa_inputs.WORKLOADS[name]
        qb, kb, vb = fa_inputs.make_qkv_for(w)
        q, k, v = (fa_inputs.to_torch(x, w.dtype).to(dev) for x in (qb, kb, vb))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
        code = fa.FA_F16 if w.dtype == "f16" else fa.FA_BF16
        t = _median_kernel_ms(stream, flush, lambda: lib.fa_fwd_dropout(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.H,
            w.kv_heads, w.S, w.D, 1, DROPOUT["p"], DROPOUT["seed"], w.scale, code,
            stream.cuda_stream))
        tf = fa_inputs.attention_flops(w.B, w.H, w.S, w.D, True) / (t * 1e-3) / 1e12
        res[f"dropout{DROPOUT['p']}_{name}/causal"] = {
            "ms": t, "tflops": tf, "pct_of_peak": 100.0 * tf / peak, "launches": 1}
        del q, k, v, o, lse
    return res


# Local attention: B2 H16 S16384 D128 bf16, causal, each query sees the 2048
# keys before it and itself; FLOPs 4*D per visible (query, key) pair.
WINDOW = dict(B=2, H=16, S=16384, D=128, left=2048, seed=1008)


def window_workload(lib, fa, dev, stream, flush, peak):
    """Kernel-timed TFLOP/s of the sliding-window workload (informational)."""
    import torch
    c = WINDOW
    qb, kb, vb = fa_inputs.make_qkv(c["B"], c["H"], c["S"], c["D"], "bf16", "normal", c["seed"])
    q, k, v = (fa_inputs.to_torch(x, "bf16").to(dev) for x in (qb, kb, vb))
    o = torch.empty_like(q)
    lse = torch.empty((c["B"], c["H"], c["S"]), dtype=torch.float32, device=dev)
    ms = []
    with torch.cuda.stream(stream):
        for i in range(13):
            flush.fill_(float(i))
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            rc = lib.fa_fwd_local(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  lse.data_ptr(), c["B"], c["H"], c["H"], c["S"], c["D"], 1,
                                  c["left"], -1, c["D"] ** -0.5, fa.FA_BF16, stream.cuda_stream)
            e1.record(stream)
            assert rc == 0
            if i >= 3:
                ms.append((e0, e1))
    torch.cuda.synchronize(dev)
    t = statistics.median(a.elapsed_time(b) for a, b in ms)
    S, L = c["S"], c["left"]
    pairs = sum(min(i, L) + 1 for i in range(S))          # visible keys per head
    flops = 4.0 * c["D"] * pairs * c["B"] * c["H"]
    tf = flops / (t * 1e-3) / 1e12
    name = f"window{L}_b{c['B']}h{c['H']}s{S}d{c['D']}/causal"
    return {name: {"ms": t, "tflops": tf, "pct_of_peak": 100.0 * tf / peak, "launches": 1}}


# Packed variable-length batch: 16 sequences of 256..8192 tokens (uniform,
# seed 1007), 16 heads, D = 128 bf16, causal; FLOPs 2*H*S_b^2*D per sequence.
VARLEN = dict(B=16, lo=256, hi=8192, seed=1007, H=16, D=128, dtype="bf16")


def varlen_workload(lib, fa, dev, stream, flush, peak):
    """Kernel-timed TFLOP/s of the packed variable-length batch (informational)."""
    import numpy as np
    import torch
    c = VARLEN
    lens = fa_inputs.varlen_lengths(c["B"], c["lo"], c["hi"], c["seed"])
    qb, kb, vb, cu = fa_inputs.make_varlen(lens, c["H"], c["D"], c["dtype"], "normal", c["seed"])
    q, k, v = (fa_inputs.to_torch(x, c["dtype"]).to(dev) for x in (qb, kb, vb))
    cu_t = torch.from_numpy(cu).to(dev)
    o = torch.empty_like(q)
    total = q.shape[0]
    lse = torch.empty((c["H"], total), dtype=torch.float32, device=dev)
    scale = c["D"] ** -0.5
    ms = []
    with torch.cuda.stream(stream):
        for i in range(13):
            flush.fill_(float(i))
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            rc = lib.fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), cu_t.data_ptr(), c["B"], int(lens.max()), total,
                                   c["H"], c["H"], c["D"], 1, scale, fa.FA_BF16, stream.cuda_stream)
            e1.record(stream)
            assert rc == 0
            if i >= 3:
                ms.append((e0, e1))
    torch.cuda.synchronize(dev)
    t = statistics.median(a.elapsed_time(b) for a, b in ms)
    flops = sum(fa_inputs.attention_flops(1, c["H"], int(s_), c["D"], True) for s_ in lens)
    tf = flops / (t * 1e-3) / 1e12
    name = f"varlen{c['B']}x{c['lo']}-{c['hi']}h{c['H']}d{c['D']}/causal"
    return {name: {"ms": t, "tflops": tf, "pct_of_peak": 100.0 * tf / peak, "launches": 1,
                   "tokens": int(total)}}


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
                    help="also time the workloads beyond the five target configurations")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the kernel-timed numbers of the other target configurations")
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
