#!/usr/bin/env python
"""Benchmark of the persistent ReLU-RNN forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
                    [--algo persistent|per_step] [--impl ours|reference]

One step = one prnn_forward over the whole workload (projection of all T
steps + the T-step recurrence) with inputs resident in HBM.  The default
workload is the sparse layer the headline metric is quoted on: H = 1792,
B = 4, T = 256, Wh row-balanced at 10 % (179 non-zeros per row), fp16 weights,
fp32 activations and accumulation.  Inputs are smaller than L2, so L2 is
flushed (a 256 MiB write) between timed steps, outside the timed events.

Prints one JSON line (rank 0).  Multi-GPU: replicas only (every rank runs the
same layer on its own GPU, no collective on the data path); value is the
timesteps all ranks processed divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_CONFIG = "sparse_f16_h1792_d10_b4_t256"
METRIC = "RNN timesteps/s (H=1792, B=4, T=256, 10% row-balanced sparse Wh)"
FLUSH_BYTES = 256 << 20


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--algo", default="persistent", choices=["persistent", "per_step"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip e2e / sync floor / per-step comparison (for profiling runs)")
    ap.add_argument("--sweep", action="store_true",
                    help="time the H x B x density sweep, persistent vs per-step path "
                         "(one JSON line per point)")
    ap.add_argument("--sweep-filter", default="", help="only sweep points whose name contains this")
    ap.add_argument("--ablation", action="store_true",
                    help="the sparse persistent RNN ablation at H=1152, B=4, 10 %%, T=256: "
                         "plain -> +wide loads -> +bank-aware layout -> +flags in the data, "
                         "each against the per-step dense path")
    ap.add_argument("--balance", action="store_true",
                    help="load-balanced versus globally pruned (unbalanced) sparse layers of "
                         "equal non-zero count, persistent, against the per-step dense path")
    ap.add_argument("--stack", action="store_true",
                    help="stacked layers: one-launch wavefront vs layer by layer, "
                         "H = 256 / 512 / 1152, L = 1 .. 8")
    ap.add_argument("--vendor", action="store_true",
                    help="persistent kernels vs per-step cuBLAS / cuSPARSE products (one JSON "
                         "line per workload)")
    ap.add_argument("--trace", action="store_true",
                    help="phase trace of the sparse persistent kernel on the config's layer "
                         "(first --trace-steps steps): where the time of a step goes")
    ap.add_argument("--trace-steps", type=int, default=16)
    ap.add_argument("--trace-out", default="", help="save the raw trace records (.npy)")
    ap.add_argument("--backward", action="store_true",
                    help="training step (forward + backward through time) of the named workloads")
    ap.add_argument("--cluster-probe", action="store_true",
                    help="step exchange through distributed shared memory inside thread-block "
                         "clusters (no arithmetic) beside the L2 exchange floor of the config")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def workload_flops(p) -> dict:
    """Algorithmic FLOPs of one forward: projection 2*T*B*H*I, recurrence
    2*T*B*nnz (nnz = H*H dense, H*k sparse)."""
    proj = 2.0 * p.T * p.B * p.H * p.I
    rec = 2.0 * p.T * p.B * p.nnz
    return {"projection": proj, "recurrence": rec, "total": proj + rec,
            "recurrence_dense_equiv": 2.0 * p.T * p.B * p.H * p.H}


# ---- clocks ---------------------------------------------------------------------
CLOCK_FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


_REASON_BITS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40),
                ("sw_thermal_slowdown", 0x20), ("sw_power_cap", 0x4))


class _NvmlPoller:
    """Reads the SM clock and the clock-event-reason mask through NVML (read
    only) every ``period_s`` on a background thread, so that even a timed
    region of a few milliseconds gets samples."""

    def __init__(self, gpu_id: str, period_s: float = 0.002):
        import ctypes
        import threading
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(gpu_id.encode(), ctypes.byref(self.dev)) != 0:
            if self.lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.dev)) != 0:
                raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) \
            or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx))
        self.max_mhz = float(mx.value)
        self.rows = []
        self.period = period_s
        self.stop = threading.Event()
        self.thread = threading.Thread(target=self._run, daemon=True)

    def _sample(self):
        ct = self.ct
        mhz, mask = ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(mhz)) != 0:
            return
        if self.reasons_fn(self.dev, ct.byref(mask)) != 0:
            return
        self.rows.append((float(mhz.value), self.max_mhz,
                          ["Active" if mask.value & bit else "Not Active"
                           for _, bit in _REASON_BITS]))

    def _run(self):
        while not self.stop.is_set():
            self._sample()
            self.stop.wait(self.period)

    def start(self):
        self._sample()
        self.thread.start()

    def finish(self):
        self.stop.set()
        self.thread.join(timeout=5)
        self._sample()
        self.lib.nvmlShutdown()
        return self.rows


class ClockSampler:
    """SM clocks and throttle reasons during the timed region: NVML polled
    every 2 ms where the library loads, else ``nvidia-smi -lms 200``."""

    def __init__(self, gpu_id: str):
        self.proc = None
        self.nvml = None
        self.gpu_id = gpu_id

    def __enter__(self):
        try:
            self.nvml = _NvmlPoller(self.gpu_id)
            self.nvml.start()
            return self
        except (OSError, AttributeError):
            self.nvml = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        self.rows = None
        if self.nvml is not None:
            self.rows = self.nvml.finish()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self) -> dict:
        rows = list(self.rows or [])
        for line in (self.out or "").strip().splitlines():
            f = [c.strip() for c in line.split(",")]
            if len(f) < 8:
                continue
            try:
                rows.append((float(f[0]), float(f[1]), f[4:8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = sorted(r[0] for r in rows)
        names = tuple(n for n, _ in _REASON_BITS)
        reasons = sorted({names[i] for r in rows for i in range(4) if r[2][i] == "Active"})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows),
                "source": "nvml 2 ms" if self.rows else "nvidia-smi 200 ms"}


# ---- reference arm: the fp64 CPU oracle -------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np  # noqa: F401
    import oracle
    from persistent_rnn_recurrence_gb300 import synth
    p = synth.named_problem(args.config)
    o = oracle.default()
    # size one step at about one second of oracle work
    t0 = time.perf_counter()
    o.forward(p, T=2)
    per_t = (time.perf_counter() - t0) / 2
    Ts = int(max(1, min(p.T, round(1.0 / max(per_t, 1e-6)))))
    for _ in range(args.warmup):
        o.forward(p, T=Ts)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        o.forward(p, T=Ts)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = Ts * args.steps / total
    sample = f"first {Ts} of {p.T} timesteps of the workload per step, single thread"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "timesteps/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(p, args, "fp64 CPU oracle"),
        "cpu_baseline": {"value": value, "unit": "timesteps/s", "cores": 1,
                         "kind": "oracle", "sample": sample, "host": host_cpu()},
        "e2e": {"value": value, "unit": "timesteps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_dict(p, args, path):
    return {"workload": p.name, "H": p.H, "I": p.I, "B": p.B, "T": p.T,
            "weights": ("row-balanced sparse, k=%d (%.1f%%)" % (p.k, 100.0 * p.k / p.H))
            if p.sparse else "dense", "wdtype": p.wdtype, "path": path,
            "l2": "flushed between timed steps (256 MiB write)", "global_batch": p.B,
            "seq_len": p.T, "parallelism": "replicas" if args.gpus > 1 else "single GPU"}


def host_cpu() -> dict:
    """Core count and CPU model of the host the oracle is timed on."""
    usable = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name:"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith("model name"):
                        model = ln.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    if model is None:
        import platform
        model = platform.processor() or platform.machine()
    return {"cpu_count": os.cpu_count(), "usable_cores": usable, "cpu_model": model}


def time_oracle(p, threads: int = 1, budget: float = 12.0) -> dict:
    """The oracle on a bounded sample of the workload: about ``budget`` seconds
    of work.  A sequence it finishes in less than that is run again until the
    time is reached; a longer one is cut to its first timesteps."""
    import oracle
    o = oracle.default()
    t0 = time.perf_counter()
    o.forward(p, T=2, threads=threads)
    per_t = (time.perf_counter() - t0) / 2
    Ts = int(max(1, min(p.T, round(budget / max(per_t, 1e-6)))))
    runs, dt = 0, 0.0
    while runs == 0 or dt < budget:
        t0 = time.perf_counter()
        o.forward(p, T=Ts, threads=threads)
        dt += time.perf_counter() - t0
        runs += 1
    how = "single thread" if threads == 1 else f"{threads} threads"
    return {"value": runs * Ts / dt, "unit": "timesteps/s", "cores": threads, "kind": "oracle",
            "sample": f"first {Ts} of {p.T} timesteps, B={p.B}, {runs} run(s) back to back, "
                      f"{how}",
            "seconds": dt}


def cpu_baseline(p) -> dict:
    """The oracle as it stands, single-threaded, about 12 s of CPU work."""
    out = time_oracle(p, threads=1)
    out["host"] = host_cpu()
    return out


def cpu_baseline_all_cores(p) -> dict:
    """The oracle's threaded driver (the same cell arithmetic, each step's
    outputs split over every usable host core), about 12 s of CPU work."""
    n = host_cpu()["usable_cores"] or 1
    out = time_oracle(p, threads=n)
    out["kind"] = "oracle, threaded driver (bit-identical output)"
    return out


SWEEP_SAMPLE_T = 32


def sweep_cpu_baseline(p, ys: dict) -> dict:
    """The sweep point's CPU-baseline leg: the oracle on every usable host core
    over the point's first SWEEP_SAMPLE_T steps, timed, and -- from that same
    output -- the parity of each GPU path's first steps (``ys``: path -> y
    [T', B, H] as numpy) under the rule max|y - y_oracle| <= 2e-2 max|y_oracle|
    (fp16 weights, fp32 accumulation)."""
    import numpy as np
    import oracle
    n = host_cpu()["usable_cores"] or 1
    Ts = min(SWEEP_SAMPLE_T, p.T)
    t0 = time.perf_counter()
    ref = oracle.default().forward(p, T=Ts, threads=n)
    dt = time.perf_counter() - t0
    scale = float(np.abs(ref).max())
    parity = {"steps": Ts, "tol": 2e-2, "pass": True}
    for path, y in ys.items():
        err = float(np.abs(y[:Ts].astype(np.float64) - ref).max()) / max(scale, 1e-30)
        parity[path + "_max_rel_err"] = err
        parity["pass"] = parity["pass"] and bool(np.isfinite(y[:Ts]).all()) and err <= 2e-2
    return {"cpu_baseline": {"value": Ts / dt, "unit": "timesteps/s", "cores": n,
                             "kind": "oracle, threaded driver",
                             "sample": f"first {Ts} of {p.T} timesteps, B={p.B}"},
            "parity": parity}


# ---- our arm ----------------------------------------------------------------------------
def run_ours(args):
    import numpy as np  # noqa: F401
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from persistent_rnn_recurrence_gb300 import prnn, synth

    p = synth.named_problem(args.config)
    lay = prnn.Layer.from_problem(p, algo=args.algo)
    lay.set_option(prnn.PRNN_OPT_TIMING, 1)
    info = lay.info()
    x = torch.from_numpy(p.x).to(dev)
    h0 = None if p.h0 is None else torch.from_numpy(p.h0).to(dev)
    y = torch.empty((p.T, p.B, p.H), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    fl = workload_flops(p)

    def step():
        prnn.prnn_forward(lay.h, p.T, p.B, x, h0, y, stream)

    for _ in range(max(3, args.warmup)):
        flush.fill_(1.0)
        step()
    torch.cuda.synchronize()
    if lay.status() != prnn.PRNN_OK:
        raise RuntimeError("warm-up forward reported " + prnn.prnn_status_string(lay.status()))

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    stage = []
    props = torch.cuda.get_device_properties(dev)
    gpu_id = getattr(props, "uuid", None)
    gpu_id = f"GPU-{gpu_id}" if gpu_id is not None and not str(gpu_id).startswith("GPU-") \
        else str(gpu_id if gpu_id is not None else local)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_id) as clk:
        wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(1.0)
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
            stage.append(prnn.prnn_get_timing(lay.h))   # synchronizes on the forward
        torch.cuda.synchronize()
        wall = time.perf_counter() - wall0
    barrier(world)
    torch.cuda.synchronize()
    if lay.status() != prnn.PRNN_OK:
        raise RuntimeError("timed forward reported " + prnn.prnn_status_string(lay.status()))
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world, dev)
    ms_step = 1e3 * total_s / args.steps
    value = world * p.T * args.steps / total_s
    rec_ms = sorted(s[1] for s in stage)
    proj_ms = sorted(s[0] for s in stage)
    rec_med = rec_ms[len(rec_ms) // 2]
    proj_med = proj_ms[len(proj_ms) // 2]
    clocks = clk.summary()

    extras = {}
    if not args.no_extras:
        extras = measure_extras(args, p, lay, x, h0, y, flush, stream, dev, world)

    # roofline of the dominant (recurrent) kernel: on-chip bound, FP32 FMA pipe
    sm_count = info["sm_count"] or props.multi_processor_count
    peaks = load_peaks()
    sm_max_mhz = peaks.get("sm_max_mhz", 2070.0)
    fma_peak_tflops = sm_count * 128 * 2 * sm_max_mhz * 1e6 / 1e12
    smem_peak_tbs = sm_count * 128 * sm_max_mhz * 1e6 / 1e12
    w_bytes = (4.0 * p.nnz) if p.sparse else (p.H * p.H * (2.0 if p.wdtype == "f16" else 4.0))
    t_fma = (2.0 * p.B * p.nnz) / (fma_peak_tflops * 1e12)
    t_smem = w_bytes / (smem_peak_tbs * 1e12)
    rec_tflops = fl["recurrence"] / (rec_med * 1e-3) / 1e12
    roof = {"bound": "alu", "kernel": "recur_sparse_kernel" if p.sparse else "recur_dense_kernel",
            "achieved": rec_tflops, "peak": fma_peak_tflops, "unit": "TFLOP/s",
            "frac": rec_tflops / fma_peak_tflops,
            "traffic": load_traffic(p.name, args.algo, p.sparse),
            "peak_source": f"derived: {sm_count} SMs x 128 FP32 lanes x 2 FLOP x {sm_max_mhz:.0f} MHz",
            "t_roof_step_ns": 1e9 * max(t_fma, t_smem),
            "t_step_ns": 1e6 * rec_med / p.T,
            "frac_of_step_roofline": 1e9 * max(t_fma, t_smem) / (1e6 * rec_med / p.T)}
    if args.algo == "per_step":
        roof["kernel"] = "step kernels (T launches)"

    line = {
        "metric": METRIC if args.config == DEFAULT_CONFIG else f"RNN timesteps/s ({p.name})",
        "value": value, "unit": "timesteps/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": config_dict(p, args, args.algo),
        "gflops_effective": fl["total"] / (ms_step * 1e-3) / 1e9 * world,
        "gflops_dense_equivalent": (fl["projection"] + fl["recurrence_dense_equiv"])
        / (ms_step * 1e-3) / 1e9 * world,
        "step_ms_stats": {"median": sorted(step_ms)[len(step_ms) // 2], "min": min(step_ms),
                          "max": max(step_ms)},
        "stage_ms": {"projection": proj_med, "recurrence": rec_med,
                     "projection_min": proj_ms[0], "recurrence_min": rec_ms[0]},
        "roofline": roof,
        "clocks": clocks,
        "gpu_launches": args.steps * ((2 if info["projection_tensor_cores"] else 1)
                                      + (1 if args.algo == "persistent" else p.T)),
        "wall_s": wall,
        "plan": {k: info[k] for k in ("n_cta", "rows_per_cta", "threads_per_cta",
                                      "threads_per_row", "k_padded", "smem_bytes",
                                      "onchip_weight_bytes", "projection_tensor_cores")},
    }
    line.update(extras)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(p)
        if getattr(p, "row_ptr", None) is None:
            line["cpu_baseline_all_cores"] = cpu_baseline_all_cores(p)
    lay.close()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def measure_extras(args, p, lay, x, h0, y, flush, stream, dev, world):
    import torch
    from persistent_rnn_recurrence_gb300 import prnn
    out = {}
    K = max(3, min(args.steps, 10))
    # end to end from pinned host memory: prnn_forward_host (x read over the host
    # link by the projection's staging kernel, h0 copied in, y written to the host
    # by the recurrent kernel as it is published), and for
    # comparison host copies around prnn_forward on device buffers
    xh = torch.from_numpy(p.x).pin_memory()
    h0h = None if h0 is None else h0.cpu().pin_memory()
    yh = torch.empty((p.T, p.B, p.H), dtype=torch.float32).pin_memory()
    xd = torch.empty_like(x)

    def via_host_call():
        prnn.prnn_forward_host(lay.h, p.T, p.B, xh, h0h, yh, stream)

    def via_copies():
        xd.copy_(xh, non_blocking=True)
        prnn.prnn_forward(lay.h, p.T, p.B, xd, h0, y, stream)
        yh.copy_(y, non_blocking=True)

    def time_e2e(fn):
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        ms = []
        for _ in range(K):
            flush.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ms.append(a.elapsed_time(b))
        return world * p.T * K / max_over_ranks(sum(ms) / 1e3, world, dev)

    h2d = (xh.numel() + (0 if h0h is None else h0h.numel())) * 4
    out["e2e"] = {"value": time_e2e(via_host_call), "unit": "timesteps/s",
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": yh.numel() * 4,
                  "call": "prnn_forward_host on pinned host buffers"}
    out["e2e_device_call_with_copies"] = {
        "value": time_e2e(via_copies), "unit": "timesteps/s", "h2d_bytes_per_step": h2d,
        "d2h_bytes_per_step": yh.numel() * 4,
        "call": "H2D copy, prnn_forward on device buffers, D2H copy"}
    # step-synchronisation floor of the same grid
    if args.algo == "persistent":
        ys = torch.empty_like(y)
        fl_ms = []
        for _ in range(K):
            prnn.prnn_probe_sync_floor(lay.h, p.T, p.B, ys, stream)
            fl_ms.append(prnn.prnn_get_timing(lay.h)[1])
        fl_ms.sort()
        out["sync_floor_ns_per_step"] = 1e6 * fl_ms[len(fl_ms) // 2] / p.T
        # in-house per-step path on the same workload, for the persistent/per-step ratio
        from persistent_rnn_recurrence_gb300 import synth  # noqa: F401
        ps = prnn.Layer.from_problem(p, algo="per_step")
        ps.set_option(prnn.PRNN_OPT_TIMING, 1)
        for _ in range(3):
            prnn.prnn_forward(ps.h, p.T, p.B, x, h0, y, stream)
        pm = []
        for _ in range(K):
            flush.fill_(1.0)
            prnn.prnn_forward(ps.h, p.T, p.B, x, h0, y, stream)
            pm.append(prnn.prnn_get_timing(ps.h))
        ps.close()
        rec = sorted(v[1] for v in pm)
        out["per_step_path"] = {"recurrence_ms": rec[len(rec) // 2],
                                "timesteps_per_s_recurrence": 1e3 * p.T / rec[len(rec) // 2]}
    return out


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return {}


KERNEL_SOURCES = {
    True: ["persistent_sparse.cu", "persistent_sparse.cuh", "persistent_sparse_regw.cu",
           "persistent_sparse_um.cu", "persistent_common.cuh", "device_common.cuh"],
    False: ["persistent_dense.cu", "persistent_common.cuh", "device_common.cuh"],
}


def kernel_source_sha1(sparse: bool) -> str:
    import hashlib
    h = hashlib.sha1()
    for name in KERNEL_SOURCES[sparse]:
        with open(os.path.join(ROOT, "persistent_rnn_recurrence_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def load_traffic(workload: str, algo: str, sparse: bool):
    """DRAM bytes per launch of the recurrent kernel from the committed ncu
    capture (profiles/traffic.json), or None when it was not captured for this
    workload or the kernel's source has changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(f"{workload}/{algo}")
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_source_sha1") != kernel_source_sha1(sparse):
        return None
    return rec.get("dram_bytes_per_launch")


def run_sweep(args):
    """Persistent vs per-step recurrence time for every sweep point (T = 256,
    fp16 weights), forward time and per-step time, L2 flushed before each
    timed forward.  Points whose layer does not fit on chip are reported as
    unsupported rather than skipped.  Unless --no-cpu-baseline, each line also
    carries its CPU-baseline leg: the oracle timed on the point's first
    steps, and the parity of both paths' first steps against that output."""
    import torch
    from persistent_rnn_recurrence_gb300 import prnn, synth
    dev = torch.device("cuda", 0)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    reps = max(3, min(args.steps, 5))
    for name, kw in synth.sweep_points():
        if args.sweep_filter and args.sweep_filter not in name:
            continue
        p = synth.make_problem(name=name, **kw)
        x = torch.from_numpy(p.x).to(dev)
        y = torch.empty((p.T, p.B, p.H), dtype=torch.float32, device=dev)
        line = {"point": name, "H": p.H, "B": p.B, "k": p.k, "density": p.k / p.H}
        first_steps = {}
        for algo in ("persistent", "per_step"):
            try:
                lay = prnn.Layer.from_problem(p, algo=algo)
            except prnn.PrnnError as e:
                line[algo] = {"unsupported": str(e)}
                continue
            lay.set_option(prnn.PRNN_OPT_TIMING, 1)
            prnn.prnn_forward(lay.h, p.T, p.B, x, None, y)
            ms = []
            for _ in range(reps):
                flush.fill_(1.0)
                prnn.prnn_forward(lay.h, p.T, p.B, x, None, y)
                ms.append(prnn.prnn_get_timing(lay.h))
            st = lay.status()
            info = lay.info()
            lay.close()
            rec = sorted(m[1] for m in ms)[len(ms) // 2]
            proj = sorted(m[0] for m in ms)[len(ms) // 2]
            first_steps[algo] = y[:SWEEP_SAMPLE_T].cpu().numpy()
            fma_peak = (info["sm_count"] or 152) * 128 * 2 * \
                load_peaks().get("sm_max_mhz", 2070.0) * 1e6
            line[algo] = {"recurrence_us_per_step": 1e3 * rec / p.T, "projection_ms": proj,
                          "frac_of_fma_peak": (2.0 * p.nnz * p.B / fma_peak) / (1e-3 * rec / p.T),
                          "timesteps_per_s": 1e3 * p.T / (rec + proj),
                          "status": prnn.prnn_status_string(st),
                          "groups": info["cta_groups"], "n_cta": info["n_cta"]}
            if algo == "persistent":
                line[algo]["kernel"] = ("ksplit" if info["dense_ksplit"]
                                        else "sparse" if p.sparse else "dense")
            if p.sparse and algo == "persistent" and not info["dense_ksplit"]:
                # the sparse kernel's gathers' shared-memory bound: every entry x
                # batch column reads its own 4-byte h word, plus the 4-byte entries
                smem_bw = (info["sm_count"] or 152) * 128 * \
                    load_peaks().get("sm_max_mhz", 2070.0) * 1e6
                t_smem = (4.0 * p.nnz * p.B + 4.0 * p.nnz) / smem_bw
                line[algo]["frac_of_smem_gather_bound"] = t_smem / (1e-6 * line[algo][
                    "recurrence_us_per_step"])
        if "recurrence_us_per_step" in line.get("persistent", {}) and \
                "recurrence_us_per_step" in line.get("per_step", {}):
            line["persistent_speedup"] = (line["per_step"]["recurrence_us_per_step"]
                                          / line["persistent"]["recurrence_us_per_step"])
        if not args.no_cpu_baseline and first_steps:
            line.update(sweep_cpu_baseline(p, first_steps))
        print(json.dumps(line), flush=True)
    return 0


def run_ablation(args):
    """The ablation rows of the sparse persistent RNN measurements (H=1152,
    B=4, 10 %, T=256), reproduced with this library's switches: each row adds
    one feature; speedups are against the non-persistent per-step path on the
    densified matrix (the dense-GEMM-per-step analogue)."""
    import numpy as np
    import torch
    from persistent_rnn_recurrence_gb300 import prnn, synth
    dev = torch.device("cuda", 0)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    p = synth.make_problem(H=1152, B=4, T=256, k=synth.sparse_k(1152, 0.10), seed=3000,
                           name="ablation_sparse_h1152_d10_b4_t256")
    x = torch.from_numpy(p.x).to(dev)
    y = torch.empty((p.T, p.B, p.H), dtype=torch.float32, device=dev)
    reps = max(5, min(args.steps, 10))

    def rec_us(lay):
        lay.set_option(prnn.PRNN_OPT_TIMING, 1)
        prnn.prnn_forward(lay.h, p.T, p.B, x, None, y)
        ms = []
        for _ in range(reps):
            flush.fill_(1.0)
            prnn.prnn_forward(lay.h, p.T, p.B, x, None, y)
            ms.append(prnn.prnn_get_timing(lay.h)[1])
        assert lay.status() == prnn.PRNN_OK
        return 1e3 * sorted(ms)[len(ms) // 2] / p.T

    # per-step dense path on the densified matrix
    dense = synth.Problem(name="densified", T=p.T, B=p.B, H=p.H, I=p.I, wdtype="f16", x=p.x,
                          Wx=p.Wx, b=p.b, h0=None, Wh=np.zeros((p.H, p.H), np.float16))
    for r in range(p.H):
        dense.Wh[r, p.cols[r].astype(np.int64)] = p.vals[r]
    lay = prnn.Layer.from_problem(dense, algo="per_step")
    base = rec_us(lay)
    lay.close()
    rows = [("sparse persistent, 32-bit loads, plain layout, grid barrier", 0, 0, 1, 0),
            ("+ wide (128-bit) loads", 1, 0, 1, 0),
            ("+ bank-aware layout", 1, 1, 1, 0),
            ("+ flags in the data (no grid barrier)", 1, 1, 0, 0),
            ("+ per-CTA bank-balancing order of the staged h", 1, 1, 0, 1)]
    out = {"workload": p.name, "per_step_dense_us_per_step": base, "rows": []}
    for label, wide, bank, barrier, staged in rows:
        lay = prnn.Layer(p.H, p.I, p.B, "f16", "persistent")
        lay.set_option(prnn.PRNN_OPT_BANK_AWARE, bank)
        lay.set_option(prnn.PRNN_OPT_STAGED_ORDER, staged)
        lay.set_problem_weights(p)
        lay.set_option(prnn.PRNN_OPT_WIDE_LOADS, wide)
        lay.set_option(prnn.PRNN_OPT_SYNC_MODE, barrier)
        us = rec_us(lay)
        info = lay.info()
        lay.close()
        out["rows"].append({"row": label, "us_per_step": us, "speedup_vs_per_step_dense": base / us,
                            "bank_cap": info["sparse_bank_cap"], "groups": info["cta_groups"]})
    print(json.dumps(out))
    # the staged order on the named sparse layers, column order vs staged, same box
    for name in [n for n in synth.NAMED if n.startswith("sparse")]:
        q = synth.named_problem(name)
        xq = torch.from_numpy(q.x).to(dev)
        yq = torch.empty((q.T, q.B, q.H), dtype=torch.float32, device=dev)
        line = {"workload": name}
        for staged in (0, 1):
            lay = prnn.Layer(q.H, q.I, q.B, "f16", "persistent")
            lay.set_option(prnn.PRNN_OPT_STAGED_ORDER, staged)
            lay.set_problem_weights(q)
            lay.set_option(prnn.PRNN_OPT_TIMING, 1)
            prnn.prnn_forward(lay.h, q.T, q.B, xq, None, yq)
            ms = []
            for _ in range(reps):
                flush.fill_(1.0)
                prnn.prnn_forward(lay.h, q.T, q.B, xq, None, yq)
                ms.append(prnn.prnn_get_timing(lay.h)[1])
            assert lay.status() == prnn.PRNN_OK
            info = lay.info()
            lay.close()
            key = "staged_order" if staged else "column_order"
            line[key] = {"us_per_step": 1e3 * sorted(ms)[len(ms) // 2] / q.T,
                         "bank_cap": info["sparse_bank_cap"], "k_padded": info["k_padded"],
                         "staged": info["sparse_staged_order"]}
        print(json.dumps(line))
    return 0


def run_balance(args):
    """Load-balanced versus straightforward pruning: one layer pruned to the
    same number of non-zeros by global magnitude pruning (rows of unequal
    length, compressed-row weights) and by per-row pruning (every row the
    same length), each run persistent; plus the per-step path on the
    densified unbalanced matrix as the non-persistent baseline."""
    import numpy as np
    import torch
    from persistent_rnn_recurrence_gb300 import prnn, synth
    dev = torch.device("cuda", 0)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    reps = max(5, min(args.steps, 10))
    out = []
    for H, d in ((2304, 0.25), (1792, 0.10), (5760, 0.05)):
        unb, bal = synth.make_pruned_pair(H=H, B=4, T=256, density=d, seed=3100 + H,
                                          name=f"pruned_h{H}_d{int(round(d * 100))}_b4_t256")
        x = torch.from_numpy(unb.x).to(dev)
        y = torch.empty((unb.T, unb.B, unb.H), dtype=torch.float32, device=dev)

        def rec_us(p, algo):
            try:
                lay = prnn.Layer.from_problem(p, algo=algo)
            except prnn.PrnnError as e:
                return None, {"error": str(e)}
            try:
                lay.set_option(prnn.PRNN_OPT_TIMING, 1)
                prnn.prnn_forward(lay.h, p.T, p.B, x, None, y)
                ms = []
                for _ in range(reps):
                    flush.fill_(1.0)
                    prnn.prnn_forward(lay.h, p.T, p.B, x, None, y)
                    ms.append(prnn.prnn_get_timing(lay.h)[1])
                assert lay.status() == prnn.PRNN_OK
                return 1e3 * sorted(ms)[len(ms) // 2] / p.T, lay.info()
            except prnn.PrnnError as e:
                return None, {"error": str(e)}
            finally:
                lay.close()

        dense = synth.Problem(name="densified", T=unb.T, B=unb.B, H=H, I=H, wdtype="f16",
                              x=unb.x, Wx=unb.Wx, b=unb.b, h0=None,
                              Wh=np.zeros((H, H), np.float16))
        rows = np.repeat(np.arange(H), np.diff(unb.row_ptr))
        dense.Wh[rows, unb.cols.astype(np.int64)] = unb.vals
        lens = np.diff(unb.row_ptr)
        rec = {"workload": unb.name, "nnz": unb.nnz, "row_len_mean": float(lens.mean()),
               "row_len_max": int(lens.max()), "row_len_min": int(lens.min())}
        for key, p, algo in (("per_step_dense", dense, "per_step"),
                             ("persistent_unbalanced", unb, "persistent"),
                             ("persistent_balanced", bal, "persistent")):
            us, info = rec_us(p, algo)
            rec[key + "_us_per_step"] = us
            if "error" in info:
                rec[key + "_error"] = info["error"]
        if rec["persistent_balanced_us_per_step"] and rec["persistent_unbalanced_us_per_step"]:
            rec["balanced_speedup"] = (rec["persistent_unbalanced_us_per_step"]
                                       / rec["persistent_balanced_us_per_step"])
        out.append(rec)
    print(json.dumps({"balance": out}))
    return 0


def run_stack(args):
    """Stacked dense fp16 layers (B=4, T=256): the one-launch wavefront against
    the layer-by-layer path (batched projection + persistent recurrence per
    layer), for H = 256, 512, 1152 and L = 1, 2, 4, 8 (where the weights fit)."""
    import torch
    from persistent_rnn_recurrence_gb300 import prnn, synth
    dev = torch.device("cuda", 0)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    reps = max(5, min(args.steps, 20))
    out = []
    for H, L in ((256, 1), (256, 2), (256, 4), (256, 8), (512, 2), (512, 4), (512, 8),
                 (1152, 1), (1152, 2), (1152, 4)):
        p = synth.make_stack_problem(L=L, H=H, B=4, T=256, wdtype="f16", seed=3200 + L,
                                     name=f"stack_l{L}_h{H}_b4_t256")
        x = torch.from_numpy(p.x).to(dev)
        y = torch.empty((L, p.T, p.B, p.H), dtype=torch.float32, device=dev)
        rec = {"workload": p.name, "layers": L, "H": H}
        for algo in ("wavefront", "layerwise"):
            try:
                st = prnn.Stack.from_problem(p, algo=algo)
            except prnn.PrnnError as e:
                rec[algo] = {"error": str(e)}
                continue
            try:
                st.set_option(prnn.PRNN_OPT_TIMING, 1)
                for _ in range(3):
                    flush.fill_(1.0)
                    st.forward(x, None, y)
                ms = []
                for _ in range(reps):
                    flush.fill_(1.0)
                    st.forward(x, None, y)
                    ms.append(prnn.prnn_stack_get_timing(st.h))
                assert st.status() == prnn.PRNN_OK
                med = sorted(ms)[len(ms) // 2]
                rec[algo] = {"ms_per_forward": med, "ms_min": min(ms), "ms_max": max(ms),
                             "timesteps_per_s": p.T / (med * 1e-3),
                             "us_per_step": 1e3 * med / p.T, "plan": st.info()}
            finally:
                st.close()
        if "ms_per_forward" in rec.get("wavefront", {}) and \
                "ms_per_forward" in rec.get("layerwise", {}):
            rec["wavefront_speedup"] = (rec["layerwise"]["ms_per_forward"]
                                        / rec["wavefront"]["ms_per_forward"])
        out.append(rec)
    print(json.dumps({"stack": out}))
    return 0


def problem_by_name(name, T=None):
    """A named workload, or a point of the sweep by its name (sweep_h..._b..._d...)."""
    from persistent_rnn_recurrence_gb300 import synth
    if name.startswith("sweep_"):
        kw = dict(synth.sweep_points())[name]
        if T is not None:
            kw = {**kw, "T": T}
        return synth.make_problem(name=name, **kw)
    return synth.named_problem(name, T=T)


def run_backward(args):
    """Training-step timing (forward + backward through time) for the named
    workloads and two wide-batch sweep points at T = 256: the forward, the
    reverse recurrence and the batched gradient products, CUDA events, L2
    flushed before every step."""
    import numpy as np
    import torch
    from persistent_rnn_recurrence_gb300 import prnn, synth
    dev = torch.device("cuda", 0)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    reps = max(5, min(args.steps, 20))
    out = []
    for name in ("sparse_f16_h1792_d10_b4_t256", "dense_f16_h1152_b4_t256",
                 "sparse_f16_h5760_d1_b4_t256", "sparse_f16_h5760_d5_b4_t256",
                 "sweep_h1152_b32_d100", "sweep_h2304_b32_d100"):
        p = problem_by_name(name)
        lay = prnn.Layer.from_problem(p)
        kernel = "ksplit" if lay.info()["dense_ksplit"] else ("sparse" if p.sparse else "dense")
        lay.set_option(prnn.PRNN_OPT_TIMING, 1)
        x = torch.from_numpy(p.x).to(dev)
        h0 = None if p.h0 is None else torch.from_numpy(p.h0).to(dev)
        y = torch.empty((p.T, p.B, p.H), dtype=torch.float32, device=dev)
        dy = torch.from_numpy(np.random.default_rng(9).normal(
            size=(p.T, p.B, p.H)).astype(np.float32)).to(dev)
        g = lay.backward(x, lay.forward(x, h0, y), dy, h0)
        fwd, rev, prod, tot = [], [], [], []
        for _ in range(reps):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            prnn.prnn_forward(lay.h, p.T, p.B, x, h0, y)
            f = prnn.prnn_get_timing(lay.h)
            prnn.prnn_backward(lay.h, p.T, p.B, x, h0, y, dy, g["delta"], g["dx"], g["dh0"],
                               g["dWx"], g["dWh"], g["db"])
            e1.record()
            b = prnn.prnn_get_timing(lay.h)
            torch.cuda.synchronize()
            fwd.append(f[0] + f[1])
            prod.append(b[0])
            rev.append(b[1])
            tot.append(e0.elapsed_time(e1))
        assert lay.status() == prnn.PRNN_OK
        lay.close()
        med = lambda v: sorted(v)[len(v) // 2]
        out.append({"workload": name, "recurrent_kernel": kernel,
                    "ms_train_step": med(tot), "ms_forward": med(fwd),
                    "ms_reverse_recurrence": med(rev), "ms_gradient_products": med(prod),
                    "us_per_step_reverse": 1e3 * med(rev) / p.T,
                    "train_timesteps_per_s": p.T / (med(tot) * 1e-3)})
    print(json.dumps({"backward": out}))
    return 0


def vendor_loops(p, dev):
    """The per-step vendor-library recurrences of problem p, each step
    h_t = ReLU(P_t + Wh h_{t-1}) with P = Wx x + b precomputed in fp32 by one
    cuBLAS product: name -> (step(h_prev, P_t, h_next), P, h0).
      cublas_sgemm   fp32 GEMM (torch.addmm, no TF32) with Wh held densely;
      cublas_hgemm   the same in fp16 (h rounded to fp16 every step);
      cusparse_spmm  CSR SpMM (torch.sparse.mm), sparse layers only.
    The libraries run as shipped; nothing of theirs is inspected."""
    import numpy as np
    import torch
    torch.backends.cuda.matmul.allow_tf32 = False
    x = torch.from_numpy(p.x).to(dev)
    h0 = torch.zeros(p.B, p.H, device=dev) if p.h0 is None else torch.from_numpy(p.h0).to(dev)
    Wx = torch.from_numpy(p.Wx.astype(np.float32)).to(dev)
    P = (x.reshape(-1, p.I) @ Wx.T + torch.from_numpy(p.b).to(dev)).reshape(p.T, p.B, p.H)
    Wd = densified_wh(p)
    WdT = torch.from_numpy(Wd).to(dev).T.contiguous()
    WdT16 = WdT.half()

    def dense32(hp, Pt, hn):
        torch.addmm(Pt, hp, WdT, out=hn)
        hn.relu_()

    def dense16(hp, Pt, hn):
        torch.addmm(Pt, hp, WdT16, out=hn)
        hn.relu_()
    loops = {"cublas_sgemm": (dense32, P, h0), "cublas_hgemm": (dense16, P.half(), h0.half())}
    if p.sparse:
        Wcsr = torch.from_numpy(Wd).to(dev).to_sparse_csr()

        def sparse32(hp, Pt, hn):
            hn.copy_(torch.sparse.mm(Wcsr, hp.T).T)
            hn.add_(Pt).relu_()
        loops["cusparse_spmm"] = (sparse32, P, h0)
    return loops


def densified_wh(p):
    """Wh of problem p as a dense fp32 [H, H] array (exact: fp16 values)."""
    import numpy as np
    if not p.sparse:
        return p.Wh.astype(np.float32)
    Wd = np.zeros((p.H, p.H), np.float32)
    if getattr(p, "row_ptr", None) is not None:
        rows = np.repeat(np.arange(p.H), np.diff(p.row_ptr))
        Wd[rows, p.cols.astype(np.int64)] = p.vals.astype(np.float32)
    else:
        Wd[np.repeat(np.arange(p.H), p.k), p.cols.astype(np.int64).ravel()] = \
            p.vals.astype(np.float32).ravel()
    return Wd


def vendor_forward(step, P, h0, T):
    """Run T steps of one vendor loop eagerly; y [T, B, H] as fp32."""
    import torch
    hs = [h0] + [torch.empty_like(h0) for _ in range(T)]
    for t in range(T):
        step(hs[t], P[t], hs[t + 1])
    return torch.stack(hs[1:]).float()


def run_vendor(args):
    """The pages' comparison points, restated on GB300: the persistent
    kernels against per-step vendor-library products (``vendor_loops``), T
    steps captured in one CUDA graph where the library allows it, and for
    sparse layers the dense persistent kernel on the same matrix held densely
    (the sparse-versus-dense persistent row of the pages' table)."""
    import numpy as np
    import torch
    from persistent_rnn_recurrence_gb300 import prnn, synth
    dev = torch.device("cuda", 0)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    reps = max(5, min(args.steps, 10))

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        ms = []
        for _ in range(reps):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ms.append(e0.elapsed_time(e1))
        return sorted(ms)[len(ms) // 2]

    def per_step(T, P, h0, step):
        """T steps of `step` (h_prev -> h) into static buffers, as a CUDA graph
        when capture succeeds; returns (callable, captured)."""
        hs = [h0] + [torch.empty_like(h0) for _ in range(T)]

        def run():
            for t in range(T):
                step(hs[t], P[t], hs[t + 1])
        run()
        torch.cuda.synchronize()
        try:
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                run()
            torch.cuda.current_stream().wait_stream(s)
            with torch.cuda.graph(g):
                run()
            return g.replay, True
        except Exception:
            return run, False

    def persistent_us(lay, p, x, h0, y):
        lay.set_option(prnn.PRNN_OPT_TIMING, 1)
        rec_ms = []
        for _ in range(reps):
            flush.fill_(1.0)
            prnn.prnn_forward(lay.h, p.T, p.B, x, h0, y)
            rec_ms.append(prnn.prnn_get_timing(lay.h)[1])
        st = lay.status()
        if st != prnn.PRNN_OK:
            raise RuntimeError(prnn.prnn_status_string(st))
        return 1e3 * sorted(rec_ms)[len(rec_ms) // 2] / p.T

    cases = [("dense_f16_h1152_b4_t256", None), ("sparse_f16_h1792_d10_b4_t256", None)]
    extra = [(1152, 0.10), (1792, 0.01), (2304, 0.10), (5760, 0.01), (5760, 0.05)]
    out = []
    problems = [synth.named_problem(n) for n, _ in cases]
    problems += [synth.make_problem(H=H, B=4, T=256, k=synth.sparse_k(H, d), seed=3300 + i,
                                    name=f"sparse_f16_h{H}_d{int(round(d * 100))}_b4_t256")
                 for i, (H, d) in enumerate(extra)]
    for p in problems:
        rec = {"workload": p.name}
        x = torch.from_numpy(p.x).to(dev)
        h0 = torch.zeros(p.B, p.H, device=dev) if p.h0 is None else torch.from_numpy(p.h0).to(dev)
        y = torch.empty(p.T, p.B, p.H, device=dev)
        lay = prnn.Layer.from_problem(p)
        rec["persistent_us_per_step"] = persistent_us(lay, p, x, h0, y)
        lay.close()
        if p.sparse:
            # the same matrix held densely (fp16) in the dense persistent kernel
            pd = dataclasses.replace(p, Wh=densified_wh(p).astype(np.float16), vals=None,
                                     cols=None, row_ptr=None, name=p.name + "_held_densely")
            try:
                lay = prnn.Layer.from_problem(pd)
            except prnn.PrnnError as e:
                rec["dense_persistent"] = {"unsupported": str(e)}
            else:
                rec["dense_persistent_us_per_step"] = persistent_us(lay, pd, x, h0, y)
                rec["sparse_vs_dense_persistent"] = (rec["dense_persistent_us_per_step"]
                                                     / rec["persistent_us_per_step"])
                lay.close()
        for key, (fn, Pv, hv) in vendor_loops(p, dev).items():
            try:
                f, cap = per_step(p.T, Pv, hv, fn)
                rec[key + "_us_per_step"] = 1e3 * timed(f) / p.T
                rec[key + "_graph"] = cap
            except Exception as e:  # e.g. a sparse product missing from the installed PyTorch
                rec[key + "_error"] = str(e)[:120]
        best_dense = min(rec["cublas_sgemm_us_per_step"], rec["cublas_hgemm_us_per_step"])
        rec["persistent_vs_dense_gemm"] = best_dense / rec["persistent_us_per_step"]
        if "cusparse_spmm_us_per_step" in rec:
            rec["persistent_vs_sparse_gemm"] = (rec["cusparse_spmm_us_per_step"]
                                                / rec["persistent_us_per_step"])
        out.append(rec)
        print(json.dumps(rec), flush=True)
    return 0


TRACE_PHASES = ["loop", "p_request", "pause", "wait_h", "stage_to_barrier", "gather", "reduce",
                "publish"]


def trace_phases(rec, clock_mhz, groups=1):
    """Where a step's time goes, from trace records rec [R, T, n_cta, 17, 16]
    (uint32; slot 0 the CTA header, slot 1 + w warp w).  For every working CTA
    and step 1 .. T-1 the CTA's critical path is taken as the latest warp at
    each stamp, and the step is cut at those stamps: previous publish -> pass
    start -> projection value requested -> pause end -> last poll fresh ->
    barrier -> gathers -> reduction -> publish (SM-clock differences, mod
    2^32).  Across CTAs, the globaltimer readings give the exchange: for each
    CTA, its barrier time minus the last publish of the previous step in its
    group ("exchange"), and the spread of the group's publishes ("publish_skew").
    Returns {name: ns array} plus "rounds" and the timer's resolution."""
    import numpy as np
    r = rec.astype(np.int64)
    hdr = r[:, :, :, 0, :]
    nw = int(hdr[..., 2].max())
    n = r.shape[2]
    active = hdr[0, 0, :, 1] == np.arange(n)
    cta_group = np.arange(n) // max(1, n // groups)
    w = r[:, :, :, 1:1 + nw, :]
    base = w[..., 0].min(axis=3, keepdims=True)            # unwrap relative to the pass start
    rel = (w[..., :8] - base[..., None]) & 0xffffffff
    rel = np.where(rel >= (1 << 31), rel - (1 << 32), rel)
    m = rel.max(axis=3)                                     # [R, T, C, 8]: latest warp
    pub = m[..., 7] + base[..., 0]                          # absolute publish (latest warp)
    ns = 1e3 / clock_mhz
    T = r.shape[1]
    sl = slice(1, T)
    d = lambda a, b: (((b - a) + (1 << 31)) & 0xffffffff) - (1 << 31)
    out = {"loop": d(pub[:, :-1], m[:, sl, :, 0] + base[:, sl, :, 0])}
    for i, name in enumerate(TRACE_PHASES[1:]):
        out[name] = m[:, sl, :, i + 1] - m[:, sl, :, i]
    out["step"] = d(pub[:, :-1], pub[:, sl])
    out["gather_warp"] = rel[:, sl, :, :, 5] - rel[:, sl, :, :, 4]
    out["trace_record_write"] = d(w[:, sl, :, :, 7], w[:, sl, :, :, 13])
    out = {k: np.asarray(v, dtype=np.float64)[:, :, active].ravel() * ns if k != "gather_warp"
           else np.asarray(v, dtype=np.float64)[:, :, active].ravel() * ns
           for k, v in out.items()}
    gbar = ((w[..., 10] << 32) | w[..., 9]).max(axis=3)      # [R, T, C] ns
    gpub = ((w[..., 12] << 32) | w[..., 11]).max(axis=3)
    exch, skew = [], []
    for g in np.unique(cta_group[active]):
        cs = np.nonzero(active & (cta_group == g))[0]
        last_pub = gpub[:, :-1][:, :, cs].max(axis=2)        # [R, T-1]
        first_pub = gpub[:, :-1][:, :, cs].min(axis=2)
        exch.append((gbar[:, 1:][:, :, cs] - last_pub[:, :, None]).ravel())
        skew.append((last_pub - first_pub).ravel())
    out["exchange"] = np.concatenate(exch).astype(np.float64)
    out["publish_skew"] = np.concatenate(skew).astype(np.float64)
    out["rounds"] = w[:, sl, :, :, 8].max(axis=3)[:, :, active].ravel()
    u = np.unique(gbar)
    du = np.diff(u)
    out["globaltimer_resolution_ns"] = float(du[du > 0].min()) if du.size else 0.0
    return out


def run_trace(args):
    """Where the time of one step of the sparse persistent kernel goes: runs
    the config's layer for --trace-steps steps with the phase trace on (L2
    flushed before each forward), checks the traced output equals the
    untraced one bit for bit, and prints one JSON line of per-phase medians
    and spreads (ns), the re-poll statistics and the trace's own overhead.
    --trace-out saves the raw records (numpy .npy)."""
    import numpy as np
    import torch
    from persistent_rnn_recurrence_gb300 import prnn, synth
    dev = torch.device("cuda", 0)
    p = problem_by_name(args.config, T=args.trace_steps)
    if not p.sparse:
        return run_trace_ksplit(args, p)
    lay = prnn.Layer.from_problem(p)
    lay.set_option(prnn.PRNN_OPT_TIMING, 1)
    info = lay.info()
    x = torch.from_numpy(p.x).to(dev)
    y0 = torch.empty(p.T, p.B, p.H, device=dev)
    y1 = torch.empty_like(y0)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    n_cta = info["n_cta"]
    W = 17 * 16
    buf = torch.full((p.T * n_cta * W,), -1, dtype=torch.int32, device=dev)
    reps = max(3, min(args.steps, 20))

    def runs(traced):
        prnn.prnn_set_trace_buffer(lay.h, buf if traced else None, buf.numel() * 4)
        ms, recs = [], []
        for i in range(reps + 2):
            flush.fill_(1.0)
            prnn.prnn_forward(lay.h, p.T, p.B, x, None, y1 if traced else y0)
            t = prnn.prnn_get_timing(lay.h)[1]
            if i >= 2:
                ms.append(t)
                if traced:
                    recs.append(buf.view(p.T, n_cta, 17, 16).cpu().numpy().view(np.uint32).copy())
        return sorted(ms)[len(ms) // 2], recs

    ms_plain, _ = runs(False)
    ms_traced, recs = runs(True)
    prnn.prnn_set_trace_buffer(lay.h, None, 0)
    torch.cuda.synchronize()
    st = lay.status()
    lay.close()
    same = bool(torch.equal(y0, y1))
    clock_mhz = load_peaks().get("sm_max_mhz", 2070.0)  # the SM clock under load
    rec = np.stack(recs)
    if args.trace_out:
        np.save(args.trace_out, rec[:2])
    ph = trace_phases(rec, clock_mhz, info["cta_groups"])

    def stats(a):
        a = np.sort(np.asarray(a, dtype=np.float64))
        q = lambda f: float(a[min(len(a) - 1, int(f * len(a)))])
        return {"median": q(0.5), "p10": q(0.1), "p90": q(0.9), "mean": float(a.mean())}

    line = {"trace": p.name, "T": p.T, "B": p.B, "n_cta": n_cta,
            "cta_groups": info["cta_groups"], "rows_per_cta": info["rows_per_cta"],
            "threads_per_cta": info["threads_per_cta"], "threads_per_row": info["threads_per_row"],
            "k_padded": info["k_padded"], "status": prnn.prnn_status_string(st),
            "traced_equals_untraced": same, "clock_mhz_assumed": clock_mhz,
            "recurrence_us_per_step": {"plain": 1e3 * ms_plain / p.T,
                                       "traced": 1e3 * ms_traced / p.T},
            "samples": int(ph["step"].size),
            "phases_ns": {k: stats(ph[k]) for k in TRACE_PHASES + ["step", "gather_warp",
                                                                  "trace_record_write",
                                                                  "exchange", "publish_skew"]},
            "repoll": {"mean_rounds": float(ph["rounds"].mean()),
                       "frac_ctas_first_poll_fresh": float((ph["rounds"] == 0).mean()),
                       "max_rounds": int(ph["rounds"].max())},
            "globaltimer_resolution_ns": ph["globaltimer_resolution_ns"]}
    print(json.dumps(line), flush=True)
    return 0 if same and st == prnn.PRNN_OK else 1


KSPLIT_PHASES = [("fill_own", 4, 5), ("fill_wait", 5, 6), ("mma", 6, 7), ("mma_issue", 6, 13),
                 ("stage", 7, 8), ("send", 8, 9), ("barrier2", 9, 10), ("receive", 10, 11),
                 ("publish", 11, 12)]


def ksplit_trace_phases(rec, clock_mhz):
    """Where a step of the dense K-split kernel goes, from trace records rec
    [R, T, n_cta, 20] (uint32 words of the kernel's record).  Per CTA and step
    1 .. T-1: SM-clock differences between its stamps (ns), the step (step
    start to step start), and from the globaltimer readings the exchange: its
    first barrier minus the last publish of the previous step over all CTAs
    (the slices draw on several clusters), and the spread of each step's
    publishes across CTAs."""
    import numpy as np
    r = rec.astype(np.int64)
    ns = 1e3 / clock_mhz
    d = lambda a, b: ((((b - a) + (1 << 31)) & 0xffffffff) - (1 << 31)).astype(np.float64)
    sl = slice(1, r.shape[1])
    out = {name: d(r[:, sl, :, a], r[:, sl, :, b]).ravel() * ns for name, a, b in KSPLIT_PHASES}
    out["step"] = d(r[:, :-1, :, 4], r[:, sl, :, 4]).ravel() * ns
    gbar = (r[..., 15] << 32) | r[..., 14]
    gpub = (r[..., 17] << 32) | r[..., 16]
    last_pub = gpub.max(axis=2)                       # [R, T]
    out["exchange"] = (gbar[:, sl, :] - last_pub[:, :-1, None]).astype(np.float64).ravel()
    out["publish_skew"] = (gpub.max(axis=2) - gpub.min(axis=2))[:, sl].astype(np.float64).ravel()
    out["rounds"] = r[:, sl, :, 18].ravel()
    return out


def run_trace_ksplit(args, p):
    """--trace for a dense layer that runs the K-split kernel: per-phase
    medians and spreads (ns) of its steps, the traced output checked against
    the untraced one bit for bit."""
    import numpy as np
    import torch
    from persistent_rnn_recurrence_gb300 import prnn
    dev = torch.device("cuda", 0)
    lay = prnn.Layer.from_problem(p)
    lay.set_option(prnn.PRNN_OPT_TIMING, 1)
    info = lay.info()
    if not info["dense_ksplit"]:
        lay.close()
        raise SystemExit("--trace needs a sparse layer or a dense one that runs the K-split kernel")
    x = torch.from_numpy(p.x).to(dev)
    y0 = torch.empty(p.T, p.B, p.H, device=dev)
    y1 = torch.empty_like(y0)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    n_cta = info["n_cta"]
    W = 17 * 16
    buf = torch.full((p.T * n_cta * W,), -1, dtype=torch.int32, device=dev)
    reps = max(3, min(args.steps, 20))

    def runs(traced):
        prnn.prnn_set_trace_buffer(lay.h, buf if traced else None, buf.numel() * 4)
        ms, recs = [], []
        for i in range(reps + 2):
            flush.fill_(1.0)
            prnn.prnn_forward(lay.h, p.T, p.B, x, None, y1 if traced else y0)
            t = prnn.prnn_get_timing(lay.h)[1]
            if i >= 2:
                ms.append(t)
                if traced:
                    recs.append(buf.view(p.T, n_cta, W)[..., :20].cpu().numpy().view(np.uint32).copy())
        return sorted(ms)[len(ms) // 2], recs

    ms_plain, _ = runs(False)
    ms_traced, recs = runs(True)
    prnn.prnn_set_trace_buffer(lay.h, None, 0)
    torch.cuda.synchronize()
    st = lay.status()
    lay.close()
    same = bool(torch.equal(y0, y1))
    clock_mhz = load_peaks().get("sm_max_mhz", 2070.0)
    ph = ksplit_trace_phases(np.stack(recs), clock_mhz)

    def stats(a):
        a = np.sort(np.asarray(a, dtype=np.float64))
        q = lambda f: float(a[min(len(a) - 1, int(f * len(a)))])
        return {"median": q(0.5), "p10": q(0.1), "p90": q(0.9), "mean": float(a.mean())}

    names = [n for n, _, _ in KSPLIT_PHASES] + ["step", "exchange", "publish_skew"]
    line = {"trace": p.name, "kernel": "recur_dense_ksplit_kernel", "T": p.T, "B": p.B, "H": p.H,
            "n_cta": n_cta, "cluster_size": info["dense_ksplit"],
            "status": prnn.prnn_status_string(st), "traced_equals_untraced": same,
            "clock_mhz_assumed": clock_mhz,
            "recurrence_us_per_step": {"plain": 1e3 * ms_plain / p.T,
                                       "traced": 1e3 * ms_traced / p.T},
            "samples": int(ph["step"].size),
            "phases_ns": {k: stats(ph[k]) for k in names},
            "repoll": {"mean_rounds": float(ph["rounds"].mean()),
                       "max_rounds": int(ph["rounds"].max())}}
    print(json.dumps(line), flush=True)
    return 0 if same and st == prnn.PRNN_OK else 1


def run_cluster_probe(args):
    """The exchange of h inside thread-block clusters through distributed
    shared memory (prnn_probe_cluster_exchange: no arithmetic, every word
    checked), at the sizes of the named layers, beside the L2 exchange floor
    of the config's layer (prnn_probe_sync_floor, same grid as its forward).
    One JSON line: ns per step for each cluster size, with one cluster per
    batch column of the config (B clusters) and with as many clusters as the
    device holds at once."""
    import torch
    from persistent_rnn_recurrence_gb300 import prnn, synth
    torch.cuda.init()
    p = synth.named_problem(args.config)
    lay = prnn.Layer.from_problem(p)
    lay.set_option(prnn.PRNN_OPT_TIMING, 1)
    ys = torch.empty(p.T, p.B, p.H, device="cuda")
    fl = []
    for _ in range(7):
        prnn.prnn_probe_sync_floor(lay.h, p.T, p.B, ys)
        fl.append(prnn.prnn_get_timing(lay.h)[1])
    lay.close()
    fl.sort()
    out = {"metric": "step exchange ns per step (no arithmetic)", "config": {"workload": args.config},
           "l2_sync_floor_ns_per_step": 1e6 * fl[len(fl) // 2] / p.T, "cluster": []}
    steps = 400
    for H in (p.H, 5760):
        for cs in (2, 4, 8, 16):
            row = {"hidden": H, "cluster_size": cs}
            if H % (4 * cs):
                continue
            for key, n in (("b_clusters", p.B), ("max_clusters", 152 // cs)):
                while n >= 1:
                    try:
                        ns, bad = prnn.prnn_probe_cluster_exchange(H, cs, n, steps)
                        best = ns
                        for _ in range(2):  # best of three
                            ns, b2 = prnn.prnn_probe_cluster_exchange(H, cs, n, steps)
                            best, bad = min(best, ns), bad + b2
                        row[key] = {"clusters": n, "ns_per_step": best, "wrong_words": bad}
                        break
                    except prnn.PrnnError as e:
                        if e.status != prnn.PRNN_ERR_UNSUPPORTED:
                            raise
                        n -= 1
            out["cluster"].append(row)
    print(json.dumps(out), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.ablation:
        return run_ablation(args)
    if args.balance:
        return run_balance(args)
    if args.stack:
        return run_stack(args)
    if args.backward:
        return run_backward(args)
    if args.trace:
        return run_trace(args)
    if args.vendor:
        return run_vendor(args)
    if args.cluster_probe:
        return run_cluster_probe(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
