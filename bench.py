"""Benchmark of the logsumexp hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-e2e] [--no-cpu-baseline]

One step is one call of the library on one batch of the workload (default
log_softmax over the last axis of fp32 x[4096, 393216]: rows a2 + a3 of the
path, one kernel launch).  Prints one JSON line (rank 0).  Under torchrun each
rank runs the whole workload on its own GPU (independent batches, weak
scaling) with no data-path collective; the timed region is bracketed by a
barrier and a device synchronize, and the slowest rank's time is reported.

--impl reference times the CPU oracle (a plain double-precision C
implementation) on a bounded sample of the same workload, on rank 0 only.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "achieved HBM GB/s and % of GB300 peak, log_softmax fp32 4096x393216"
DEFAULT_WORKLOAD = "log_softmax_4096x393216"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


# ------------------------------------------------------------------ workloads

def algorithmic_bytes(w: synth.Workload) -> int:
    """Unique bytes one step must move: each input element read once, each output
    element written once (fp32)."""
    if w.op == "lse_dim0":
        R = w.shape[0]
        inner = w.numel // R
        return 4 * (w.numel + inner)
    if w.op in ("log_softmax", "softmax", "log_softmax_dim0"):
        return 4 * 2 * w.numel
    if w.op == "gn_act_lse":
        N, C, H, W = w.shape
        return 4 * (w.numel + 2 * C + N * H * W)
    if w.op in GN_ELEMENTWISE:
        C = w.shape[1]
        return 4 * (2 * w.numel + 2 * C)
    if w.op == "conv_gn_act_lse":
        # x once, y written once by the conv and read once by the GroupNorm pass, out;
        # weights, bias, gamma, beta
        N, Cin, H, W = w.shape
        Cout = w.params["Cout"]
        ohw = (H - 2) * (W - 2)
        return 4 * (w.numel + 2 * N * Cout * ohw + N * ohw + Cout * (Cin * 9 + 3))
    raise KeyError(w.op)


GN_ELEMENTWISE = ("group_norm", "gn_act_residual")

# Kernels each step launches (the dominant kernel first).
LAUNCHES = {
    "lse_dim0": ["lse_strided_kernel"],
    "log_softmax": ["lsm_ws_kernel"],
    "gn_act_lse": ["gn_fused_kernel"],
    "softmax": ["lsm_ws_kernel"],
    "log_softmax_dim0": ["lse_strided_kernel"],
    "group_norm": ["gn_tma_kernel"],
    "gn_act_residual": ["gn_tma_kernel"],
    "conv_gn_act_lse": ["conv2d_tc_kernel", "gn_fused_kernel"],
}


def make_step(L, w: synth.Workload, inputs, out, stream):
    if w.op == "lse_dim0":
        R = w.shape[0]
        inner = w.numel // R
        x = inputs["x"]
        return lambda: L.lse_reduce(x, out, 1, R, inner, stream=stream)
    if w.op in ("log_softmax", "softmax"):
        rows, cols = w.shape
        x = inputs["x"]
        fn = L.log_softmax_lastdim if w.op == "log_softmax" else L.softmax_lastdim
        return lambda: fn(x, out, rows, cols, stream=stream)
    if w.op == "log_softmax_dim0":
        R = w.shape[0]
        inner = w.numel // R
        x = inputs["x"]
        return lambda: L.log_softmax_dim(x, out, 1, R, inner, stream=stream)
    if w.op == "conv_gn_act_lse":
        N, Cin, H, W = w.shape
        x, wt, b, g, be = (inputs[k] for k in ("x", "w", "bias", "gamma", "beta"))
        G, eps, Cout = w.params["G"], w.params["eps"], w.params["Cout"]
        return lambda: L.conv_gn_act_lse(x, wt, b, g, be, out, N, Cin, H, W, Cout, G, eps, stream=stream)
    if w.op == "gn_act_lse" or w.op in GN_ELEMENTWISE:
        N, C, H, W = w.shape
        y, g, b = inputs["y"], inputs["gamma"], inputs["beta"]
        G, eps = w.params["G"], w.params["eps"]
        fn = getattr(L, w.op)
        return lambda: fn(y, g, b, out, N, C, H * W, G, eps, stream=stream)
    raise KeyError(w.op)


def out_shape(w: synth.Workload):
    if w.op == "lse_dim0":
        return w.shape[1:]
    if w.op == "gn_act_lse":
        N, C, H, W = w.shape
        return (N, 1, H, W)
    if w.op == "conv_gn_act_lse":
        N, Cin, H, W = w.shape
        return (N, 1, H - 2, W - 2)
    return w.shape


def oracle_call(w: synth.Workload, inputs) -> int:
    """Runs the oracle on host inputs of the workload's kind (any size); returns
    the algorithmic bytes of that call."""
    import oracle
    if w.op in ("log_softmax", "softmax"):
        x = inputs["x"]
        (oracle.log_softmax if w.op == "log_softmax" else oracle.softmax)(x)
        return 8 * x.numel()
    if w.op in ("lse_dim0", "log_softmax_dim0"):
        x = inputs["x"].reshape(inputs["x"].shape[0], -1)
        if w.op == "lse_dim0":
            oracle.lse_reduce(x, 1, x.shape[0], x.shape[1])
            return 4 * (x.numel() + x.shape[1])
        oracle.log_softmax_dim(x, 1, x.shape[0], x.shape[1])
        return 8 * x.numel()
    if w.op == "conv_gn_act_lse":
        x = inputs["x"]
        oracle.conv_gn_act_lse(x, inputs["w"], inputs["bias"], inputs["gamma"], inputs["beta"], w.params["G"],
                               w.params["eps"])
        N, Cin, H, W = x.shape
        Cout = w.params["Cout"]
        ohw = (H - 2) * (W - 2)
        return 4 * (x.numel() + 2 * N * Cout * ohw + N * ohw)
    y, g, b = inputs["y"], inputs["gamma"], inputs["beta"]
    getattr(oracle, w.op)(y, g, b, w.params["G"], w.params["eps"])
    if w.op == "gn_act_lse":
        return 4 * (y.numel() + y.shape[0] * y.shape[2] * y.shape[3])
    return 8 * y.numel()


# ------------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(v: float, world: int, device=None) -> float:
    """The largest v over all ranks (the slowest rank's time)."""
    if world <= 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(v: float, world: int, device=None) -> float:
    if world <= 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def rank_seed_offset(rank: int) -> int:
    """Each rank draws its own batch: seeds shifted by 1000 * rank."""
    return 1000 * rank


# ------------------------------------------------------------------ peaks, traffic, clocks

def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources that determine each dominant kernel's code (with the shared headers).
KERNEL_SOURCES = {
    "lsm_ws_kernel": ["log_softmax.cu"],
    "lse_strided_kernel": ["lse_strided.cu"],
    "gn_fused_kernel": ["gn_act_lse.cu", "gn_common.cuh"],
    "gn_tma_kernel": ["gn_tma.cu", "gn_common.cuh"],
    "conv2d_tc_kernel": ["conv.cu", "conv_tile.cuh", "gn_common.cuh"],
}


def kernel_source_sha(kernel: str) -> str:
    """sha256 (first 16 hex digits) over the kernel's source files and common.cuh (the
    device code it is built from; launch.h holds host declarations only)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "log_softmax_gb300", "csrc")
    for f in sorted(KERNEL_SOURCES[kernel] + ["common.cuh"]):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + b"\0" + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary, or None
    when none was taken or the kernels changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    sha = kernel_source_sha(kernel)
    with open(p) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kv = dict(item.split("=", 1) for item in line.split() if "=" in item)
            if kv.get("kernel") == kernel and kv.get("workload") == workload:
                if kv.get("source_sha") != sha:
                    return None
                return float(kv["bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, every 100 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []  # (wall time, fields)
        self.proc = None
        self.thread = None
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            pass
        self.target = (["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid] if uuid else
                       ["-i", str(device_index)])

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.target, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.strip().split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        window = "timed region"
        if not inside:
            inside = [p for (_, p) in self.samples]
            window = "whole run (no sample fell inside the timed region)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(p[0]) for p in inside if num(p[0]) is not None]
        smax = [num(p[1]) for p in inside if num(p[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in inside for n, v in zip(names, p[4:8]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(inside), "window": window}


# ------------------------------------------------------------------ CPU oracle timing

def host_cpu() -> str:
    """The host's logical core count and CPU model (for the CPU baseline's record)."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware") and ":" in line:
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not model:
        import platform
        model = platform.machine()
    return f"{os.cpu_count()} logical cores, {model}"


def time_oracle(w: synth.Workload, sample, budget_s: float, unit: int):
    """Runs the oracle over successive slices of `unit` rows / columns / samples of
    the host sample, cycling through it, until budget_s has passed.  Returns
    (bytes, seconds, slices done)."""
    if w.op in ("lse_dim0", "log_softmax_dim0"):
        n_units = sample["x"].shape[1] // unit
    else:
        n_units = sample["x" if "x" in sample else "y"].shape[0] // unit
    n_units = max(1, n_units)
    t0 = time.perf_counter()
    done_bytes = 0
    units = 0
    while True:
        k = units % n_units
        if w.op in ("lse_dim0", "log_softmax_dim0"):
            sl = {"x": sample["x"][:, k * unit:(k + 1) * unit].contiguous()}
        elif w.op == "conv_gn_act_lse":
            sl = dict(sample, x=sample["x"][k * unit:(k + 1) * unit])
        elif "x" in sample:
            sl = {"x": sample["x"][k * unit:(k + 1) * unit]}
        else:
            sl = dict(sample, y=sample["y"][k * unit:(k + 1) * unit])
        done_bytes += oracle_call(w, sl)
        units += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return done_bytes, time.perf_counter() - t0, units


def _units_of(w: synth.Workload, sample) -> int:
    if w.op in ("lse_dim0", "log_softmax_dim0"):
        return sample["x"].shape[1]
    return sample["x" if "x" in sample else "y"].shape[0]


def _share(w: synth.Workload, sample, lo: int, hi: int):
    """Units [lo, hi) of a host sample (rows, columns or samples, as time_oracle slices)."""
    if w.op in ("lse_dim0", "log_softmax_dim0"):
        return {"x": sample["x"][:, lo:hi].contiguous()}
    if w.op == "conv_gn_act_lse":
        return dict(sample, x=sample["x"][lo:hi])
    if "x" in sample:
        return {"x": sample["x"][lo:hi]}
    return dict(sample, y=sample["y"][lo:hi])


def time_oracle_threads(w: synth.Workload, sample, budget_s: float, unit: int, threads: int):
    """The oracle as it stands on `threads` host threads at once (its C calls run
    without the interpreter lock), each cycling over its own disjoint share of the
    sample for budget_s.  Returns (bytes, seconds, threads used, slices done)."""
    n = _units_of(w, sample) // unit
    threads = max(1, min(threads, n))
    shares = [_share(w, sample, (n * i // threads) * unit, (n * (i + 1) // threads) * unit) for i in range(threads)]
    results = [None] * threads
    errors = []

    def run(i):
        try:
            results[i] = time_oracle(w, shares[i], budget_s, unit)
        except Exception as e:  # reported to the caller
            errors.append(e)

    ts = [threading.Thread(target=run, args=(i,)) for i in range(threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    if errors:
        raise errors[0]
    return sum(r[0] for r in results), max(r[1] for r in results), threads, sum(r[2] for r in results)


def host_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_sample(w: synth.Workload, inputs_dev, rows: int):
    """The first `rows` units (rows / columns / samples) of the workload on the
    host, and the slice size one oracle call takes."""
    if w.op in ("log_softmax", "softmax"):
        return {"x": inputs_dev["x"][:rows].cpu().contiguous()}, 1
    if w.op in ("lse_dim0", "log_softmax_dim0"):
        R = w.shape[0]
        inner = w.numel // R
        cols = min(inner, rows * 4096)
        return {"x": inputs_dev["x"].view(R, inner)[:, :cols].cpu().contiguous()}, 4096
    if w.op == "conv_gn_act_lse":
        smp = {k: v.cpu().contiguous() for k, v in inputs_dev.items() if k != "x"}
        smp["x"] = inputs_dev["x"][:max(1, rows // 64)].cpu().contiguous()
        return smp, 1
    y = inputs_dev["y"][:max(1, rows // 64)].cpu().contiguous()
    return {"y": y, "gamma": inputs_dev["gamma"].cpu(), "beta": inputs_dev["beta"].cpu()}, 1


def sample_text(w: synth.Workload, sample, units: int) -> str:
    if w.op in ("log_softmax", "softmax"):
        return f"{units} row passes over the first {sample['x'].shape[0]} rows x {w.shape[1]}"
    if w.op in ("lse_dim0", "log_softmax_dim0"):
        return (f"{units} passes of R={w.shape[0]} x 4096 columns over the first "
                f"{sample['x'].shape[1]} columns")
    key = "x" if w.op == "conv_gn_act_lse" else "y"
    return (f"{units} sample passes over the first {sample[key].shape[0]} samples of "
            f"{list(w.shape[1:])}")


# ------------------------------------------------------------------ arms

def run_reference(args, w: synth.Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    shape = list(w.shape)
    # one step = a bounded sample: 4 rows / 4096x32 columns / 1 sample
    if w.op in ("log_softmax", "softmax"):
        shape[0] = min(shape[0], 4)
        sample = f"{shape[0]} rows of {w.shape[1]}"
    elif w.op in ("lse_dim0", "log_softmax_dim0"):
        shape[1:] = [1, min(w.numel // w.shape[0], 4096 * 32)]
        sample = f"R={w.shape[0]} x {shape[2]} columns"
    else:
        shape[0] = 1
        sample = "1 sample of the chain"
    inputs = synth.make_inputs(w, shape=tuple(shape))
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        nbytes = oracle_call(w, inputs)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / len(times), 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "shape": list(w.shape), "recipe": w.recipe,
                   "sample_per_step": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample + " per step (single-threaded C, double precision)",
                         "host": host_cpu()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, w: synth.Workload):
    world, rank, local = dist_env()
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    init_dist(world, backend)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from log_softmax_gb300 import build as libbuild
    libbuild.build()
    import log_softmax_gb300 as L
    L.load_library()

    # inputs resident in HBM before the timed region
    seed_shift = rank_seed_offset(rank)
    params = dict(w.params)
    for k in list(params):
        if k.endswith("seed"):
            params[k] = params[k] + seed_shift
    wr = synth.Workload(w.name, w.op, w.shape, w.recipe, params)
    inputs = synth.make_inputs(wr, device=dev)
    out = torch.empty(out_shape(w), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    step = make_step(L, w, inputs, out, stream)
    nbytes = algorithmic_bytes(w)
    in_bytes = sum(t.numel() * 4 for t in inputs.values())
    flush = None
    if in_bytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    for _ in range(args.warmup):
        if flush is not None:
            flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)
    if L.lse_device_status() != 0:
        raise SystemExit("device status reported a bounded-wait timeout during warm-up")

    sampler = ClockSampler(local).start() if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_all0.record(stream)
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(1.0)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    wall1 = time.time()
    if sampler:
        time.sleep(0.15)
        sampler.stop()
    status = L.lse_device_status()

    per_step_ms = [a.elapsed_time(b) for a, b in ev]
    kernel_ms = sum(per_step_ms)
    region_ms = t_all0.elapsed_time(t_all1)
    # With inputs larger than L2 nothing runs between steps: time the whole region.
    # Otherwise an L2 flush runs between steps; time the steps alone.
    local_ms = kernel_ms if flush is not None else region_ms
    slow_ms = max_over_ranks(local_ms, world, dev)
    total_bytes = sum_over_ranks(float(nbytes * args.steps), world, dev)
    value = total_bytes / (slow_ms / 1e3) / 1e9

    # roofline of the dominant kernel (one launch of it per step)
    peak, peak_kind = hbm_peak()
    launch_ms = statistics.mean(per_step_ms)
    achieved = nbytes / (launch_ms / 1e3) / 1e9
    dominant = LAUNCHES[w.op][0]
    achieved_note = ("one launch per step" if len(LAUNCHES[w.op]) == 1 else
                     f"{len(LAUNCHES[w.op])} launches per step ({', '.join(LAUNCHES[w.op])}); achieved over the whole step")
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": ncu_traffic(dominant, w.name),
                "kernel": dominant, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6800 GB/s",
                "note": achieved_note}

    # end to end through the public API: pinned host in -> device -> host out, every step
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(L, w, inputs, args, dev, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        sample, unit = oracle_sample(w, inputs, 256)
        b, s, units = time_oracle(w, sample, budget_s=args.cpu_seconds, unit=unit)
        what = sample_text(w, sample, units)
        cpu = {"value": round(b / s / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": what + f", {s:.1f} s single-threaded", "host": host_cpu()}
        try:
            # the same oracle on every host core, each thread on its own share
            nthr = host_threads()
            per_sample = w.op in ("gn_act_lse", "group_norm", "gn_act_residual", "conv_gn_act_lse")
            big, unit2 = oracle_sample(w, inputs, 64 * nthr if per_sample else 256)
            b2, s2, used, done2 = time_oracle_threads(w, big, args.cpu_seconds, unit2, nthr)
            cpu["all_cores"] = {"value": round(b2 / s2 / 1e9, 4), "unit": "GB/s", "cores": used,
                                "sample": f"{sample_text(w, big, done2)}, split over {used} threads, {s2:.1f} s"}
        except Exception as e:  # the single-threaded figure stands alone
            cpu["all_cores"] = {"unavailable": repr(e)[:200]}

    if rank != 0:
        return 0
    clocks = sampler.summary(wall0, wall1) if sampler else None
    line = {
        "metric": METRIC if w.name == DEFAULT_WORKLOAD else
        f"achieved HBM GB/s and % of GB300 peak, {w.name}",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(slow_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "shape": list(w.shape), "recipe": w.recipe,
                   "algorithmic_bytes_per_step": nbytes,
                   "l2": ("inputs larger than L2 (129 MB); no flush" if flush is None else
                          "L2 flushed (256 MB write) between steps; steps timed alone"),
                   "parallelism": f"replicas x{world} (independent batches)"},
        "roofline": roofline,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "gpu_launches": len(LAUNCHES[w.op]) * args.steps,
        "device_status": L.lse_status_string(status),
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def host_link(host_in, dev, max_bytes=1 << 30, min_bytes=64 << 20):
    """Copy-engine bandwidth of this process's host link on its own pinned input buffer
    (after the end-to-end timing, which no longer needs it): host to device from its
    first half, device to host into its second half, and both at once (two streams),
    GB/s.  None when the buffer is too small to time bandwidth rather than latency."""
    buf = max(host_in.values(), key=lambda t: t.numel()).view(-1)
    n = int(min(buf.numel() // 2, max_bytes // 4))
    if n * 4 < min_bytes:
        return None
    src, dst = buf[:n], buf[n:2 * n]
    a = torch.empty(n, device=dev)
    b = torch.empty(n, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        fn()
        torch.cuda.synchronize(dev)
        return time.perf_counter() - t0

    def both():
        with torch.cuda.stream(s1):
            b.copy_(src, non_blocking=True)
        with torch.cuda.stream(s2):
            dst.copy_(a, non_blocking=True)

    # every direction once untimed (the first copy into fresh pinned pages pays for
    # mapping them), then the best of two timings of each
    a.copy_(src, non_blocking=True)
    dst.copy_(a, non_blocking=True)
    both()
    torch.cuda.synchronize(dev)
    h2d = n * 4 / min(timed(lambda: a.copy_(src, non_blocking=True)) for _ in range(2)) / 1e9
    d2h = n * 4 / min(timed(lambda: dst.copy_(a, non_blocking=True)) for _ in range(2)) / 1e9
    bi = 2 * n * 4 / min(timed(both) for _ in range(2)) / 1e9
    return {"h2d_gbs": round(h2d, 1), "d2h_gbs": round(d2h, 1), "both_gbs": round(bi, 1), "bytes_each": n * 4}


def e2e_ceiling(nbytes, h2d_bytes, d2h_bytes, link):
    """The e2e value (algorithmic bytes per second, GB/s) if every step took only the
    time its copies need on `link`: one direction at a time, or both at once."""
    t = max(h2d_bytes / (link["h2d_gbs"] * 1e9), d2h_bytes / (link["d2h_gbs"] * 1e9),
            (h2d_bytes + d2h_bytes) / (link["both_gbs"] * 1e9))
    return nbytes / t / 1e9 if t > 0 else None


def run_e2e(L, w: synth.Workload, inputs, args, dev, world):
    """Same metric through the public Python API with pinned host buffers: each step
    copies its input host->device, runs the call and copies the result back."""
    host_in = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in inputs.items()}
    for k in inputs:
        host_in[k].copy_(inputs[k])
    host_out = torch.empty(out_shape(w), dtype=torch.float32, pin_memory=True)
    steps = max(1, min(args.steps, args.e2e_steps))

    def one():
        if w.op == "log_softmax":
            L.log_softmax(host_in["x"], out=host_out)
        elif w.op == "softmax":
            L.softmax(host_in["x"], out=host_out)
        elif w.op == "lse_dim0":
            L.logsumexp(host_in["x"], dim=0, out=host_out)
        elif w.op == "log_softmax_dim0":
            L.log_softmax(host_in["x"], out=host_out, dim=0)
        elif w.op == "conv_gn_act_lse":
            L.conv_gn_act_lse_forward(*(host_in[k] for k in ("x", "w", "bias", "gamma", "beta")), w.params["G"],
                                      w.params["eps"], out=host_out)
        else:
            fn = {"gn_act_lse": L.gn_act_lse_forward, "group_norm": L.group_norm_forward,
                  "gn_act_residual": L.gn_act_residual_forward}[w.op]
            fn(host_in["y"], host_in["gamma"], host_in["beta"], w.params["G"], w.params["eps"],
               out=host_out)

    one()
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    torch.cuda.synchronize(dev)
    dt = time.perf_counter() - t0
    barrier(world)
    dt = max_over_ranks(dt, world, dev)
    nbytes = algorithmic_bytes(w)
    total = sum_over_ranks(float(nbytes * steps), world, dev)
    h2d = sum(t.numel() * 4 for t in host_in.values())
    d2h = host_out.numel() * 4
    value = round(total / dt / 1e9, 3)
    out = {"value": value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": steps,
           "note": "pinned host buffers; every step copies its input in and its result out "
                   "(log_softmax: chunked pipeline overlapping both copies with the call)"}
    link = host_link(host_in, dev)
    if link is not None:
        ceil = e2e_ceiling(nbytes, h2d, d2h, link)
        out["host_link"] = link
        if ceil:
            out["link_ceiling"] = round(ceil, 1)
            out["frac_of_link"] = round(value / world / ceil, 4)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--shape", default=None,
                    help="comma-separated shape: the workload's recipe at another size "
                         "(smaller cases for profiling; not a bench line)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    w = synth.WORKLOADS[args.workload]
    if args.shape:
        shape = tuple(int(v) for v in args.shape.split(","))
        w = synth.Workload(w.name + "@" + "x".join(map(str, shape)), w.op, shape, w.recipe, w.params)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
