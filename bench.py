"""Benchmark of the logsumexp hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-e2e] [--no-cpu-baseline] [--no-configs]

One step is one call of the library on one batch of the workload (default
log_softmax over the last axis of fp32 x[4096, 393216]: rows a2 + a3 of the
path, one kernel launch).  Prints one JSON line (rank 0).  Under torchrun each
rank runs the whole workload on its own GPU (independent batches, weak
scaling) with no data-path collective; the timed region is bracketed by a
barrier and a device synchronize, and the slowest rank's time is reported.

On one GPU, for the default workload, the line also carries `configs`: every other workload of the path
(the logsumexp over dim 0 and log_softmax cases, the GroupNorm chain, and the
operations beside them) measured in the same run after the default one, each
with its time per call and its fraction of the HBM (or tf32 tensor) peak.

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
        # the method's bytes: x once, the weights, bias, gamma and beta, out (the
        # intermediate y is this design's choice, not the method's; see design_bytes)
        N, Cin, H, W = w.shape
        Cout = w.params["Cout"]
        ohw = (H - 2) * (W - 2)
        return 4 * (w.numel + N * ohw + Cout * (Cin * 9 + 3))
    raise KeyError(w.op)


def design_bytes(w: synth.Workload) -> int:
    """Bytes this design moves per step where it differs from the algorithmic bytes:
    the conv-fed chain writes y and reads it back once (L2 serves part of the re-read)."""
    if w.op == "conv_gn_act_lse":
        N, Cin, H, W = w.shape
        return algorithmic_bytes(w) + 4 * 2 * N * w.params["Cout"] * (H - 2) * (W - 2)
    return algorithmic_bytes(w)


def conv_flops(w: synth.Workload) -> int:
    """Multiply-adds of the 3 x 3 convolution counted as 2 flops each (the method's own
    count; the 3xTF32 split executes three products per multiply-add)."""
    N, Cin, H, W = w.shape
    return 2 * N * w.params["Cout"] * (H - 2) * (W - 2) * Cin * 9


GN_ELEMENTWISE = ("group_norm", "gn_act_residual")

# Kernels each step launches (the dominant kernel first).
LAUNCHES = {
    "lse_dim0": ["lse_strided_kernel"],
    "log_softmax": ["row_tmem_kernel"],
    "gn_act_lse": ["gn_fused_kernel"],
    "softmax": ["row_tmem_kernel"],
    "log_softmax_dim0": ["lse_strided_kernel"],
    "group_norm": ["row_tmem_kernel"],
    "gn_act_residual": ["row_tmem_kernel"],
    "conv_gn_act_lse": ["conv2d_ws_kernel", "gn_fused_kernel"],
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
        return 4 * (x.numel() + N * (H - 2) * (W - 2))
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

def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except Exception:
        return None


def hbm_peak():
    d = _peaks()
    try:
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


FALLBACK_BF16_TFLOPS = 1900.0
# Nominal dense tensor rates of GB300 (PFLOP/s): tf32 1.1 against bf16 2.25.
TF32_OVER_BF16 = 1.1 / 2.25


def tf32_peak():
    """The tf32 tensor peak: the measured bf16 burst times the nominal tf32 / bf16 ratio."""
    d = _peaks()
    try:
        return float(d["bf16_tflops"]) * TF32_OVER_BF16, "measured bf16 burst x 1.1/2.25"
    except Exception:
        return FALLBACK_BF16_TFLOPS * TF32_OVER_BF16, "fallback 1900 TFLOP/s bf16 x 1.1/2.25"


# Special-function (MUFU) results per clock per SM on GB300, measured with a
# throughput kernel of independent chains: ex2.approx 31.7, rcp.approx 15.9 (the
# base-2 exponential runs at twice the reciprocal's rate).  The GroupNorm chain's apply
# step issues per element of y two exponentials (tanh's and the channel lse's) and one
# reciprocal (tanh's): 2/32 + 1/16 = 1/8 SM clock per element on the special-function unit.
SFU_EX2_PER_CLK_PER_SM = 32
SFU_RCP_PER_CLK_PER_SM = 16
GN_CHAIN_SFU = {"ex2": 2, "rcp": 1}


def gn_chain_sfu_clocks_per_element() -> float:
    return GN_CHAIN_SFU["ex2"] / SFU_EX2_PER_CLK_PER_SM + GN_CHAIN_SFU["rcp"] / SFU_RCP_PER_CLK_PER_SM


# The sources that determine each dominant kernel's code (with the shared headers).
KERNEL_SOURCES = {
    "row_tmem_kernel": ["row_tmem.cuh", "tmem.cuh", "log_softmax.cu", "gn_rows.cu", "gn_common.cuh"],
    "lse_strided_kernel": ["lse_strided.cu"],
    "gn_fused_kernel": ["gn_act_lse.cu", "gn_common.cuh"],
    "gn_tma_kernel": ["gn_tma.cu", "gn_common.cuh"],
    "conv2d_ws_kernel": ["conv.cu", "conv_tile.cuh", "gn_common.cuh"],
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


CLOCK_REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                     0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


def summarize_clocks(samples, windows):
    """Median SM clock, highest max clock, the throttle reasons seen and the sample
    count of the samples inside any of `windows` ((t0, t1) wall-clock pairs); all
    samples when none falls inside.  A sample is (wall time, sm MHz, max MHz, reasons,
    power W), with None for a field that could not be read."""
    inside = [p for p in samples if any(t0 <= p[0] <= t1 for (t0, t1) in windows)]
    window = "timed region"
    if not inside:
        inside = list(samples)
        window = "whole run (no sample fell inside the timed region)"
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                "note": "no clock source available"}
    sm = [p[1] for p in inside if p[1] is not None]
    smax = [p[2] for p in inside if p[2] is not None]
    power = [p[4] for p in inside if p[4] is not None]
    reasons = sorted({r for p in inside for r in p[3]})
    out = {"sm_mhz": statistics.median(sm) if sm else None,
           "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
           "samples": len(inside), "window": window}
    if sm:
        out["sm_mhz_min"] = min(sm)
    if power:
        out["power_w_max"] = round(max(power), 1)
    return out


class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (no setting is changed)."""
    CLOCK_SM = 1

    def __init__(self, device_index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(self.h)) != 0:
            raise OSError("nvmlDeviceGetHandleByUUID failed")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        v = ctypes.c_uint()
        self.max_mhz = (float(v.value) if self.lib.nvmlDeviceGetMaxClockInfo(self.h, self.CLOCK_SM,
                                                                            ctypes.byref(v)) == 0 else None)
        if self.read()[0] is None:
            raise OSError("nvmlDeviceGetClockInfo failed")

    def read(self):
        ct = self.ct
        c, r, pw = ct.c_uint(), ct.c_ulonglong(), ct.c_uint()
        mhz = float(c.value) if self.lib.nvmlDeviceGetClockInfo(self.h, self.CLOCK_SM, ct.byref(c)) == 0 else None
        reasons = ([n for bit, n in CLOCK_REASON_BITS.items() if r.value & bit]
                   if self.reasons_fn(self.h, ct.byref(r)) == 0 else [])
        watts = pw.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.h, ct.byref(pw)) == 0 else None
        return mhz, self.max_mhz, reasons, watts


class ClockSampler:
    """SM clock, throttle reasons and power sampled during the run: in process through
    NVML every 2 ms (so that even a timed region of a few tens of milliseconds holds
    samples), else from `nvidia-smi -lms 100`."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period: float = 0.002):
        self.samples = []  # (wall time, sm MHz, max MHz, reasons, power W)
        self.period = period
        self.proc = None
        self.thread = None
        self.stop_flag = threading.Event()
        self.active = threading.Event()
        self.active.set()
        self.source = None
        try:
            self.nvml = _Nvml(device_index)
            self.source = "nvml"
        except Exception:
            self.nvml = None
        self.device_index = device_index

    def start(self):
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._poll_nvml, daemon=True)
            self.thread.start()
            return self
        uuid = None
        try:
            uuid = str(torch.cuda.get_device_properties(self.device_index).uuid)
        except Exception:
            pass
        target = (["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid] if uuid else
                  ["-i", str(self.device_index)])
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *target, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except Exception:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read_smi, daemon=True)
        self.thread.start()
        return self

    def pause(self):
        """Stops polling (between timed regions) until resume()."""
        self.active.clear()

    def resume(self):
        self.active.set()

    def _poll_nvml(self):
        while not self.stop_flag.is_set():
            if not self.active.wait(timeout=0.05):
                continue
            try:
                mhz, mx, reasons, watts = self.nvml.read()
                self.samples.append((time.time(), mhz, mx, reasons, watts))
            except Exception:
                return
            time.sleep(self.period)

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        for line in self.proc.stdout:
            p = [q.strip() for q in line.strip().split(",")]
            if len(p) >= 8:
                reasons = [n for n, v in zip(names, p[4:8]) if v == "Active"]
                self.samples.append((time.time(), num(p[0]), num(p[1]), reasons, num(p[2])))

    def stop(self):
        self.stop_flag.set()
        self.active.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        out = summarize_clocks(list(self.samples), [(t0, t1)])
        out["source"] = self.source
        return out


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


def time_steps(step, steps, flush, stream, dev, world=1):
    """Times `steps` calls of `step` on `stream` with CUDA events, each preceded by an
    L2 flush (a write of `flush`) when `flush` is given; bracketed by a barrier and a
    device synchronize.  Returns (per-step ms, whole-region ms, wall t0, wall t1)."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    t_all0.record(stream)
    for i in range(steps):
        if flush is not None:
            flush.fill_(1.0)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    wall1 = time.time()
    return [a.elapsed_time(b) for a, b in ev], t_all0.elapsed_time(t_all1), wall0, wall1


def l2_flush_buffer(inputs, dev):
    """A buffer of twice the L2 size to write between steps when the inputs would fit
    in L2 (None when they are larger than twice L2 and need no flush)."""
    in_bytes = sum(t.numel() * 4 for t in inputs.values())
    if in_bytes < 2 * L2_BYTES:
        return torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    return None


def hbm_roofline(nbytes, launch_ms, dominant, workload, note):
    peak, peak_kind = hbm_peak()
    achieved = nbytes / (launch_ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": ncu_traffic(dominant, workload),
            "kernel": dominant, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6800 GB/s",
            "note": note}


# The workloads measured beside the default line, in the same run (SURVEY rows in
# brackets): the five configurations of the path, then the rows next to it.
CONFIG_ROLES = (
    ("lse_dim0_4x10x32", "C1 (a1)", "latency"),
    ("log_softmax_256x4096", "C2 (a2+a3)", "latency"),
    ("lse_dim0_32x8192x4096", "C3 (a1)", "hbm"),
    ("log_softmax_4096x393216", "C4 (a2+a3)", "default"),
    ("gn_act_lse_128x64x126x126", "C5 (a4+a5)", "hbm"),
    ("softmax_4096x393216", "NEXT-2", "hbm"),
    ("group_norm_128x64x126x126", "NEXT-3", "hbm"),
    ("gn_act_residual_128x64x126x126", "NEXT-3", "hbm"),
    ("log_softmax_dim0_32x8192x4096", "NEXT-4", "hbm"),
    ("conv_gn_act_lse_128x8x128x128", "NEXT-1", "tensor"),
)


def measure_config(L, name: str, role: str, kind: str, dev, stream, steps: int, warmup: int, sampler):
    """One workload of CONFIG_ROLES measured on this GPU: time per call and, for the
    bandwidth-bound ones, GB/s on algorithmic bytes and the fraction of the HBM peak;
    latency-bound ones report microseconds per call after an L2 flush and warm."""
    w = synth.WORKLOADS[name]
    inputs = synth.make_inputs(w, device=dev)
    out = torch.empty(out_shape(w), dtype=torch.float32, device=dev)
    step = make_step(L, w, inputs, out, stream)
    if sampler is not None:
        sampler.resume()
    nbytes = algorithmic_bytes(w)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if kind == "latency" \
        else l2_flush_buffer(inputs, dev)
    for _ in range(warmup):
        if flush is not None:
            flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)
    per, region, t0, t1 = time_steps(step, steps, flush, stream, dev)
    res = {"role": role, "kernels": LAUNCHES[w.op], "steps": steps, "shape": list(w.shape),
           "algorithmic_bytes": nbytes}
    windows = [(t0, t1)]
    if kind == "latency":
        med = statistics.median(per)
        res.update({"us_per_call_l2_flushed": round(1e3 * med, 2),
                    "gbs_l2_flushed": round(nbytes / (med / 1e3) / 1e9, 2)})
        # warm: the calls captured back to back in one CUDA graph and replayed, so that
        # neither the host's enqueue time nor an L2 flush sits between them
        gstep = make_step(L, w, inputs, out, None)
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            gstep()  # outside the capture: the library's first-call set-up
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(steps):
                gstep()
        graph.replay()
        torch.cuda.synchronize(dev)
        per_w, _, t0w, t1w = time_steps(graph.replay, 3, None, stream, dev)
        us_w = 1e3 * min(per_w) / steps
        res.update({"us_per_call_warm": round(us_w, 3),
                    "gbs_warm": round(nbytes / (us_w / 1e6) / 1e9, 2),
                    "note": "flushed: median CUDA-event time of one call after a 258 MB write; warm: "
                            f"{steps} calls back to back in one CUDA graph, best of 3 replays / {steps}"})
        windows.append((t0w, t1w))
        del graph
    else:
        ms = statistics.mean(per) if flush is not None else region / steps
        peak, _ = hbm_peak()
        gbs = nbytes / (ms / 1e3) / 1e9
        res.update({"ms_per_step": round(ms, 5), "gbs": round(gbs, 2), "frac_of_hbm_peak": round(gbs / peak, 4),
                    "l2": "inputs larger than L2; no flush" if flush is None else
                    "L2 flushed between steps; steps timed alone"})
        if w.op == "gn_act_lse":
            res["sfu"] = {"ops_per_element": dict(GN_CHAIN_SFU)}
        if kind == "tensor":
            fl = conv_flops(w)
            tpk, src = tf32_peak()
            res.update({"tflops_method": round(fl / (ms / 1e3) / 1e12, 2), "tf32_peak_tflops": round(tpk, 1),
                        "frac_of_tf32_peak": round(fl / (ms / 1e3) / 1e12 / tpk, 4), "tf32_peak_source": src,
                        "design_bytes": design_bytes(w),
                        "note": "bytes are the method's (x, parameters, out); the design also writes the "
                                "conv output y and reads it back (design_bytes)"})
            # the convolution alone, into a y buffer
            N, Cin, H, W = w.shape
            Cout = w.params["Cout"]
            y = torch.empty((N, Cout, H - 2, W - 2), dtype=torch.float32, device=dev)
            xc, wc, bc = inputs["x"], inputs["w"], inputs["bias"]
            conv = lambda: L.conv2d_3x3(xc, wc, bc, y, N, Cin, H, W, Cout, stream=stream)  # noqa: E731
            for _ in range(warmup):
                if flush is not None:
                    flush.fill_(1.0)
                conv()
            per_c, _, t0c, t1c = time_steps(conv, steps, flush, stream, dev)
            ms_c = statistics.mean(per_c)
            res["conv2d_3x3"] = {"kernel": "conv2d_ws_kernel", "ms_per_call": round(ms_c, 5),
                                 "tflops_method": round(fl / (ms_c / 1e3) / 1e12, 2),
                                 "frac_of_tf32_peak": round(fl / (ms_c / 1e3) / 1e12 / tpk, 4)}
            windows.append((t0c, t1c))
            del y
    if sampler is not None:
        sampler.pause()
        c = summarize_clocks(list(sampler.samples), windows)
        res["clocks"] = {k: c.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons", "samples", "window")}
        if w.op == "gn_act_lse" and c.get("sm_mhz"):
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            floor_s = gn_chain_sfu_clocks_per_element() * w.numel / sms / (c["sm_mhz"] * 1e6)
            res["sfu"].update({"floor_ms": round(1e3 * floor_s, 5),
                               "frac": round(floor_s / (res["ms_per_step"] / 1e3), 4),
                               "note": f"ex2 at {SFU_EX2_PER_CLK_PER_SM} and rcp at {SFU_RCP_PER_CLK_PER_SM} "
                                       f"results per clock per SM, {sms} SMs, median SM clock of the window"})
    del inputs, out, flush
    torch.cuda.empty_cache()
    return res


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
    flush = l2_flush_buffer(inputs, dev)
    l2_note = ("inputs larger than L2 (129 MB); no flush" if flush is None else
               "L2 flushed (256 MB write) between steps; steps timed alone")

    for _ in range(args.warmup):
        if flush is not None:
            flush.fill_(1.0)
        step()
    torch.cuda.synchronize(dev)
    if L.lse_device_status() != 0:
        raise SystemExit("device status reported a bounded-wait timeout during warm-up")

    sampler = ClockSampler(local).start() if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    per_step_ms, region_ms, wall0, wall1 = time_steps(step, args.steps, flush, stream, dev, world)
    if sampler:
        time.sleep(0.01)
        sampler.pause()  # no polling during the end-to-end and CPU measurements
    status = L.lse_device_status()

    kernel_ms = sum(per_step_ms)
    # With inputs larger than L2 nothing runs between steps: time the whole region.
    # Otherwise an L2 flush runs between steps; time the steps alone.
    local_ms = kernel_ms if flush is not None else region_ms
    slow_ms = max_over_ranks(local_ms, world, dev)
    total_bytes = sum_over_ranks(float(nbytes * args.steps), world, dev)
    value = total_bytes / (slow_ms / 1e3) / 1e9

    # roofline of the dominant kernel (one launch of it per step)
    launch_ms = statistics.mean(per_step_ms)
    dominant = LAUNCHES[w.op][0]
    achieved_note = ("one launch per step" if len(LAUNCHES[w.op]) == 1 else
                     f"{len(LAUNCHES[w.op])} launches per step ({', '.join(LAUNCHES[w.op])}); achieved over the whole step")
    if w.op == "conv_gn_act_lse":
        tpk, src = tf32_peak()
        ach = conv_flops(w) / (launch_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "achieved": round(ach, 2), "peak": round(tpk, 1), "unit": "TFLOP/s",
                    "frac": round(ach / tpk, 4), "traffic": ncu_traffic(dominant, w.name), "kernel": dominant,
                    "peak_source": src, "note": achieved_note + "; flops are the convolution's multiply-adds x 2",
                    "hbm": hbm_roofline(nbytes, launch_ms, dominant, w.name, "the method's bytes (x, out)")}
    else:
        roofline = hbm_roofline(nbytes, launch_ms, dominant, w.name, achieved_note)

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

    # the other workloads of the path, measured in this same run (one GPU, default workload)
    configs = None
    if rank == 0 and world == 1 and not args.no_configs and w.name == DEFAULT_WORKLOAD:
        del inputs, out, flush, step
        torch.cuda.empty_cache()
        configs = {}
        for name, role, kind in CONFIG_ROLES:
            if kind == "default":
                configs[name] = {"role": role, "see": "this line's value" if name == w.name else
                                 "python bench.py (default workload)"}
                if name != w.name:
                    kind = "hbm"
                else:
                    continue
            try:
                configs[name] = measure_config(L, name, role, kind, dev, stream, args.config_steps, 3, sampler)
            except Exception as e:  # one workload's failure does not hide the others
                configs[name] = {"role": role, "error": repr(e)[:300]}
        status = status or L.lse_device_status()
    if sampler:
        time.sleep(0.05)
        sampler.stop()

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
                   "l2": l2_note,
                   "parallelism": f"replicas x{world} (independent batches)"},
        "roofline": roofline,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "gpu_launches": len(LAUNCHES[w.op]) * args.steps,
        "device_status": L.lse_status_string(status),
        "configs": configs,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def host_link(host_in, dev, host_out=None, max_bytes=1 << 30, min_bytes=64 << 20):
    """Copy-engine bandwidth of this process's host link on its own pinned input buffer
    (after the end-to-end timing, which no longer needs it): host to device from its
    first half, device to host into its second half, and both at once (two streams),
    GB/s; and device to host into the output buffer the end-to-end steps wrote
    (`d2h_out_gbs`: pinned buffers can differ in how fast the copy engines reach them).
    None when the buffer is too small to time bandwidth rather than latency."""
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
    res = {"h2d_gbs": round(h2d, 1), "d2h_gbs": round(d2h, 1), "both_gbs": round(bi, 1), "bytes_each": n * 4}
    if host_out is not None and host_out.numel() >= n:
        dout = host_out.view(-1)[:n]
        dout.copy_(a, non_blocking=True)
        res["d2h_out_gbs"] = round(n * 4 / min(timed(lambda: dout.copy_(a, non_blocking=True)) for _ in range(2)) / 1e9, 1)
    return res


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
    link = host_link(host_in, dev, host_out)
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
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads measured after the default line")
    ap.add_argument("--config-steps", type=int, default=20)
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
