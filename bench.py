"""Throughput of the tcgen05 GEMM hot path on GB300, one JSON line per run.

A step is one pass of the hot path over one batch of resident synthetic input
at M = N = K = 8192:
  * bf16 x bf16 -> fp32 accumulate -> bf16 D (alpha = 1, beta = 0)
  * E4M3 x E4M3 with per-tensor fp32 dequantisation scales and a bf16 bias
    -> bf16 D
  * 2:4 structured-sparse bf16 A: compress of the logical A (keep the two
    largest of every four along K, ordered metadata) and the sparse GEMM on
    the compressed A and its canonical metadata
value = 2*M*N*K of the step's two dense GEMMs (the bf16 and FP8 GEMMs the
metric names) / step time, in TFLOP/s.  The sparse GEMM runs inside the step
but its (logical) FLOPs are reported only in its own part.

Besides the step, the default run times every configured workload as a part
outside `value` (512^3 with C, 4096^3 fp16 and bf16, the three LLM shapes, the
skinny 16 x 28672 x 8192 decode shape against HBM bandwidth, E4M3 x E5M2) and,
in the CPU-baseline leg, checks the timed step's outputs against the CPU
oracle on whole output rows (exit status 1 if any exceeds the bound).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tcm|reference]

With torchrun (N > 1) every rank runs an independent replica on its own GPU
(weak scaling); the slowest rank's time counts.  ``--impl reference`` times
the CPU oracle instead (rank 0 only), on bounded samples of the same work.
``--shapes`` times a longer list of workloads (block-scaled, fused, FP4), one
JSON line each, instead of the step.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
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

import synth_inputs as si  # noqa: E402

SIZE = 8192
FLOP_PER_GEMM = 2.0 * SIZE ** 3
DENSE_GEMMS_PER_STEP = 2  # bf16 and E4M3: the FLOPs `value` counts
METRIC = "GEMM TFLOP/s (2MNK/t) at 8192³ bf16 and FP8; % of GB300 dense tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 / bf16 tensor rates (GB300)
FP8_OVER_BF16 = 4.5 / 2.25  # nominal dense ratio
# dense bf16 tcgen05 rate of one SM per clock (the ncu tensor-pipe utilisation of the
# bf16 8192^3 kernel, 88.8 % of elapsed cycles at 1.647 GHz for 1822 TFLOP/s, gives 8197)
BF16_FLOP_PER_CLK_PER_SM = 8192
L2_BYTES = 129 * 10 ** 6
SUSTAINED_AFTER_S = 1.0  # timed regions at least this long are compared with the sustained peak
# the bf16 kernel and the host code that plans its launch (tile order, split): the recorded
# DRAM traffic holds only while none of them changed
KERNEL_SOURCES = ["tensor_core_matrix_gb300/csrc/tcm_gemm_kernel.cuh", "tensor_core_matrix_gb300/csrc/tcm_kernel_common.cuh",
                  "tensor_core_matrix_gb300/csrc/tcm_ptx.cuh", "tensor_core_matrix_gb300/csrc/tcm_gemm_pair.cu",
                  "tensor_core_matrix_gb300/csrc/tcm_api.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_kernel_bf16_8192cubed.json")
SLEEP_CYCLES = 400_000  # ~0.2 ms: lets the host enqueue a launch before its start event


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["tcm", "reference"], default="tcm")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parts", action="store_true", help="skip the per-config parts")
    ap.add_argument("--no-workspace", action="store_true",
                    help="dense GEMMs of the step through tcm_gemm_ex without a workspace (no split tail): "
                         "the same kernels in a non-cooperative launch, for profilers that cannot replay "
                         "cooperative launches")
    ap.add_argument("--part-iters", type=int, default=20)
    ap.add_argument("--shapes", action="store_true",
                    help="instead of the step, time every configured workload shape (one JSON line each)")
    ap.add_argument("--shape-iters", type=int, default=20)
    ap.add_argument("--only", default="", help="with --shapes: only workloads whose name contains this text")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def bf16_peak_for(region_s, peaks_used):
    """(peak TFLOP/s, label): the burst figure for a timed region shorter than a second,
    the figure measured over a seconds-long loop otherwise."""
    p, src = peaks_used
    if region_s >= SUSTAINED_AFTER_S:
        return (float(p.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])),
                f"{src} bf16_tflops_sustained (timed region {region_s:.3f} s, seconds-long)")
    return (float(p.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
            f"{src} bf16_tflops burst (timed region {region_s:.3f} s, under {SUSTAINED_AFTER_S:g} s)")


def kernel_source_sha():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of the bf16 8192^3 kernel from the committed ncu record, if the
    kernel sources are still the ones it was captured from (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha") != kernel_source_sha():
        return None
    try:
        return float(rec["dram_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
        return None


def smi_gpu_id(dev_index):
    """The NVML / nvidia-smi name of CUDA device `dev_index`: its UUID (they number the
    machine's GPUs themselves and ignore CUDA_VISIBLE_DEVICES, so an index may name another GPU)."""
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    return vis[dev_index].strip() if dev_index < len(vis) else str(dev_index)


# NVML clock-event reason bits (nvmlClocksEventReason*), the ones a timing must report
REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU, polled every `period` seconds
    while a timed region runs.  Read-only NVML queries through ctypes (libnvidia-ml ships
    with the driver); falls back to `nvidia-smi -lms` if NVML cannot be opened.  Each
    sample carries a host timestamp so that summaries can keep only the samples taken
    inside given windows (the timed regions)."""

    def __init__(self, index, period=0.001):
        self.index = index
        self.period = period
        self.samples = []  # (t, sm_mhz, max_mhz, power_w, reasons)
        self.source = None
        self.error = ""
        self._stop = threading.Event()
        self._thread = None
        self._proc = None

    def _open_nvml(self):
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(smi_gpu_id(self.index).encode()), ctypes.byref(h)) != 0:
            raise OSError("nvmlDeviceGetHandleByUUID failed")
        reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))  # NVML_CLOCK_SM = 1
        return nv, h, reasons, float(mx.value)

    def _poll_nvml(self, nv, h, reasons, max_mhz):
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            t = time.perf_counter()
            ok = nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0
            nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
            reasons(h, ctypes.byref(rs))
            if ok:
                self.samples.append((t, float(clk.value), max_mhz, pw.value / 1000.0, int(rs.value)))
            time.sleep(self.period)

    def __enter__(self):
        try:
            nv, h, reasons, max_mhz = self._open_nvml()
            self.source = f"nvml every {self.period * 1e3:g} ms"
            self._thread = threading.Thread(target=self._poll_nvml, args=(nv, h, reasons, max_mhz), daemon=True)
            self._thread.start()
            while not self.samples and self._thread.is_alive():
                time.sleep(0.001)
            return self
        except (OSError, AttributeError) as e:
            self.error = f"nvml: {e}"
        try:
            self._path = os.path.join("/tmp", f"tcm_clocks_{os.getpid()}.csv")
            self._out = open(self._path, "w")
            q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                 "clocks_event_reasons.sw_power_cap")
            self._proc = subprocess.Popen(["nvidia-smi", "-i", smi_gpu_id(self.index), f"--query-gpu={q}",
                                           "--format=csv,noheader,nounits", "-lms", "20"],
                                          stdout=self._out, stderr=subprocess.DEVNULL)
            self.source = "nvidia-smi -lms 20"
            self._t_start = time.perf_counter()
            deadline = time.time() + 15.0
            while time.time() < deadline and self._proc.poll() is None and os.path.getsize(self._path) == 0:
                time.sleep(0.05)
        except (OSError, FileNotFoundError) as e:
            self.error += f"; nvidia-smi: {e}"
            self._proc = None
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=5)
        if self._proc is not None:
            t_end = time.perf_counter()
            self._proc.terminate()
            try:
                self._proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
            self._out.close()
            rows = []
            for line in open(self._path):
                f = [x.strip() for x in line.split(",")]
                try:
                    bits = sum(b for b, v in zip((0x8, 0x40, 0x20, 0x4), f[3:7]) if v.lower() == "active")
                    rows.append((float(f[0]), float(f[1]), float(f[2]), bits))
                except (ValueError, IndexError):
                    continue
            os.unlink(self._path)
            # nvidia-smi rows carry no timestamps: spread them evenly over the sampling period
            n = len(rows)
            for i, r in enumerate(rows):
                t = self._t_start + (t_end - self._t_start) * (i + 0.5) / max(n, 1)
                self.samples.append((t, r[0], r[1], r[2], r[3]))

    def summary(self, windows=None):
        """Median SM clock etc. over the samples inside `windows` ([(t0, t1), ...]; all if None)."""
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0,
                    "source": self.source, "error": self.error}
        inside = [s for s in self.samples if windows is None or any(a <= s[0] <= b for a, b in windows)]
        use = inside or self.samples
        reasons = sorted({name for s in use for bit, name in REASON_BITS.items() if s[4] & bit})
        return {"sm_mhz": statistics.median(s[1] for s in use), "sm_mhz_min": min(s[1] for s in use),
                "sm_max_mhz": max(s[2] for s in self.samples), "reasons": reasons,
                "samples": len(self.samples), "samples_under_load": len(inside),
                "power_w_max": max(s[3] for s in use), "source": self.source}


def gpu_local_cpus(device_index):
    """CPUs the kernel lists as local to the GPU (sysfs), or None if unknown."""
    try:
        props = torch.cuda.get_device_properties(device_index)
        bdf = f"{props.pci_domain_id:04x}:{props.pci_bus_id:02x}:{props.pci_device_id:02x}.0"
        text = open(f"/sys/bus/pci/devices/{bdf}/local_cpulist").read().strip()
        cpus = set()
        for part in text.split(","):
            lo, _, hi = part.partition("-")
            cpus.update(range(int(lo), int(hi or lo) + 1))
        cpus &= os.sched_getaffinity(0)
        return cpus or None
    except (AttributeError, OSError, ValueError):
        return None


def slowest_rank(pg, values, device):
    """Element-wise maximum of `values` over all ranks (the slowest rank's times decide)."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if pg is not None:
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(x) for x in t]


def whole_job_rate(world, units_per_rank, seconds):
    """Throughput of the whole job: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank / seconds


def local_rank_index(device):
    return device.index if device.index is not None else torch.cuda.current_device()


def step_host_inputs():
    dense = si.llm_case(SIZE, SIZE, SIZE, seed=2)  # bf16 A ~ N(0,1), B ~ N(0, 0.02)
    f8 = si.fp8_case(SIZE, SIZE, SIZE, b_fmt="e4m3", seed=3)
    sp = si.sparse_case(SIZE, SIZE, SIZE, seed=4)
    return {
        "A": dense["A"], "B": dense["B"],
        "A8": f8["A"], "B8": f8["B"], "bias": f8["bias"],
        "sa": torch.tensor([f8["sa"]], dtype=torch.float32), "sb": torch.tensor([f8["sb"]], dtype=torch.float32),
        "Asp": sp["A_logical"], "Bsp": sp["B"],
    }


def make_inputs(device, workspace=True):
    """Resident device inputs of one step plus their pinned host copies (for the end-to-end leg);
    workspace=False: the dense GEMMs run without one (dev["ws"] is None)."""
    host = step_host_inputs()
    pinned = {k: v.pin_memory() for k, v in host.items()}
    dev = {k: v.to(device) for k, v in host.items()}
    for k in ("D", "D8", "Dsp"):
        dev[k] = torch.empty((SIZE, SIZE), dtype=torch.bfloat16, device=device)
    dev["Ac"] = torch.empty((SIZE, SIZE // 2), dtype=torch.bfloat16, device=device)
    dev["meta"] = torch.empty((SIZE, SIZE // 32), dtype=torch.int32, device=device)
    # workspace of the dense GEMMs (tail tiles split over K); one buffer serves both, in turn
    import tensor_core_matrix_gb300 as tcm
    ws = max(tcm.tcm_gemm_workspace_bytes(SIZE, SIZE, SIZE, torch.bfloat16),
             tcm.tcm_gemm_workspace_bytes(SIZE, SIZE, SIZE, torch.float8_e4m3fn))
    dev["ws"] = torch.empty(max(ws, 16), dtype=torch.uint8, device=device) if workspace else None
    return host, pinned, dev


def run_step(tcm, dev, stream, events=None, probes=None):
    """One pass of the hot path; events[0..4] bracket the four launches on `stream`;
    probes: per-GEMM clock-probe counters (tcm_set_clock_probe) or None."""
    def mark(i):
        if events:
            events[i].record(stream)

    def probe(key):
        if probes is not None:
            tcm.tcm_set_clock_probe(probes.get(key))
    mark(0)
    probe("bf16_dense")
    tcm.tcm_gemm_ex(dev["A"], dev["B"], dev["D"], workspace=dev["ws"], stream=stream)
    mark(1)
    probe("e4m3_scaled_bias")
    tcm.tcm_gemm_ex(dev["A8"], dev["B8"], dev["D8"], a_scale=dev["sa"], b_scale=dev["sb"], bias=dev["bias"],
                    workspace=dev["ws"], stream=stream)
    mark(2)
    probe(None)
    tcm.tcm_sp_compress(dev["Asp"], dev["Ac"], dev["meta"], stream=stream)
    mark(3)
    probe("sp24_gemm_bf16")
    tcm.tcm_gemm_sp(dev["Ac"], dev["meta"], dev["Bsp"], dev["Dsp"], stream=stream)
    mark(4)
    probe(None)


def probe_mhz(counters):
    """SM clock (MHz) of the launches a clock probe saw: cycles / global-timer ns of their first CTA."""
    c = counters.cpu().tolist()
    return 1e3 * c[0] / c[1] if c[1] > 0 else None


KERNELS_PER_STEP = 4
# compress: read A, write A_comp and the canonical metadata
COMPRESS_BYTES = SIZE * SIZE * 2 + SIZE * (SIZE // 2) * 2 + SIZE * (SIZE // 32) * 4


class OracleSample:
    """The CPU oracle on whole output rows of the step's three GEMMs (and the 2:4 compress of
    those rows); keeps its results so that the GPU's outputs of the same rows can be checked."""

    def __init__(self, host):
        import oracle
        self.oracle = oracle
        oracle.build()
        self.a, self.b = si.codes(host["A"]), si.codes(host["B"])
        self.a8, self.b8, self.bias = si.codes(host["A8"]), si.codes(host["B8"]), si.codes(host["bias"])
        self.sa, self.sb = float(host["sa"][0]), float(host["sb"][0])
        self.asp, self.bsp = si.codes(host["Asp"]), si.codes(host["Bsp"])
        self.last = None

    def rows(self, r):
        """Rows 0 .. r-1 of every GEMM of the step; returns (dense FLOPs, all FLOPs) computed."""
        import numpy as np
        o = self.oracle
        rows = np.repeat(np.arange(r, dtype=np.int64), SIZE)
        cols = np.tile(np.arange(SIZE, dtype=np.int64), r)
        out = {"D": o.gemm(self.a, self.b, "bf16", "bf16", rows=rows, cols=cols),
               "D8": o.gemm(self.a8, self.b8, "e4m3", "e4m3", bias=self.bias, sa=self.sa, sb=self.sb,
                            rows=rows, cols=cols)}
        ac, meta = o.sp_compress(np.ascontiguousarray(self.asp[:r]), "bf16")
        out["Dsp"] = o.gemm(o.sp_decompress(ac, meta, "bf16"), self.bsp, "bf16", "bf16", rows=rows, cols=cols)
        out["Ac"], out["meta"] = ac, meta
        self.last = (r, out)
        flop = 2.0 * r * SIZE * SIZE
        return DENSE_GEMMS_PER_STEP * flop, 3 * flop

    def calibrate(self, seconds):
        t0 = time.perf_counter()
        self.rows(1)
        per_row = max(time.perf_counter() - t0, 1e-6)
        return max(1, int(seconds / per_row))

    def check(self, gpu):
        """max err / bound of the GPU's rows of each GEMM and bit-equality of the compress;
        `gpu` holds CPU copies of the first r rows of D, D8, Dsp, Ac and meta."""
        import numpy as np
        o = self.oracle
        r, out = self.last
        res = {"rows": r}
        for key, name, scale in (("D", "bf16_dense", 1.0), ("D8", "e4m3_scaled_bias", self.sa * self.sb),
                                 ("Dsp", "sp24_gemm_bf16", 1.0)):
            ref, S = out[key]
            res[name] = o.err_over_bound(si.codes(gpu[key][:r]).reshape(-1), "bf16", ref, S, scale)
        res["sp24_compress_bit_exact"] = bool(
            np.array_equal(si.codes(gpu["Ac"][:r]), out["Ac"]) and
            np.array_equal(si.codes(gpu["meta"][:r]).view(np.uint32), out["meta"]))
        res["ok"] = all(res[k] <= 1.0 for k in ("bf16_dense", "e4m3_scaled_bias", "sp24_gemm_bf16")) and \
            res["sp24_compress_bit_exact"]
        return res


def cpu_baseline_sample(host, seconds, gpu_rows):
    """Time the CPU oracle on about `seconds` of whole output rows of the step's GEMMs and check
    the GPU's outputs of the same rows against it.  Returns (baseline, check)."""
    o = OracleSample(host)
    r = min(o.calibrate(seconds), min(t.shape[0] for t in gpu_rows.values()))
    t0 = time.perf_counter()
    dense_flop, flop = o.rows(r)
    t = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    base = {"value": dense_flop / t / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{r} full output rows (8192 outputs of K=8192 each) of each of the step's three GEMMs "
                      f"(bf16, E4M3 with scales+bias, 2:4-sparse bf16 incl. compress of those rows), "
                      f"{t:.1f} s on {cores} host threads (OpenMP); value counts the two dense GEMMs' FLOPs "
                      f"like the GPU line",
            "extrapolated_full_step_s": t * SIZE / r,
            "extrapolated_note": "extrapolated: sample time x M / rows (per-MAC time x M*N*K of each GEMM)"}
    return base, o.check(gpu_rows)


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    o = OracleSample(step_host_inputs())
    cores = len(os.sched_getaffinity(0))
    r = o.calibrate(90.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        o.rows(r)
    t0 = time.perf_counter()
    flop = 0.0
    for _ in range(args.steps):
        flop += o.rows(r)[0]
    t = time.perf_counter() - t0
    value = flop / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16+e4m3",
        "data": "synthetic", "config": config_block(world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {r} full output rows of each of the three 8192^3 GEMMs "
                                   f"(fp64 CPU oracle, {cores} host threads); value counts the two dense "
                                   f"GEMMs' FLOPs"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ per-config parts

class LaunchTimer:
    """Device time of single launches and of back-to-back runs on one stream.

    single(): before each launch the stream sleeps ~0.2 ms (torch's device-side sleep)
    so that the host has enqueued the launch before its start event is reached: the
    event pair then brackets the kernel alone, not the host-side cost of the call.
    `flush` writes 256 MiB (more than L2) before each launch."""

    def __init__(self, device, stream):
        self.stream = stream
        self.flush_buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
        self.windows = []

    def single(self, launch, iters, flush, sleep=True):
        times = []
        t0 = time.perf_counter()
        for _ in range(iters):
            with torch.cuda.stream(self.stream):
                if flush:
                    self.flush_buf.fill_(1)
                if sleep and hasattr(torch.cuda, "_sleep"):
                    torch.cuda._sleep(SLEEP_CYCLES)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(self.stream)
                launch()
                e1.record(self.stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        self.windows.append((t0, time.perf_counter()))
        return times

    def back_to_back(self, launch, iters):
        t0 = time.perf_counter()
        with torch.cuda.stream(self.stream):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            for _ in range(iters):
                launch()
            e1.record(self.stream)
        e1.synchronize()
        self.windows.append((t0, time.perf_counter()))
        return e0.elapsed_time(e1) / iters


class Workload:
    """One GEMM workload on the device: its launch closure (on `stream`), sizes, algorithmic
    bytes and the tensor-peak multiple of its input format (bf16 = 1)."""

    def __init__(self, name, case, tcm, device, stream):
        self.name = name
        sparse = "A_logical" in case
        A = (case["A_logical"] if sparse else case["A"]).to(device)
        B = case["B"].to(device)
        M = A.shape[0]
        N = B.shape[0]
        fp4 = case.get("nv") or case.get("a_fmt") == "e2m1"          # packed operands: K/2 bytes per row
        K = A.shape[1] * (2 if fp4 else 1)
        out_dtype = torch.float32 if case.get("out_fmt") == "f32" else torch.bfloat16
        if case.get("fused"):
            out_dtype = torch.float8_e4m3fn
        if case.get("i8"):
            out_dtype = torch.int32
        D = torch.empty((M, N), dtype=out_dtype, device=device)
        C = case["C"].to(device) if case.get("C") is not None else None
        kw = dict(C=C, alpha=case.get("alpha", 1.0), beta=case.get("beta", 0.0), stream=stream)
        self.workspace_bytes = 0
        self.peak_mult = 1.0
        if "sa" in case:
            kw.update(a_scale=torch.tensor([case["sa"]], device=device), b_scale=torch.tensor([case["sb"]], device=device))
            if case.get("bias") is not None:
                kw.update(bias=case["bias"].to(device))
        if case.get("b_fmt") == "e2m1" and case.get("a_fmt") != "e2m1":
            kw.update(b_fmt="e2m1")  # W4A8: B holds N x K/2 bytes of packed FP4
        if case.get("i8"):
            # exact INT8 on the bf16 tensor path: 2MNK integer ops against the bf16 rate, the
            # int8 -> bf16 conversion of A and B included
            self.workspace_bytes = tcm.tcm_gemm_i8_workspace_bytes(M, N, K)
            ws = torch.empty(self.workspace_bytes, dtype=torch.uint8, device=device)
            self.launch = lambda: tcm.tcm_gemm_i8(A, B, D, workspace=ws, stream=stream)
        elif sparse:
            self.peak_mult = 2.0  # logical FLOPs against the 2:4 rate
            Ac, meta = tcm.tcm_sp_compress(A)
            if case.get("tc"):
                meta_tc = tcm.tcm_sp_meta_pack(meta, K)
                self.launch = lambda: tcm.tcm_gemm_sp_tc(Ac, meta_tc, B, D, C=C, alpha=kw["alpha"], beta=kw["beta"],
                                                         stream=stream)
            else:
                self.launch = lambda: tcm.tcm_gemm_sp(Ac, meta, B, D, C=C, alpha=kw["alpha"], beta=kw["beta"],
                                                      stream=stream)
        elif case.get("nv"):
            self.peak_mult = FP4_OVER_BF16
            SA = tcm.tcm_nvfp4_pack_scales(case["SA"].to(device), K)
            SB = tcm.tcm_nvfp4_pack_scales(case["SB"].to(device), K)
            self.launch = lambda: tcm.tcm_gemm_nvfp4(A, SA, B, SB, D, alpha=case["alpha"], stream=stream)
        elif "SA" in case:
            # scales packed once into the blocked layout (as a quantiser would emit them)
            self.peak_mult = FP4_OVER_BF16 if fp4 else FP8_OVER_BF16
            SA = tcm.tcm_mx_pack_scales(case["SA"].to(device), K)
            SB = tcm.tcm_mx_pack_scales(case["SB"].to(device), K)
            fmt = "e2m1" if fp4 else None
            self.launch = lambda: tcm.tcm_gemm_mx(A, SA, B, SB, D, stream=stream, fmt=fmt)
        elif case.get("fused"):
            self.peak_mult = FP8_OVER_BF16
            d_scale = torch.tensor([2.0], device=device)
            amax = torch.zeros(1, device=device)
            self.launch = lambda: tcm.tcm_gemm_fused(A, B, D, act=case["fused"], d_scale=d_scale, amax=amax, **kw)
        else:
            if A.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
                self.peak_mult = FP8_OVER_BF16
            if kw.get("b_fmt") is None:
                self.workspace_bytes = tcm.tcm_gemm_workspace_bytes(M, N, K, A.dtype, B.dtype)
                if self.workspace_bytes > 0:
                    kw.update(workspace=torch.empty(self.workspace_bytes, dtype=torch.uint8, device=device))
            self.launch = lambda: tcm.tcm_gemm_ex(A, B, D, **kw)
        self.M, self.N, self.K = M, N, K
        self.in_bytes = (A.numel() // (2 if sparse else 1)) * A.element_size() + B.numel() * B.element_size()
        self.bytes = self.in_bytes + D.numel() * D.element_size() + (C.numel() * C.element_size() if C is not None else 0)
        self.flop = 2.0 * M * N * K
        self.tensors = (A, B, C, D)


def part_cases():
    """(name, builder, bound) of every configured workload besides the step's, then the
    block-scaled, fused and FP4 workloads of the library."""
    return [
        ("c1_bf16_512_C_f32", lambda: si.small_case(), "launch"),
        ("c2_f16_4096", lambda: si.square_case(4096, "f16"), "tensor"),
        ("c2_bf16_4096", lambda: si.square_case(4096, "bf16"), "tensor"),
        ("c3_bf16_8192x28672x8192", lambda: si.llm_case(8192, 28672, 8192), "tensor"),
        ("c3_bf16_8192x8192x28672", lambda: si.llm_case(8192, 8192, 28672), "tensor"),
        ("c3_bf16_8192x24576x8192", lambda: si.llm_case(8192, 24576, 8192), "tensor"),
        ("c3_skinny_bf16_16x28672x8192", lambda: si.llm_case(16, 28672, 8192), "hbm"),
        ("c4_e4m3xe5m2_8192", lambda: si.fp8_case(b_fmt="e5m2"), "tensor"),
        ("f1_mxfp8_e4m3_8192", lambda: si.mx_case(), "tensor"),
        ("f1_nvfp4_8192", lambda: dict(si.nvfp4_case(), nv=True), "tensor"),
        ("f1_mxfp4_8192", lambda: si.mxfp4_case(), "tensor"),
        ("f2_fused_e4m3_gelu_e4m3out_amax_8192", lambda: dict(si.fp8_case(b_fmt="e4m3"), fused="gelu"), "tensor"),
        ("f3_w4a8_e4m3xe2m1_8192", lambda: si.w4a8_case(), "tensor"),
        ("f4_int8_exact_bf16path_8192", lambda: si.int8_case(), "tensor"),
    ]


def run_parts(tcm, device, iters, peaks_used):
    """Each configured workload timed on its own, outside `value`: median device time of
    single launches (L2 flushed first when the inputs fit in it), the mean of back-to-back
    launches, TFLOP/s against the burst tensor peak of its input format and, for the
    HBM-bound skinny shape, GB/s of its algorithmic bytes against the measured copy bandwidth."""
    p, src = peaks_used
    bf16_peak = float(p.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(p.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    stream = torch.cuda.Stream(device=device)
    timer = LaunchTimer(device, stream)
    parts = {}
    for name, build, bound in part_cases():
        w = Workload(name, build(), tcm, device, stream)
        for _ in range(5):
            w.launch()
        flush = w.in_bytes < L2_BYTES
        probe = torch.zeros(3, dtype=torch.int64, device=device)
        tcm.tcm_set_clock_probe(probe)
        t_single = timer.single(w.launch, iters, flush)
        t_b2b = timer.back_to_back(w.launch, iters)
        tcm.tcm_set_clock_probe(None)
        ms = statistics.median(t_single)
        peak = bf16_peak * w.peak_mult
        tf = w.flop / (ms * 1e-3) / 1e12
        rec = {"M": w.M, "N": w.N, "K": w.K, "ms": ms, "ms_min": min(t_single), "ms_back_to_back": t_b2b,
               "tflops": tf, "tflops_back_to_back": w.flop / (t_b2b * 1e-3) / 1e12,
               "frac_of_tensor_peak": tf / peak, "peak_tflops": peak, "bound": bound,
               "device_measured_mhz": probe_mhz(probe), "workspace_bytes": w.workspace_bytes,
               "timing": f"median of {iters} single launches (device sleep before each start event, "
                         f"{'L2 flushed before each' if flush else 'inputs larger than L2, no flush'}); "
                         f"mean of {iters} back-to-back launches"}
        if bound == "hbm":
            t_flushed = timer.single(w.launch, iters, True)
            t_call = timer.single(w.launch, iters, False, sleep=False)
            msf = statistics.median(t_flushed)
            gbs = lambda t: w.bytes / (t * 1e-3) / 1e9
            rec.update({"algorithmic_bytes": w.bytes, "gbs": gbs(ms), "frac_of_hbm": gbs(ms) / hbm_peak,
                        "ms_l2_flushed": msf, "gbs_l2_flushed": gbs(msf), "frac_of_hbm_l2_flushed": gbs(msf) / hbm_peak,
                        "gbs_back_to_back": gbs(t_b2b), "frac_of_hbm_back_to_back": gbs(t_b2b) / hbm_peak,
                        "ms_per_call_synchronised": statistics.median(t_call),
                        "host_call_us": 1e3 * (statistics.median(t_call) - ms)})
        parts[name] = rec
        del w
    torch.cuda.synchronize(device)
    code, site = tcm.tcm_get_device_status(stream)
    if code != 0:
        raise SystemExit(f"device status {code} at site {site} in the per-config parts")
    return parts, timer.windows, (f"{src} bf16_tflops burst (single launches) x the format's nominal dense "
                                  f"ratio: FP8 x{FP8_OVER_BF16:g}, FP4 x{FP4_OVER_BF16:g}, 2:4 logical x2; hbm_gbs")


# ------------------------------------------------------------------ --shapes (extended list)

def shape_cases():
    """(name, builder) for every configured workload shape; builders return CPU inputs."""
    return [
        ("small bf16 512^3 +C fp32 (alpha=beta=1)", lambda: si.small_case()),
        ("square fp16 4096^3", lambda: si.square_case(4096, "f16")),
        ("square bf16 4096^3", lambda: si.square_case(4096, "bf16")),
        ("llm bf16 8192x28672x8192", lambda: si.llm_case(8192, 28672, 8192)),
        ("llm bf16 8192x8192x28672", lambda: si.llm_case(8192, 8192, 28672)),
        ("llm bf16 8192x24576x8192", lambda: si.llm_case(8192, 24576, 8192)),
        ("skinny bf16 16x28672x8192", lambda: si.llm_case(16, 28672, 8192)),
        ("fp8 e4m3xe4m3 8192^3 +scales+bias", lambda: si.fp8_case(b_fmt="e4m3")),
        ("fp8 e4m3xe5m2 8192^3 +scales+bias", lambda: si.fp8_case(b_fmt="e5m2")),
        ("sparse 2:4 bf16 8192^3", lambda: si.sparse_case()),
        ("sparse-tc 2:4 bf16 8192^3 (hardware-ordered metadata)", lambda: dict(si.sparse_case(), tc=True)),
        ("mxfp8 e4m3 8192^3 (E8M0 scales per 32)", lambda: si.mx_case()),
        ("nvfp4 e2m1 8192^3 (UE4M3 scales per 16, per-tensor scales in alpha)", lambda: dict(si.nvfp4_case(), nv=True)),
        ("mxfp4 e2m1 8192^3 (E8M0 scales per 32)", lambda: si.mxfp4_case()),
        ("w4a8 fp8 e4m3 x fp4 e2m1 8192^3 +scales", lambda: si.w4a8_case()),
        ("int8 exact (bf16 tensor path, int32 out, conversions included) 8192^3", lambda: si.int8_case()),
        ("fused fp8 e4m3 8192^3 +scales+bias -> GELU -> e4m3 out (d_scale 2) + amax",
         lambda: dict(si.fp8_case(b_fmt="e4m3"), fused="gelu")),
    ]


def run_shapes(args, tcm, device, peaks_used):
    """Median device time of each configured shape (single launches, L2 flushed when the
    inputs fit in it) and the mean of back-to-back launches; one JSON line each."""
    p, src = peaks_used
    bf16_peak = float(p.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm_peak = float(p.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    stream = torch.cuda.Stream(device=device)
    timer = LaunchTimer(device, stream)
    for name, build in shape_cases():
        if args.only and args.only not in name:
            continue
        w = Workload(name, build(), tcm, device, stream)
        torch.cuda.synchronize(device)
        for _ in range(5):
            w.launch()
        flush = w.in_bytes < L2_BYTES
        probe = torch.zeros(3, dtype=torch.int64, device=device)
        tcm.tcm_set_clock_probe(probe)
        times = timer.single(w.launch, args.shape_iters, flush)
        ms_b2b = timer.back_to_back(w.launch, args.shape_iters)
        tcm.tcm_set_clock_probe(None)
        code, site = tcm.tcm_get_device_status(stream)
        ms = statistics.median(times)
        tf = w.flop / (ms * 1e-3) / 1e12
        gbs = w.bytes / (ms * 1e-3) / 1e9
        peak = bf16_peak * w.peak_mult
        line = {"kind": "shape", "workload": name, "M": w.M, "N": w.N, "K": w.K, "ms_median": ms, "ms_min": min(times),
                "tflops": tf, "frac_of_tensor_peak": tf / peak, "algorithmic_bytes": w.bytes, "gbs": gbs,
                "frac_of_hbm": gbs / hbm_peak, "bound": "hbm" if w.M <= 64 else "tensor", "device_status": code,
                "ms_back_to_back": ms_b2b, "tflops_back_to_back": w.flop / (ms_b2b * 1e-3) / 1e12,
                "device_measured_mhz": probe_mhz(probe), "workspace_bytes": w.workspace_bytes,
                "timing": f"5 warm-up launches, then the median of {args.shape_iters} single launches (device "
                          f"sleep before each start event; " + (
                              "L2 flushed before each)" if flush else "inputs larger than L2, no flush)") +
                          f"; mean of {args.shape_iters} back-to-back launches",
                "peak_source": f"{src} bf16_tflops burst x {w.peak_mult:g}"}
        print(json.dumps(line), flush=True)
        del w


def config_block(world, workspace=True):
    route = ("both through tcm_gemm_ex_ws: the last round's tiles split over K" if workspace
             else "both through tcm_gemm_ex without a workspace: no split tail")
    return {"workload": "GEMM 8192^3 (M=N=K=8192): bf16 x bf16 -> bf16; E4M3 x E4M3 with per-tensor "
                        f"scales + bf16 bias -> bf16 ({route}); 2:4-sparse bf16 A (compress + sparse GEMM on "
                        "canonical metadata) -> bf16; A row-major, B K-major, fp32 accumulate",
            "M": SIZE, "N": SIZE, "K": SIZE,
            "value_counts": "2*M*N*K of the bf16 and E4M3 GEMMs per step (the sparse GEMM runs in the step; "
                            "its logical FLOPs are reported in parts.sp24_gemm_bf16 only)",
            "inputs": "bf16 A ~ N(0,1), B ~ N(0,0.02) (seed 2); E4M3 A, B ~ N(0,1) scaled so amax = 448 (seed 3); "
                      "sparse: logical A, B ~ N(0,1) bf16 (seed 4)",
            "l2": "no flush: each GEMM's inputs (256 MiB bf16, 128 MiB E4M3) exceed the 129 MB L2",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def main():
    args = parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
        return
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
        pg = dist

    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if pg:
        pg.barrier()
    import tensor_core_matrix_gb300 as tcm
    tcm.load_library()
    tcm.tcm_clear_device_status()

    if args.shapes:
        run_shapes(args, tcm, device, peaks())
        return
    # allocate (first-touch) the pinned host buffers from CPUs local to the GPU,
    # so host<->device copies do not cross the CPU-to-CPU link
    saved_affinity = os.sched_getaffinity(0)
    local_cpus = gpu_local_cpus(local_rank_index(device))
    if local_cpus:
        os.sched_setaffinity(0, local_cpus)
    host, pinned, dev = make_inputs(device, workspace=not args.no_workspace)
    # the end-to-end results' pinned buffers (two sets), first-touched here as well
    outs = [{k: torch.empty((SIZE, SIZE), dtype=torch.bfloat16).pin_memory() for k in ("D", "D8", "Dsp")}
            for _ in range(2)] if args.e2e_steps > 0 else None
    os.sched_setaffinity(0, saved_affinity)
    stream = torch.cuda.Stream(device=device)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            run_step(tcm, dev, stream)
    stream.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    # SM clock measured on the device: each GEMM's first CTA adds its cycles and ns
    probes = {k: torch.zeros(3, dtype=torch.int64, device=device)
              for k in ("bf16_dense", "e4m3_scaled_bias", "sp24_gemm_bf16")}
    if pg:
        pg.barrier()
    torch.cuda.synchronize(device)
    with ClockSampler(local_rank_index(device)) as clocks:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        h0 = time.perf_counter()
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for i in range(args.steps):
                run_step(tcm, dev, stream, ev[i], probes)
            t_end.record(stream)
        t_end.synchronize()
        h1 = time.perf_counter()
    torch.cuda.synchronize(device)
    device_mhz = {k: probe_mhz(v) for k, v in probes.items()}
    elapsed_ms = t_start.elapsed_time(t_end)
    bf16_ms = [e[0].elapsed_time(e[1]) for e in ev]
    fp8_ms = [e[1].elapsed_time(e[2]) for e in ev]
    cmp_ms = [e[2].elapsed_time(e[3]) for e in ev]
    sp_ms = [e[3].elapsed_time(e[4]) for e in ev]
    code, site = tcm.tcm_get_device_status(stream)
    if code != 0:
        raise SystemExit(f"device status {code} at site {site}")
    step_clocks = clocks.summary([(h0, h1)])
    # the last timed step's outputs, for the oracle check of the CPU-baseline leg
    check_rows = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = 1024
        check_rows = {k: dev[k][:n].cpu() for k in ("D", "D8", "Dsp", "Ac", "meta")}

    # end-to-end: every step copies all of its inputs in from pinned host memory
    # and all three results back out.  Copies run on their own streams and are
    # pipelined against the GEMMs of the neighbouring steps (two device sets).
    e2e_ms = None
    h2d = sum(pinned[k].numel() * pinned[k].element_size() for k in pinned)
    d2h = 3 * SIZE * SIZE * 2
    if args.e2e_steps > 0:
        sets = [dev, {k: torch.empty_like(v) for k, v in dev.items()}]
        s_in, s_out = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)

        def e2e_steps(n):
            """n pipelined end-to-end steps; returns their total time in ms (s_in start to s_out end)."""
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_comp = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(s_in)
            for i in range(n):
                d = sets[i % 2]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(ev_comp[i - 2])  # the GEMMs of step i-2 finished reading this set
                    for k in pinned:
                        d[k].copy_(pinned[k], non_blocking=True)
                    ev_in[i].record(s_in)
                with torch.cuda.stream(stream):
                    stream.wait_event(ev_in[i])
                    if i >= 2:
                        stream.wait_event(ev_out[i - 2])  # results of step i-2 copied out of this set
                    run_step(tcm, d, stream)
                    ev_comp[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_comp[i])
                    for k in outs[i % 2]:
                        outs[i % 2][k].copy_(d[k], non_blocking=True)
                    ev_out[i].record(s_out)
            s_out.wait_event(ev_out[-1])
            e1.record(s_out)
            e1.synchronize()
            return e0.elapsed_time(e1)

        # untimed warm-up of the copy path: after the device-only loop above, the first
        # host copies run far slower (measured: 111 ms for one step's 671 MB in)
        e2e_steps(max(8, args.warmup))
        if pg:
            pg.barrier()
        torch.cuda.synchronize(device)
        e2e_ms = e2e_steps(args.e2e_steps) / args.e2e_steps
        del sets

    elapsed_ms, e2e_max = slowest_rank(pg, [elapsed_ms, e2e_ms or 0.0], device)

    parts_cfg, parts_clocks, parts_peak = {}, None, None
    if not args.no_parts and rank == 0:
        del dev
        torch.cuda.empty_cache()
        with ClockSampler(local_rank_index(device)) as pclocks:
            parts_cfg, windows, parts_peak = run_parts(tcm, device, args.part_iters, peaks())
        parts_clocks = pclocks.summary(windows)

    exit_code = 0
    if rank == 0:
        p, src = peaks()
        region_s = elapsed_ms * 1e-3
        bf16_peak, peak_label = bf16_peak_for(region_s, (p, src))
        ms_step = elapsed_ms / args.steps
        flop_step = DENSE_GEMMS_PER_STEP * FLOP_PER_GEMM
        value = whole_job_rate(world, flop_step * args.steps, elapsed_ms * 1e-3) / 1e12
        t_bf16 = statistics.mean(bf16_ms)
        t_fp8 = statistics.mean(fp8_ms)
        ach_bf16 = FLOP_PER_GEMM / (t_bf16 * 1e-3) / 1e12
        ach_fp8 = FLOP_PER_GEMM / (t_fp8 * 1e-3) / 1e12
        fp8_peak = bf16_peak * FP8_OVER_BF16
        t_cmp = statistics.mean(cmp_ms)
        t_sp = statistics.mean(sp_ms)
        ach_sp = FLOP_PER_GEMM / (t_sp * 1e-3) / 1e12
        hbm_peak = float(p.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        cmp_gbs = COMPRESS_BYTES / (t_cmp * 1e-3) / 1e9
        sms = torch.cuda.get_device_properties(device).multi_processor_count
        mhz = device_mhz.get("bf16_dense")
        clock_peak = sms * BF16_FLOP_PER_CLK_PER_SM * mhz * 1e6 / 1e12 if mhz else None
        step_clocks["device_measured_mhz"] = device_mhz
        step_clocks["device_measured_note"] = ("SM clock during each GEMM of the timed region, measured on the "
                                               "device: %clock64 cycles / %globaltimer ns of each launch's first CTA")
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16+e4m3", "data": "synthetic",
            "config": config_block(world, not args.no_workspace),
            "parts": {
                "bf16_dense": {"tflops": ach_bf16, "ms": t_bf16, "frac_of_bf16_peak": ach_bf16 / bf16_peak},
                "e4m3_scaled_bias": {"tflops": ach_fp8, "ms": t_fp8, "frac_of_fp8_peak": ach_fp8 / fp8_peak},
                "sp24_compress": {"gbs": cmp_gbs, "ms": t_cmp, "frac_of_hbm": cmp_gbs / hbm_peak,
                                  "bytes": COMPRESS_BYTES},
                "sp24_gemm_bf16": {"tflops_logical": ach_sp, "ms": t_sp,
                                   "frac_of_2to4_peak": ach_sp / (2 * bf16_peak),
                                   "note": "logical 2*M*N*K (twice the issued MMA work); peak = 2 x dense bf16"},
                "peak_source": peak_label,
                **parts_cfg,
            },
            "roofline": {"bound": "tensor", "achieved": ach_bf16, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": ach_bf16 / bf16_peak, "traffic": recorded_traffic(),
                         "kernel": "gemm_kernel<kind::f16, 256x256 CTA-pair tile, 6 stages> bf16 8192^3",
                         "peak_source": peak_label, "timed_region_s": region_s,
                         "algorithmic_flop_per_launch": FLOP_PER_GEMM},
            "gpu_launches": KERNELS_PER_STEP * args.steps,
            "clocks": step_clocks,
        }
        if clock_peak:
            line["roofline"]["clock_derived"] = {
                "sm_mhz": mhz, "sms": sms, "flop_per_clk_per_sm": BF16_FLOP_PER_CLK_PER_SM,
                "peak_tflops": clock_peak, "frac": ach_bf16 / clock_peak,
                "kernel_time_x_mhz_mcycles": t_bf16 * 1e-3 * mhz,
                "note": "SMs x dense bf16 FLOP per clock per SM x the SM clock measured on the device during "
                        "the bf16 launches of the timed region"}
        if parts_clocks is not None:
            line["parts"]["clocks"] = parts_clocks
            line["parts"]["config_peak_source"] = parts_peak
        if e2e_ms:
            line["e2e"] = {"value": whole_job_rate(world, flop_step, e2e_max * 1e-3) / 1e12, "unit": "TFLOP/s",
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                           "note": f"{args.e2e_steps} steps after {max(8, args.warmup)} untimed ones; every step "
                                   f"copies all inputs in from pinned host "
                                   f"memory and all three D out; copies overlap the GEMMs of neighbouring steps; "
                                   f"pinned buffers allocated from "
                                   f"{'GPU-local CPUs ' + str(len(local_cpus)) if local_cpus else 'the default CPU set'}"}
        if check_rows is not None:
            base, check = cpu_baseline_sample(host, args.cpu_seconds, check_rows)
            line["cpu_baseline"] = base
            line["check"] = check
            if not check["ok"]:
                exit_code = 1
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    if exit_code:
        raise SystemExit(f"timed outputs outside the oracle bound: {line['check']}")


if __name__ == "__main__":
    main()
