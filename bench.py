"""Throughput of the tcgen05 GEMM hot path on GB300, one JSON line per run.

A step is one pass of the hot path over one batch of resident synthetic
input at M = N = K = 8192:
  * bf16 x bf16 -> fp32 accumulate -> bf16 D (alpha = 1, beta = 0)
  * E4M3 x E4M3 with per-tensor fp32 dequantisation scales and a bf16 bias
    -> bf16 D
  * 2:4 structured-sparse bf16 A: compress of the logical A plus the sparse
    GEMM (logical FLOPs), once that path is available in the library
value = sum of 2*M*N*K over the step's GEMMs / step time (TFLOP/s).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tcm|reference]

With torchrun (N > 1) every rank runs an independent replica on its own GPU
(weak scaling); the slowest rank's time counts.  ``--impl reference`` times
the CPU oracle instead (rank 0 only), on bounded samples of the same work.
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

import torch  # noqa: E402

import synth_inputs as si  # noqa: E402

SIZE = 8192
FLOP_PER_GEMM = 2.0 * SIZE ** 3
METRIC = "GEMM TFLOP/s (2MNK/t) at 8192^3 bf16 and FP8; % of GB300 dense tensor peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP8_OVER_BF16 = 4.5 / 2.25  # nominal dense ratio
KERNEL_SOURCES = ["tensor_core_matrix_gb300/csrc/tcm_gemm.cu", "tensor_core_matrix_gb300/csrc/tcm_ptx.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_kernel_bf16_8192cubed.md")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["tcm", "reference"], default="tcm")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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


def kernel_source_sha():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """dram bytes per launch of the bf16 8192^3 kernel from the committed ncu summary, if still current."""
    try:
        text = open(TRAFFIC_FILE).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if "=" in line and line.strip().startswith(("dram_bytes_per_launch", "kernel_source_sha")):
            k, v = line.split("=", 1)
            vals[k.strip().strip("`- ")] = v.strip().strip("` ")
    if vals.get("kernel_source_sha") != kernel_source_sha():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"tcm_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        loaded = [r for r in rows if r[2] > 300.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r[2] for r in rows)}


def make_inputs(device):
    """Resident device inputs of one step plus their pinned host copies (for the end-to-end leg)."""
    dense = si.llm_case(SIZE, SIZE, SIZE, seed=2)  # bf16 A ~ N(0,1), B ~ N(0, 0.02)
    f8 = si.fp8_case(SIZE, SIZE, SIZE, b_fmt="e4m3", seed=3)
    host = {
        "A": dense["A"], "B": dense["B"],
        "A8": f8["A"], "B8": f8["B"], "bias": f8["bias"],
        "sa": torch.tensor([f8["sa"]], dtype=torch.float32), "sb": torch.tensor([f8["sb"]], dtype=torch.float32),
    }
    pinned = {k: v.pin_memory() for k, v in host.items()}
    dev = {k: v.to(device) for k, v in host.items()}
    dev["D"] = torch.empty((SIZE, SIZE), dtype=torch.bfloat16, device=device)
    dev["D8"] = torch.empty((SIZE, SIZE), dtype=torch.bfloat16, device=device)
    return host, pinned, dev


def run_step(tcm, dev, stream, events=None):
    """One pass of the hot path; events = (e0, e1, e2) brackets the two GEMMs on `stream`."""
    if events:
        events[0].record(stream)
    tcm.tcm_gemm_ex(dev["A"], dev["B"], dev["D"], stream=stream)
    if events:
        events[1].record(stream)
    tcm.tcm_gemm_ex(dev["A8"], dev["B8"], dev["D8"], a_scale=dev["sa"], b_scale=dev["sb"], bias=dev["bias"],
                    stream=stream)
    if events:
        events[2].record(stream)


KERNELS_PER_STEP = 2


def cpu_baseline_sample(host, seconds):
    """Time the CPU oracle on whole output rows of the step's two GEMMs for about `seconds`."""
    import numpy as np

    import oracle

    a, b = si.codes(host["A"]), si.codes(host["B"])
    a8, b8, bias = si.codes(host["A8"]), si.codes(host["B8"]), si.codes(host["bias"])
    sa, sb = float(host["sa"][0]), float(host["sb"][0])

    def rows_run(r, gemm):
        rows = np.repeat(np.arange(r, dtype=np.int64), SIZE)
        cols = np.tile(np.arange(SIZE, dtype=np.int64), r)
        if gemm == 0:
            oracle.gemm(a, b, "bf16", "bf16", rows=rows, cols=cols)
        else:
            oracle.gemm(a8, b8, "e4m3", "e4m3", bias=bias, sa=sa, sb=sb, rows=rows, cols=cols)

    t0 = time.perf_counter()
    rows_run(1, 0)
    rows_run(1, 1)
    per_pair = max(time.perf_counter() - t0, 1e-6)
    r = max(1, int(seconds / per_pair))
    t0 = time.perf_counter()
    rows_run(r, 0)
    rows_run(r, 1)
    t = time.perf_counter() - t0
    flop = 2 * (2.0 * r * SIZE * SIZE)
    cores = len(os.sched_getaffinity(0))
    return {"value": flop / t / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{r} full output rows (8192 outputs of K=8192 each) of the bf16 and of the E4M3 GEMM, "
                      f"{t:.1f} s on {cores} host threads (OpenMP)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    oracle.build()
    dense = si.llm_case(SIZE, SIZE, SIZE, seed=2)
    f8 = si.fp8_case(SIZE, SIZE, SIZE, b_fmt="e4m3", seed=3)
    a, b = si.codes(dense["A"]), si.codes(dense["B"])
    a8, b8, bias = si.codes(f8["A"]), si.codes(f8["B"]), si.codes(f8["bias"])
    cores = len(os.sched_getaffinity(0))

    def step(r):
        rows = np.repeat(np.arange(r, dtype=np.int64), SIZE)
        cols = np.tile(np.arange(SIZE, dtype=np.int64), r)
        oracle.gemm(a, b, "bf16", "bf16", rows=rows, cols=cols)
        oracle.gemm(a8, b8, "e4m3", "e4m3", bias=bias, sa=f8["sa"], sb=f8["sb"], rows=rows, cols=cols)

    t0 = time.perf_counter()
    step(1)
    per_row = max(time.perf_counter() - t0, 1e-6)
    budget = 90.0 / max(1, args.steps + args.warmup)
    r = max(1, int(budget / per_row))
    for _ in range(args.warmup):
        step(r)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step(r)
    t = time.perf_counter() - t0
    value = args.steps * 2 * (2.0 * r * SIZE * SIZE) / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16+e4m3",
        "data": "synthetic", "config": config_block(world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {r} full output rows of the bf16 and of the E4M3 8192^3 GEMM "
                                   f"(fp64 CPU oracle, {cores} host threads)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(world):
    return {"workload": "GEMM 8192^3 (M=N=K=8192): bf16 x bf16 -> bf16, and E4M3 x E4M3 with per-tensor "
                        "scales + bf16 bias -> bf16; A row-major, B K-major, fp32 accumulate",
            "M": SIZE, "N": SIZE, "K": SIZE,
            "inputs": "bf16 A ~ N(0,1), B ~ N(0,0.02) (seed 2); E4M3 A, B ~ N(0,1) scaled so amax = 448 (seed 3)",
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

    host, pinned, dev = make_inputs(device)
    stream = torch.cuda.Stream(device=device)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            run_step(tcm, dev, stream)
    stream.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize(device)
    with ClockSampler(local) as clocks:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for i in range(args.steps):
                run_step(tcm, dev, stream, ev[i])
            t_end.record(stream)
        t_end.synchronize()
    torch.cuda.synchronize(device)
    elapsed_ms = t_start.elapsed_time(t_end)
    bf16_ms = [e[0].elapsed_time(e[1]) for e in ev]
    fp8_ms = [e[1].elapsed_time(e[2]) for e in ev]
    code, site = tcm.tcm_get_device_status(stream)
    if code != 0:
        raise SystemExit(f"device status {code} at site {site}")

    # end-to-end: pinned host inputs -> device, the step, result -> host, every step
    e2e_ms = None
    h2d = sum(pinned[k].numel() * pinned[k].element_size() for k in pinned)
    d2h = 2 * SIZE * SIZE * 2
    if args.e2e_steps > 0:
        outD = torch.empty((SIZE, SIZE), dtype=torch.bfloat16).pin_memory()
        outD8 = torch.empty((SIZE, SIZE), dtype=torch.bfloat16).pin_memory()
        if pg:
            pg.barrier()
        torch.cuda.synchronize(device)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.e2e_steps):
                for k in pinned:
                    dev[k].copy_(pinned[k], non_blocking=True)
                run_step(tcm, dev, stream)
                outD.copy_(dev["D"], non_blocking=True)
                outD8.copy_(dev["D8"], non_blocking=True)
            e1.record(stream)
        e1.synchronize()
        e2e_ms = e0.elapsed_time(e1) / args.e2e_steps

    # slowest rank decides
    times = torch.tensor([elapsed_ms, e2e_ms or 0.0], dtype=torch.float64, device=device)
    if pg:
        pg.all_reduce(times, op=pg.ReduceOp.MAX)
    elapsed_ms, e2e_max = float(times[0]), float(times[1])

    if rank == 0:
        p, src = peaks()
        bf16_peak = float(p.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        ms_step = elapsed_ms / args.steps
        flop_step = KERNELS_PER_STEP * FLOP_PER_GEMM
        value = world * flop_step * args.steps / (elapsed_ms * 1e-3) / 1e12
        t_bf16 = statistics.mean(bf16_ms)
        t_fp8 = statistics.mean(fp8_ms)
        ach_bf16 = FLOP_PER_GEMM / (t_bf16 * 1e-3) / 1e12
        ach_fp8 = FLOP_PER_GEMM / (t_fp8 * 1e-3) / 1e12
        fp8_peak = bf16_peak * FP8_OVER_BF16
        traffic = recorded_traffic()
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16+e4m3", "data": "synthetic", "config": config_block(world),
            "parts": {
                "bf16_dense": {"tflops": ach_bf16, "ms": t_bf16, "frac_of_bf16_peak": ach_bf16 / bf16_peak},
                "e4m3_scaled_bias": {"tflops": ach_fp8, "ms": t_fp8, "frac_of_fp8_peak": ach_fp8 / fp8_peak},
            },
            "roofline": {"bound": "tensor", "achieved": ach_bf16, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": ach_bf16 / bf16_peak, "traffic": traffic,
                         "kernel": "gemm_kernel<kind::f16, BN=256> bf16 8192^3",
                         "peak_source": f"{src} bf16_tflops_sustained (kernel timed inside a multi-second "
                                        f"back-to-back loop)",
                         "algorithmic_flop_per_launch": FLOP_PER_GEMM},
            "gpu_launches": KERNELS_PER_STEP * args.steps,
            "clocks": clocks.summary(),
        }
        if e2e_ms:
            line["e2e"] = {"value": world * flop_step / (e2e_max * 1e-3) / 1e12, "unit": "TFLOP/s",
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                           "note": "pinned host inputs copied in and both D copied out every step"}
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline_sample(host, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
