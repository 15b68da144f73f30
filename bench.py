"""Throughput of the tcgen05 GEMM hot path on GB300, one JSON line per run.

A step is one pass of the hot path over one batch of resident synthetic
input at M = N = K = 8192:
  * bf16 x bf16 -> fp32 accumulate -> bf16 D (alpha = 1, beta = 0)
  * E4M3 x E4M3 with per-tensor fp32 dequantisation scales and a bf16 bias
    -> bf16 D
  * 2:4 structured-sparse bf16 A: compress of the logical A (keep the two
    largest of every four along K, ordered metadata), a copy of the metadata
    into the sparse MMA's tensor-memory order, and the sparse GEMM, counted
    at its logical 2*M*N*K
value = sum of 2*M*N*K over the step's three GEMMs / step time (TFLOP/s).

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
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 / bf16 tensor rates (GB300)
FP8_OVER_BF16 = 4.5 / 2.25  # nominal dense ratio
L2_BYTES = 129 * 10 ** 6
KERNEL_SOURCES = ["tensor_core_matrix_gb300/csrc/tcm_gemm_kernel.cuh", "tensor_core_matrix_gb300/csrc/tcm_kernel_common.cuh",
                  "tensor_core_matrix_gb300/csrc/tcm_ptx.cuh", "tensor_core_matrix_gb300/csrc/tcm_gemm_pair.cu"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_kernel_bf16_8192cubed.md")


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["tcm", "reference"], default="tcm")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
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
        entry = line.strip().lstrip("-* ").strip("`")
        if "=" in entry and entry.startswith(("dram_bytes_per_launch", "kernel_source_sha")):
            k, v = entry.split("=", 1)
            vals[k.strip().strip("`")] = v.strip().strip("` ")
    if vals.get("kernel_source_sha") != kernel_source_sha():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def smi_gpu_id(dev_index):
    """nvidia-smi's name for CUDA device `dev_index`: its UUID (nvidia-smi numbers the
    machine's GPUs itself and ignores CUDA_VISIBLE_DEVICES, so an index may name another GPU)."""
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        if u:
            return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        pass
    vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    return vis[dev_index].strip() if dev_index < len(vis) else str(dev_index)


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
            self.err = open(self.path + ".err", "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", smi_gpu_id(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=self.err)
        except (OSError, FileNotFoundError):
            self.proc = None
            return self
        # do not start the timed region before the sampler is producing samples
        deadline = time.time() + 15.0
        while time.time() < deadline and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.05)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()
            self.err.close()

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
        err = ""
        if os.path.exists(self.path + ".err"):
            err = open(self.path + ".err").read().strip().splitlines()[:1]
            err = err[0][:200] if err else ""
            os.unlink(self.path + ".err")
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples" + (f": {err}" if err else "")],
                    "samples": 0}
        loaded = [r for r in rows if r[2] > 300.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": max(r[2] for r in rows)}


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


def make_inputs(device):
    """Resident device inputs of one step plus their pinned host copies (for the end-to-end leg)."""
    dense = si.llm_case(SIZE, SIZE, SIZE, seed=2)  # bf16 A ~ N(0,1), B ~ N(0, 0.02)
    f8 = si.fp8_case(SIZE, SIZE, SIZE, b_fmt="e4m3", seed=3)
    sp = si.sparse_case(SIZE, SIZE, SIZE, seed=4)
    host = {
        "A": dense["A"], "B": dense["B"],
        "A8": f8["A"], "B8": f8["B"], "bias": f8["bias"],
        "sa": torch.tensor([f8["sa"]], dtype=torch.float32), "sb": torch.tensor([f8["sb"]], dtype=torch.float32),
        "Asp": sp["A_logical"], "Bsp": sp["B"],
    }
    pinned = {k: v.pin_memory() for k, v in host.items()}
    dev = {k: v.to(device) for k, v in host.items()}
    for k in ("D", "D8", "Dsp"):
        dev[k] = torch.empty((SIZE, SIZE), dtype=torch.bfloat16, device=device)
    dev["Ac"] = torch.empty((SIZE, SIZE // 2), dtype=torch.bfloat16, device=device)
    dev["meta"] = torch.empty((SIZE, SIZE // 32), dtype=torch.int32, device=device)
    dev["meta_tc"] = torch.empty(META_TC_BYTES, dtype=torch.uint8, device=device)
    return host, pinned, dev


def run_step(tcm, dev, stream, events=None):
    """One pass of the hot path; events[0..4] bracket the four launches on `stream`."""
    def mark(i):
        if events:
            events[i].record(stream)
    mark(0)
    tcm.tcm_gemm_ex(dev["A"], dev["B"], dev["D"], stream=stream)
    mark(1)
    tcm.tcm_gemm_ex(dev["A8"], dev["B8"], dev["D8"], a_scale=dev["sa"], b_scale=dev["sb"], bias=dev["bias"],
                    stream=stream)
    mark(2)
    tcm.tcm_sp_compress(dev["Asp"], dev["Ac"], dev["meta"], stream=stream)
    tcm.tcm_sp_meta_pack(dev["meta"], SIZE, dev["meta_tc"], stream=stream)
    mark(3)
    tcm.tcm_gemm_sp_tc(dev["Ac"], dev["meta_tc"], dev["Bsp"], dev["Dsp"], stream=stream)
    mark(4)


KERNELS_PER_STEP = 5
# hardware-ordered metadata: ceil(M/128) * ceil(K/128) * 2048 bytes
META_TC_BYTES = (SIZE // 128) * (SIZE // 128) * 2048
GEMMS_PER_STEP = 3
# compress (read A, write A_comp + canonical metadata) and metadata pack (read it, write meta_tc)
COMPRESS_BYTES = SIZE * SIZE * 2 + SIZE * (SIZE // 2) * 2 + 2 * SIZE * (SIZE // 32) * 4 + META_TC_BYTES


class OracleSample:
    """The CPU oracle on whole output rows of the step's three GEMMs (and the 2:4 compress of those rows)."""

    def __init__(self, host):
        import oracle
        self.oracle = oracle
        oracle.build()
        self.a, self.b = si.codes(host["A"]), si.codes(host["B"])
        self.a8, self.b8, self.bias = si.codes(host["A8"]), si.codes(host["B8"]), si.codes(host["bias"])
        self.sa, self.sb = float(host["sa"][0]), float(host["sb"][0])
        self.asp, self.bsp = si.codes(host["Asp"]), si.codes(host["Bsp"])

    def rows(self, r):
        import numpy as np
        o = self.oracle
        rows = np.repeat(np.arange(r, dtype=np.int64), SIZE)
        cols = np.tile(np.arange(SIZE, dtype=np.int64), r)
        o.gemm(self.a, self.b, "bf16", "bf16", rows=rows, cols=cols)
        o.gemm(self.a8, self.b8, "e4m3", "e4m3", bias=self.bias, sa=self.sa, sb=self.sb, rows=rows, cols=cols)
        ac, meta = o.sp_compress(np.ascontiguousarray(self.asp[:r]), "bf16")
        o.gemm(o.sp_decompress(ac, meta, "bf16"), self.bsp, "bf16", "bf16", rows=rows, cols=cols)
        return GEMMS_PER_STEP * 2.0 * r * SIZE * SIZE

    def calibrate(self, seconds):
        t0 = time.perf_counter()
        self.rows(1)
        per_row = max(time.perf_counter() - t0, 1e-6)
        return max(1, int(seconds / per_row))


def cpu_baseline_sample(host, seconds):
    """Time the CPU oracle on about `seconds` of whole output rows of the step's GEMMs."""
    o = OracleSample(host)
    r = o.calibrate(seconds)
    t0 = time.perf_counter()
    flop = o.rows(r)
    t = time.perf_counter() - t0
    cores = len(os.sched_getaffinity(0))
    return {"value": flop / t / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{r} full output rows (8192 outputs of K=8192 each) of each of the step's three GEMMs "
                      f"(bf16, E4M3 with scales+bias, 2:4-sparse bf16 incl. compress of those rows), "
                      f"{t:.1f} s on {cores} host threads (OpenMP)"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    dense = si.llm_case(SIZE, SIZE, SIZE, seed=2)
    f8 = si.fp8_case(SIZE, SIZE, SIZE, b_fmt="e4m3", seed=3)
    sp = si.sparse_case(SIZE, SIZE, SIZE, seed=4)
    host = {"A": dense["A"], "B": dense["B"], "A8": f8["A"], "B8": f8["B"], "bias": f8["bias"],
            "sa": torch.tensor([f8["sa"]]), "sb": torch.tensor([f8["sb"]]),
            "Asp": sp["A_logical"], "Bsp": sp["B"]}
    o = OracleSample(host)
    cores = len(os.sched_getaffinity(0))
    r = o.calibrate(90.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        o.rows(r)
    t0 = time.perf_counter()
    flop = 0.0
    for _ in range(args.steps):
        flop += o.rows(r)
    t = time.perf_counter() - t0
    value = flop / t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16+e4m3",
        "data": "synthetic", "config": config_block(world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {r} full output rows of each of the three 8192^3 GEMMs "
                                   f"(fp64 CPU oracle, {cores} host threads)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


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
        ("mxfp8 e4m3 8192^3 (E8M0 scales per 32)", lambda: si.mx_case()),
        ("nvfp4 e2m1 8192^3 (UE4M3 scales per 16, per-tensor scales in alpha)", lambda: dict(si.nvfp4_case(), nv=True)),
        ("w4a8 fp8 e4m3 x fp4 e2m1 8192^3 +scales", lambda: si.w4a8_case()),
        ("fused fp8 e4m3 8192^3 +scales+bias -> GELU -> e4m3 out (d_scale 2) + amax",
         lambda: dict(si.fp8_case(b_fmt="e4m3"), fused="gelu")),
    ]


def run_shapes(args, tcm, device, peaks_used):
    """Median device time of each configured shape, L2 flushed before every timed launch."""
    p, src = peaks_used
    bf16_peak = float(p.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    hbm_peak = float(p.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    for name, build in shape_cases():
        if args.only and args.only not in name:
            continue
        case = build()
        sparse = "A_logical" in case
        A = (case["A_logical"] if sparse else case["A"]).to(device)
        B = case["B"].to(device)
        M, K = A.shape
        N = B.shape[0]
        out_dtype = torch.float32 if case.get("out_fmt") == "f32" else torch.bfloat16
        if case.get("fused"):
            out_dtype = torch.float8_e4m3fn
        D = torch.empty((M, N), dtype=out_dtype, device=device)
        C = case["C"].to(device) if case.get("C") is not None else None
        kw = dict(C=C, alpha=case.get("alpha", 1.0), beta=case.get("beta", 0.0))
        if "sa" in case:
            kw.update(a_scale=torch.tensor([case["sa"]], device=device), b_scale=torch.tensor([case["sb"]], device=device))
            if case.get("bias") is not None:
                kw.update(bias=case["bias"].to(device))
        if case.get("b_fmt") == "e2m1":
            kw.update(b_fmt="e2m1")  # B holds N x K/2 bytes of packed FP4
        if sparse:
            Ac, meta = tcm.tcm_sp_compress(A)
            meta_tc = tcm.tcm_sp_meta_pack(meta, K)
            launch = lambda: tcm.tcm_gemm_sp_tc(Ac, meta_tc, B, D, C=C, alpha=kw["alpha"], beta=kw["beta"])
        elif case.get("nv"):
            SA = tcm.tcm_nvfp4_pack_scales(case["SA"].to(device), 2 * K)
            SB = tcm.tcm_nvfp4_pack_scales(case["SB"].to(device), 2 * K)
            K = 2 * K  # A holds K/2 bytes per row
            launch = lambda: tcm.tcm_gemm_nvfp4(A, SA, B, SB, D, alpha=case["alpha"])
        elif "SA" in case:
            # scales packed once into the blocked layout (as a quantiser would emit them)
            SA = tcm.tcm_mx_pack_scales(case["SA"].to(device), K)
            SB = tcm.tcm_mx_pack_scales(case["SB"].to(device), K)
            launch = lambda: tcm.tcm_gemm_mx(A, SA, B, SB, D)
        elif case.get("fused"):
            d_scale = torch.tensor([2.0], device=device)
            amax = torch.zeros(1, device=device)
            launch = lambda: tcm.tcm_gemm_fused(A, B, D, act=case["fused"], d_scale=d_scale, amax=amax, **kw)
        else:
            launch = lambda: tcm.tcm_gemm_ex(A, B, D, **kw)
        for _ in range(5):
            launch()
        in_bytes_total = sum(t.numel() * t.element_size() for t in (A, B) if t is not None)
        needs_flush = in_bytes_total < L2_BYTES  # inputs larger than L2 are not flushed
        times = []
        for _ in range(args.shape_iters):
            if needs_flush:
                flush.fill_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            launch()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        ms_b2b = ms_flushed = None
        if not needs_flush:
            # also with L2 flushed before each launch (the inputs exceed L2, so this changes little)
            flushed = []
            for _ in range(args.shape_iters):
                flush.fill_(1)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                launch()
                e1.record(stream)
                e1.synchronize()
                flushed.append(e0.elapsed_time(e1))
            ms_flushed = statistics.median(flushed)
            # the same launches back to back (inputs exceed L2 anyway): the host-side cost of
            # each call (tensor maps, launch) overlaps the previous kernel instead of adding to it
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.shape_iters):
                launch()
            e1.record(stream)
            e1.synchronize()
            ms_b2b = e0.elapsed_time(e1) / args.shape_iters
        code, site = tcm.tcm_get_device_status()
        ms = statistics.median(times)
        flop = 2.0 * M * N * K
        in_bytes = (A.numel() // (2 if sparse else 1)) * A.element_size() + B.numel() * B.element_size()
        byts = in_bytes + D.numel() * D.element_size() + (C.numel() * C.element_size() if C is not None else 0)
        tf = flop / (ms * 1e-3) / 1e12
        gbs = byts / (ms * 1e-3) / 1e9
        peak = bf16_peak * (FP4_OVER_BF16 if "nvfp4" in name else
                            FP8_OVER_BF16 if ("fp8" in name or "mx" in name) else 1.0)  # fused, w4a8: FP8 rate
        line = {"kind": "shape", "workload": name, "M": M, "N": N, "K": K, "ms_median": ms, "ms_min": min(times),
                "tflops": tf, "frac_of_tensor_peak": tf / peak, "algorithmic_bytes": byts, "gbs": gbs,
                "frac_of_hbm": gbs / hbm_peak, "bound": "hbm" if M <= 64 else "tensor", "device_status": code,
                "ms_back_to_back": ms_b2b, "ms_median_l2_flushed": ms_flushed,
                "timing": f"5 warm-up launches, then the median of {args.shape_iters} launches, each synchronised; " + (
                    "L2 flushed (256 MiB write) before each" if needs_flush else "inputs larger than L2, no flush"),
                "peak_source": src}
        print(json.dumps(line), flush=True)
        del A, B, D, C, case


def config_block(world):
    return {"workload": "GEMM 8192^3 (M=N=K=8192): bf16 x bf16 -> bf16; E4M3 x E4M3 with per-tensor "
                        "scales + bf16 bias -> bf16; 2:4-sparse bf16 A (compress + metadata pack + sparse GEMM) -> bf16; "
                        "A row-major, B K-major, fp32 accumulate",
            "M": SIZE, "N": SIZE, "K": SIZE,
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
    local = gpu_local_cpus(local_rank_index(device))
    if local:
        os.sched_setaffinity(0, local)
    host, pinned, dev = make_inputs(device)
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
    cmp_ms = [e[2].elapsed_time(e[3]) for e in ev]
    sp_ms = [e[3].elapsed_time(e[4]) for e in ev]
    code, site = tcm.tcm_get_device_status(stream)
    if code != 0:
        raise SystemExit(f"device status {code} at site {site}")

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

        # untimed warm-up of the copy path: after the seconds-long device-only loop above, the
        # first host copies run far slower (measured: 111 ms for one step's 671 MB in)
        e2e_steps(max(8, args.warmup))
        if pg:
            pg.barrier()
        torch.cuda.synchronize(device)
        e2e_ms = e2e_steps(args.e2e_steps) / args.e2e_steps

    elapsed_ms, e2e_max = slowest_rank(pg, [elapsed_ms, e2e_ms or 0.0], device)

    if rank == 0:
        p, src = peaks()
        bf16_peak = float(p.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        ms_step = elapsed_ms / args.steps
        flop_step = GEMMS_PER_STEP * FLOP_PER_GEMM
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
        traffic = recorded_traffic()
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16+e4m3", "data": "synthetic", "config": config_block(world),
            "parts": {
                "bf16_dense": {"tflops": ach_bf16, "ms": t_bf16, "frac_of_bf16_peak": ach_bf16 / bf16_peak},
                "e4m3_scaled_bias": {"tflops": ach_fp8, "ms": t_fp8, "frac_of_fp8_peak": ach_fp8 / fp8_peak},
                "sp24_compress_and_meta_pack": {"gbs": cmp_gbs, "ms": t_cmp, "frac_of_hbm": cmp_gbs / hbm_peak,
                                                "bytes": COMPRESS_BYTES},
                "sp24_gemm_bf16": {"tflops_logical": ach_sp, "ms": t_sp,
                                   "frac_of_dense_bf16_peak": ach_sp / bf16_peak},
            },
            "roofline": {"bound": "tensor", "achieved": ach_bf16, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": ach_bf16 / bf16_peak, "traffic": traffic,
                         "kernel": "gemm_kernel<kind::f16, 256x256 CTA-pair tile, 6 stages> bf16 8192^3",
                         "peak_source": f"{src} bf16_tflops_sustained (kernel timed inside a multi-second "
                                        f"back-to-back loop)",
                         "algorithmic_flop_per_launch": FLOP_PER_GEMM},
            "gpu_launches": KERNELS_PER_STEP * args.steps,
            "clocks": clocks.summary(),
        }
        if e2e_ms:
            line["e2e"] = {"value": whole_job_rate(world, flop_step, e2e_max * 1e-3) / 1e12, "unit": "TFLOP/s",
                           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                           "note": f"{args.e2e_steps} steps after {max(8, args.warmup)} untimed ones; every step "
                                   f"copies all inputs in from pinned host "
                                   f"memory and all three D out; copies overlap the GEMMs of neighbouring steps; "
                                   f"pinned buffers allocated from "
                                   f"{'GPU-local CPUs ' + str(len(local)) if local else 'the default CPU set'}"}
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline_sample(host, args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
