"""Host-side pieces of bench.py that need no GPU: the recorded DRAM traffic of the
roofline kernel (read from its committed ncu record only while the kernel source is
unchanged), the choice of the peak from the timed region's length, the clock summary
over the timed windows, and the oracle check of the timed outputs."""
import json

import numpy as np
import pytest
import torch

import bench
import oracle
import synth_inputs as si


def test_recorded_traffic_reads_the_committed_record(tmp_path, monkeypatch):
    rec = tmp_path / "rec.json"
    rec.write_text(json.dumps({"dram_bytes_per_launch": 1234, "kernel_source_sha": bench.kernel_source_sha()}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    assert bench.recorded_traffic() == 1234.0


def test_recorded_traffic_is_null_once_the_kernel_changed(tmp_path, monkeypatch):
    rec = tmp_path / "rec.json"
    rec.write_text(json.dumps({"dram_bytes_per_launch": 1234, "kernel_source_sha": "0000000000000000"}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    assert bench.recorded_traffic() is None


def test_committed_traffic_record_is_well_formed():
    rec = json.load(open(bench.TRAFFIC_FILE))
    assert rec["dram_bytes_per_launch"] > 0 and len(rec["kernel_source_sha"]) == 16


def test_burst_peak_for_short_regions_sustained_for_long_ones():
    p = ({"bf16_tflops": 1938.1, "bf16_tflops_sustained": 1730.8}, "measured")
    peak, label = bench.bf16_peak_for(0.027, p)
    assert peak == 1938.1 and "burst" in label and "0.027" in label
    peak, label = bench.bf16_peak_for(4.0, p)
    assert peak == 1730.8 and "sustained" in label


def test_clock_summary_keeps_samples_inside_the_windows():
    c = bench.ClockSampler(0)
    c.source = "test"
    # (t, sm_mhz, max_mhz, power_w, reasons)
    c.samples = [(0.0, 2070.0, 2070.0, 150.0, 0x1), (1.0, 1500.0, 2070.0, 1300.0, 0x4),
                 (1.5, 1600.0, 2070.0, 1350.0, 0x4), (2.0, 1700.0, 2070.0, 1200.0, 0x0), (9.0, 2070.0, 2070.0, 140.0, 0)]
    s = c.summary([(0.9, 2.1)])
    assert s["sm_mhz"] == 1600.0 and s["samples_under_load"] == 3 and s["samples"] == 5
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2070.0
    assert c.summary()["samples_under_load"] == 5


@pytest.fixture
def small_step(monkeypatch):
    """bench's step inputs at 64 x 64 x 64 (same generators and seeds, smaller SIZE)."""
    monkeypatch.setattr(bench, "SIZE", 64)
    oracle.build()
    g = si.generator(1)
    f8 = si.fp8_case(64, 64, 64, seed=3)
    return {"A": si.normal((64, 64), g), "B": si.normal((64, 64), g, std=0.02), "A8": f8["A"], "B8": f8["B"],
            "bias": f8["bias"], "sa": torch.tensor([f8["sa"]]), "sb": torch.tensor([f8["sb"]]),
            "Asp": si.normal((64, 64), g), "Bsp": si.normal((64, 64), g)}


def _rounded_outputs(o, r):
    """What a correct GPU would return for rows 0..r-1: the oracle's values rounded to bf16."""
    _, out = o.last
    gpu = {k: torch.from_numpy(out[k][0].reshape(r, 64)).to(torch.bfloat16) for k in ("D", "D8", "Dsp")}
    gpu["Ac"] = si.from_codes(out["Ac"], "bf16")
    gpu["meta"] = torch.from_numpy(out["meta"].view(np.int32).copy())
    return gpu


def test_oracle_check_accepts_correct_rows_and_rejects_a_wrong_one(small_step):
    o = bench.OracleSample(small_step)
    dense, total = o.rows(8)
    assert dense == 2 * 2.0 * 8 * 64 * 64 and total == 3 * 2.0 * 8 * 64 * 64
    gpu = _rounded_outputs(o, 8)
    res = o.check(gpu)
    assert res["ok"] and res["rows"] == 8 and res["sp24_compress_bit_exact"]
    assert max(res["bf16_dense"], res["e4m3_scaled_bias"], res["sp24_gemm_bf16"]) <= 1.0
    gpu["D8"][3, 5] += 1.0  # one wrong output
    assert not o.check(gpu)["ok"]
    gpu = _rounded_outputs(o, 8)
    gpu["meta"][0, 0] ^= 1  # one wrong metadata bit
    assert not o.check(gpu)["sp24_compress_bit_exact"]
