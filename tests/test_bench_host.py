"""Host-side pieces of bench.py that need no GPU: the recorded DRAM traffic of the
roofline kernel is read from its committed ncu summary only while the kernel source is
unchanged."""
import bench


def test_recorded_traffic_reads_the_committed_summary(tmp_path, monkeypatch):
    summary = tmp_path / "summary.md"
    summary.write_text("text\n\n- dram_bytes_per_launch = 1234\n- kernel_source_sha = "
                       + bench.kernel_source_sha() + "\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(summary))
    assert bench.recorded_traffic() == 1234.0


def test_recorded_traffic_is_null_once_the_kernel_changed(tmp_path, monkeypatch):
    summary = tmp_path / "summary.md"
    summary.write_text("- dram_bytes_per_launch = 1234\n- kernel_source_sha = 0000000000000000\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(summary))
    assert bench.recorded_traffic() is None

