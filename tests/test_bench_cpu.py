"""Host logic of bench.py, without a GPU: which workloads flush L2 between
steps, the tie between committed ncu counters and the kernel sources, the
clock-sample parsing behind the "clocks" key, and the whole-job rate."""
import os
import tempfile

import pytest

import bench
from tiled_matrix_multiplication_output_gb300 import inputs


def test_l2_flush_rule_on_the_named_workloads():
    # A + B + C of the four smaller workloads fit in the 129 MB L2 (4096^3 FP16:
    # 96 MiB), so their steps run with L2 overwritten in between; 8192^3 BF16
    # (384 MiB) streams from HBM on its own.
    for name in ("worked_9x9", "square_128_f16", "edge_96x200x1000_bf16", "square_4096_f16"):
        assert bench.needs_flush(inputs.WORKLOADS[name]), name
    w = inputs.WORKLOADS["square_8192_bf16"]
    assert bench.footprint_bytes(w) == 3 * 8192 * 8192 * 2
    assert not bench.needs_flush(w)
    assert "flushed" in bench.config_of(inputs.WORKLOADS["square_128_f16"], "k")["l2"]
    assert bench.config_of(w, "k")["l2"] == "A+B+C larger than L2"


def test_committed_traffic_is_tied_to_the_kernel_sources(tmp_path, monkeypatch):
    # the committed summary of the benchmarked kernel counts only while its
    # digest is today's (a source change voids it until it is recaptured)
    path = os.path.join(bench.PROFILES, "tc_gemm_256x256_square_8192_bf16.md")
    current = f"`{bench.source_digest()}`" in open(path).read()
    got = bench.committed_traffic("tc_gemm_256x256", "square_8192_bf16")
    if current:
        assert isinstance(got, int) and got > 3 * 8192 * 8192 * 2 // 2
    else:
        assert got is None
    # a summary taken from other sources is ignored
    (tmp_path / "k_w.md").write_text("- dram_bytes_per_launch: 123\n- source_sha256: `00`\n")
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    assert bench.committed_traffic("k", "w") is None
    (tmp_path / "k_w.md").write_text(
        f"- dram_bytes_per_launch: 123\n- source_sha256: `{bench.source_digest()}`\n")
    assert bench.committed_traffic("k", "w") == 123
    assert bench.committed_traffic("k", "missing") is None


class _DoneProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler_with(rows):
    s = bench.ClockSampler(0)
    s.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    s.tmp.write("\n".join(rows) + "\n")
    s.tmp.flush()
    s.proc = _DoneProc()
    return s


def test_clock_sampler_parsing():
    not_active = "Not Active"
    rows = [
        # idx, sm, max, power, active mask, hw_slow, hw_thermal, sw_thermal, sw_power_cap
        f"0, 345, 2070, 150.0, 0x0, {not_active}, {not_active}, {not_active}, {not_active}",
        f"0, 1470, 2070, 1370.0, 0x4, {not_active}, {not_active}, {not_active}, Active",
        f"0, 1455, 2070, 1371.0, 0x4, {not_active}, {not_active}, {not_active}, Active",
        f"0, 1481, 2070, 1369.0, 0x4, {not_active}, {not_active}, {not_active}, Active",
        "garbage line",
    ]
    got = _sampler_with(rows).stop()
    # the idle sample (below half the highest clock) is left out of the median
    assert got == {"sm_mhz": 1470.0, "sm_max_mhz": 2070.0, "samples": 4,
                   "reasons": ["sw_power_cap"]}
    hot = _sampler_with([f"0, 900, 2070, 500.0, 0x40, Active, {not_active}, Active, {not_active}"])
    assert hot.stop()["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert _sampler_with(["nothing useful"]).stop() is None
    assert bench.ClockSampler(0).stop() is None   # never started (no nvidia-smi)


def test_job_rate_counts_every_rank():
    flops = 2.0 * 8192 ** 3
    one = bench.job_rate(flops, 10, 1, 6.5)
    assert one == pytest.approx(flops * 10 / 6.5e-3 / 1e12)
    # two replicas in the same (slowest-rank) time: twice the job's rate
    assert bench.job_rate(flops, 10, 2, 6.5) == pytest.approx(2 * one)


def test_reference_block_keeps_every_core_busy_within_the_step_budget():
    # 8192^3 at 2000 + 20 steps on 16 cores: 0.06 s per step, 27 us per entry
    rows, cols = bench.reference_block(8192, 8192, 16, 27e-6, 120.0 / 2020)
    assert rows == 16 and 1 <= cols < 8192
    assert cols * 27e-6 <= 120.0 / 2020
    # a generous budget widens to full rows, then adds rows by the thread count
    rows, cols = bench.reference_block(8192, 8192, 16, 27e-6, 2.0)
    assert cols == 8192 and rows % 16 == 0 and rows * 8192 * 27e-6 / 16 <= 2.0
    # never beyond C, never empty
    assert bench.reference_block(9, 9, 16, 1e-9, 100.0) == (9, 9)
    assert bench.reference_block(4, 3, 16, 10.0, 1e-3) == (4, 1)


def test_source_digest_covers_the_kernel_files():
    for name in bench.KERNEL_SOURCES:
        assert os.path.exists(os.path.join(bench.CSRC, name)), name
    assert len(bench.source_digest()) == 64


PEAKS = {"hbm_gbs": 6754.8, "bf16_tflops": 1957.5, "bf16_tflops_sustained": 1745.9,
         "sm_max_mhz": 2070.0}


def _flops(w):
    return 2.0 * w.M * w.N * w.K


@pytest.mark.parametrize("name, bound", [
    ("worked_9x9", "hbm"),               # 1.5 FLOP/B
    ("square_128_f16", "hbm"),           # 32 FLOP/B
    ("edge_96x200x1000_bf16", "hbm"),    # 57 FLOP/B
    ("square_4096_f16", "tensor"),       # 1365 FLOP/B, ridge about 290
    ("square_8192_bf16", "tensor"),      # 2731 FLOP/B
])
def test_roofline_bound_follows_arithmetic_intensity(name, bound):
    w = inputs.WORKLOADS[name]
    r = bench.roofline_of(w, _flops(w), 0.01, PEAKS, "measured", None)
    assert r["bound"] == bound
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    if bound == "hbm":
        assert r["unit"] == "GB/s" and r["peak"] == 6754.8
        assert r["achieved"] == pytest.approx(bench.footprint_bytes(w) / 1e-5 / 1e9)
    else:
        assert r["unit"] == "TFLOP/s" and r["peak"] == 1957.5
        assert r["achieved"] == pytest.approx(_flops(w) / 1e-5 / 1e12)
        assert r["frac_of_sustained"] == pytest.approx(r["achieved"] / 1745.9)


def test_roofline_fp32_compute_bound_is_the_fma_pipes():
    w = inputs.Workload("f32_4096", 4096, 4096, 4096, "f32", "f32", "normal", 0)
    r = bench.roofline_of(w, _flops(w), 3.0, PEAKS, "measured", None)
    assert r["bound"] == "alu"
    assert r["peak"] == pytest.approx(152 * 128 * 2 * 2070e6 / 1e12)


def test_roofline_carries_the_theoretical_tensor_peak():
    # 152 SMs x 8192 dense FLOP per cycle x 2070 MHz = 2577.7 TFLOP/s; at a
    # sampled 1485 MHz under the power cap, 1849.3
    w = inputs.WORKLOADS["square_8192_bf16"]
    r = bench.roofline_of(w, _flops(w), 0.6, PEAKS, "measured", None, sms=152, run_mhz=1485.0)
    assert r["theoretical_peak"] == pytest.approx(152 * 8192 * 2070e6 / 1e12)
    assert r["frac_of_theoretical"] == pytest.approx(r["achieved"] / r["theoretical_peak"])
    assert r["theoretical_peak_at_run_clock"] == pytest.approx(152 * 8192 * 1485e6 / 1e12)
    assert r["frac_of_theoretical_at_run_clock"] == pytest.approx(
        r["achieved"] / r["theoretical_peak_at_run_clock"])
    # the measured cuBLAS burst lies below the theoretical peak
    assert PEAKS["bf16_tflops"] < r["theoretical_peak"]
    # no sampled clock: no run-clock fraction; HBM-bound lines carry none of it
    assert "frac_of_theoretical_at_run_clock" not in bench.roofline_of(
        w, _flops(w), 0.6, PEAKS, "measured", None)
    small = inputs.WORKLOADS["square_128_f16"]
    assert "theoretical_peak" not in bench.roofline_of(small, _flops(small), 0.01, PEAKS,
                                                        "measured", None)


def test_trimmed_mean_drops_the_tails():
    assert bench.trimmed_mean([1.0] * 8 + [100.0, -50.0]) == pytest.approx(1.0)
    assert bench.trimmed_mean([2.0, 4.0]) == pytest.approx(3.0)


def test_parse_sweep_shapes():
    assert bench.parse_sweep_shapes("") == list(bench.SMALL_SWEEP_SHAPES)
    assert bench.parse_sweep_shapes("256x128x64, 8X8X8") == [("bf16", "bf16", 256, 128, 64),
                                                            ("bf16", "bf16", 8, 8, 8)]
    for bad in ("256x128", "0x8x8", "8x8x-1", "axbxc", "8x8x8,"):
        with pytest.raises(ValueError):
            bench.parse_sweep_shapes(bad)
