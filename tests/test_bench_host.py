"""Host-side arithmetic of bench.py (no GPU): the algorithmic bytes against
independently computed per-configuration figures, the traffic lookup's source
check, the L2-flush rule and the CPU-baseline sample size."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

# (N, W, K, algorithmic GB per step) of the five benchmark configurations,
# worked out by hand from the layouts' tensor sizes and the bytes each
# coordinate and each kept value move, independently of this code, and
# rounded to three significant figures.
CONFIGS = [
    (1 << 20, 4, 104_704, 0.097),
    (1 << 26, 8, 6_710_272, 11.30),
    (1 << 26, 8, 670_720, 10.86),
    (354_823_168, 8, 3_546_282, 57.4),
    (557_774_080, 8, 5_574_677, 90.3),
    (557_774_080, 8, 55_772_302, 93.9),
    (1_775_372_288, 4, 17_743_970, 158.1),
]


@pytest.mark.parametrize("N,W,K,gb", CONFIGS)
def test_algorithmic_bytes_match_the_tabulated_figures(N, W, K, gb):
    got = bench.alg_bytes(N, W, K)["step"] / 1e9
    assert abs(got - gb) <= 0.051 * max(1.0, gb / 10), (got, gb)


def test_traffic_lookup_needs_the_captured_source(tmp_path, monkeypatch):
    src = tmp_path / "sparse_communication_distributed_gb300" / "csrc"
    src.mkdir(parents=True)
    (src / "k_fused.cu").write_text("kernel source A\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    import hashlib
    h = hashlib.sha256(b"kernel source A\n").hexdigest()[:16]
    (prof / "ncu_traffic.txt").write_text(f"# header\nstep_chunks some-case 80.0 {h}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    t, where = bench.ncu_traffic("step_chunks", 1000)
    assert t == 80_000.0 and "some-case" in where
    (src / "k_fused.cu").write_text("kernel source B\n")  # the kernel changed since the capture
    assert bench.ncu_traffic("step_chunks", 1000) == (None, None)
    assert bench.ncu_traffic("other_kernel", 1000) == (None, None)


def test_l2_flush_rule():
    l2 = 126 << 20
    assert bench.needs_l2_flush(61 << 20, l2)          # the 2^20 layout: flushed
    assert not bench.needs_l2_flush(3 << 30, l2)       # the 2^25 profiling case: not
    assert not bench.needs_l2_flush(100 << 30, l2)     # the 1.8B layout: not


def test_baseline_sample_size():
    # large layout: 14 steps over as many chunks as the time allows
    assert bench.baseline_sample_size(1_775_372_288, 65536, 6.4e6, 15.0) == (104, 14)
    # small layout: every chunk, more steps
    assert bench.baseline_sample_size(1 << 20, 4096, 7.9e6, 15.0) == (256, 113)
    # never below 14 steps or one chunk
    assert bench.baseline_sample_size(1 << 20, 4096, 1.0, 15.0) == (1, 14)


def test_clock_parse_and_throttle_rule():
    lines = "\n".join([
        "2070, 2070, 900.1, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1100.5, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 1200.0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ])
    c = bench.ClockSampler.parse(lines)
    assert c["sm_mhz"] == 2070 and c["sm_max_mhz"] == 2070 and c["samples"] == 3
    assert c["reasons"] == ["sw_power_cap"]
    assert not (bench.THROTTLED & set(c["reasons"]))  # a power cap is only noted
    c = bench.ClockSampler.parse("1800, 2070, 1300, Active, Not Active, Not Active, Not Active")
    assert bench.THROTTLED & set(c["reasons"]) == {"hw_slowdown"}  # re-measured
    assert bench.ClockSampler.parse("") is None

