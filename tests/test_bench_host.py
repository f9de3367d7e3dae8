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
    (prof / "ncu_traffic.txt").write_text(f"# header\nstep_chunks some-case 80.0 {h}\n"
                                          f"step_chunks the-bench 81.0 {h}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    t, where = bench.ncu_traffic("step_chunks", 1000)
    assert t == 80_000.0 and "some-case" in where
    t, where = bench.ncu_traffic("step_chunks", 1000, "the-bench")  # a capture of the workload itself
    assert t == 81_000.0 and "itself" in where
    t, where = bench.ncu_traffic("step_chunks", 1000, "another")
    assert t == 80_000.0 and "scaled" in where
    (src / "k_fused.cu").write_text("kernel source B\n")  # the kernel changed since the capture
    assert bench.ncu_traffic("step_chunks", 1000) == (None, None)
    assert bench.ncu_traffic("other_kernel", 1000) == (None, None)


def test_l2_flush_rule():
    l2 = 126 << 20
    assert bench.needs_l2_flush(61 << 20, l2)          # the 2^20 layout: flushed
    assert not bench.needs_l2_flush(3 << 30, l2)       # the 2^25 profiling case: not
    assert not bench.needs_l2_flush(100 << 30, l2)     # the 1.8B layout: not


def test_baseline_sample_size():
    # large layout: 13 timed steps over as many chunks as the work allows
    assert bench.baseline_sample_size(1_775_372_288, 65536, 4) == (187, 13)
    assert bench.baseline_sample_size(557_774_080, 65536, 8) == (93, 13)
    # small layout: every chunk, more steps
    assert bench.baseline_sample_size(1 << 20, 4096, 4) == (256, 152)
    # never below 13 steps or one chunk
    assert bench.baseline_sample_size(1 << 20, 4096, 4, work=1.0) == (1, 13)


@pytest.mark.parametrize("name,density,K", [
    ("flat-2^20-w4", 0.10, 104_704), ("flat-2^26-w8-ties", 0.01, 670_720),
    ("gpt2-medium-w8", 0.01, 3_546_282), ("llama-500m-w8", 0.10, 55_772_302),
    ("llama-1.8b-w4", 0.01, 17_743_970)])
def test_static_K_matches_the_tabulated_counts(name, density, K):
    assert bench.static_K(bench.synth.WORKLOADS[name], density) == K


def test_line_config_is_the_same_on_both_arms():
    import types
    args = types.SimpleNamespace(per_tensor=False, residual_host=False, union_mask=False)
    wl = bench.synth.WORKLOADS["llama-1.8b-w4"]
    c = bench.line_config(wl, 0.01, args, 1)
    assert c["K"] == 17_743_970 and c["l2"].startswith("no flush")
    assert bench.line_config(wl, 0.01, args, 1) == c
    small = bench.line_config(bench.synth.WORKLOADS["flat-2^20-w4"], 0.1, args, 1)
    assert small["l2"].startswith("flushed before every timed step")


def test_sweep_rows_cover_every_config_and_density():
    rows = {(n, d) for n, d in bench.SWEEP}
    for name in ("flat-2^20-w4", "flat-2^26-w8-ties", "gpt2-medium-w8", "llama-500m-w8",
                 "llama-1.8b-w4"):
        for d in bench.synth.WORKLOADS[name].densities:
            assert (name, d) in rows
    assert len(rows) == 7
    # timed steps: at least the requested count, enough for 400 ms, capped
    assert bench.sweep_steps(20, 23.6) == 20
    assert bench.sweep_steps(20, 1.7) == 236
    assert bench.sweep_steps(20, 0.03) == 5000


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

