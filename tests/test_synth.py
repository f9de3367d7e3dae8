"""The seeded input generator on the CPU: its log against libm, the normal
deviates' moments, bf16 rounding, determinism, and the workload layouts."""
import math

import numpy as np

import synth


def test_series_log_matches_libm():
    c = synth.cpu()
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.uniform(1e-7, 1.0, 2000), 10.0 ** -rng.uniform(0, 30, 200)])
    for x in xs.astype(np.float32):
        if x <= 0 or x >= 1:
            continue
        ref = math.log(float(x))
        assert abs(c.logf(float(x)) - ref) <= 4e-7 * abs(ref) + 1e-7


def test_normals_moments():
    z = synth.cpu().normals(7, 2, 0, 0, 0, 1 << 20).astype(np.float64)
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1) < 5e-3
    assert abs(((z - z.mean()) ** 4).mean() / z.var() ** 2 - 3) < 0.05
    assert abs(np.mean(np.abs(z) > 1.959964) - 0.05) < 2e-3


def test_grads_bf16_and_deterministic():
    wl = synth.WORKLOADS["flat-2^20-w4"]
    c = synth.cpu()
    g1 = c.grads(wl, 1, 3, i0=1000, n=5000)
    g2 = c.grads(wl, 1, 3, idx=np.arange(1000, 6000))
    assert np.array_equal(g1, g2)
    assert not np.array_equal(g1, c.grads(wl, 2, 3, i0=1000, n=5000))
    f = (g1.astype(np.uint32) << 16).view(np.float32)
    assert abs(f.std() - 1e-3 * math.sqrt(1.25)) < 1e-4


def test_student_t_grid_and_ties():
    wl = synth.WORKLOADS["flat-2^26-w8-ties"]
    g = synth.cpu().grads(wl, 0, 0, n=65536)
    f = (g.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.all(f * 16384 == np.round(f * 16384))  # multiples of 2^-14
    assert np.unique(np.abs(f)).size < 400  # 65536 values on a few hundred levels


def test_layout_sizes():
    assert synth.WORKLOADS["gpt2-medium-w8"].N == 354_823_168
    assert len(synth.WORKLOADS["gpt2-medium-w8"].tensors) == 292
    assert synth.WORKLOADS["llama-500m-w8"].N == 557_774_080
    assert len(synth.WORKLOADS["llama-500m-w8"].tensors) == 219
    assert synth.WORKLOADS["llama-1.8b-w4"].N == 1_775_372_288
    assert len(synth.WORKLOADS["llama-1.8b-w4"].tensors) == 291
    s = synth.WORKLOADS["gpt2-medium-w8"].sigmas()
    assert s[0] == np.float32(0.02 / 32)  # wte: fan_in 1024
