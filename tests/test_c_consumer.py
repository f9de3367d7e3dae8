"""libscape from a plain C99 program (tests/c/scape_c_consumer.c): it includes
only include/scape.h, links only libscape.so and hands the library host
pointers, with no Python binding in between.  Without a GPU it checks the
argument errors; on a GPU it steps a small layout from host gradients and its
parameters, mask and synchronized buffer match the oracle bit for bit."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import synth
from sparse_communication_distributed_gb300 import build, scape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "scape_c_consumer.c")


@pytest.fixture(scope="module")
def consumer(tmp_path_factory):
    if not os.path.exists(scape.LIB_PATH):
        build.build()
    exe = str(tmp_path_factory.mktemp("c") / "scape_c_consumer")
    libdir = os.path.dirname(scape.LIB_PATH)
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           SRC, "-L", libdir, "-lscape", f"-Wl,-rpath,{libdir}", "-lm", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_consumer_argument_errors(consumer):
    r = subprocess.run([consumer, "args"], capture_output=True, text=True)
    assert r.returncode == 0 and "args ok" in r.stdout, r.stdout + r.stderr


@pytest.mark.gpu
def test_c_consumer_matches_oracle(consumer, tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    N, W, C, density, steps = 3 * 4096 + 1000, 3, 4096, 0.05, 4
    wl = synth.tiny(N, W, C, density, kind=synth.SYN_STUDENT_Q, seed=23)
    o = oracle.Oracle.for_workload(wl, density)
    theta0 = synth.cpu().theta0(wl, o.index)
    o.set(oracle.THETA, theta0)
    grads = np.stack([np.stack([synth.cpu().grads(wl, w, t, n=N) for w in range(W)])
                      for t in range(steps)])
    theta0.tofile(tmp_path / "theta.bin")
    grads.astype(np.uint16).tofile(tmp_path / "grads.bin")
    for t in range(steps):
        o.step(grads[t])
    r = subprocess.run([consumer, "run", str(N), str(W), str(C), repr(density), str(steps),
                        str(tmp_path)], capture_output=True, text=True)
    assert r.returncode == 0 and "run ok" in r.stdout, r.stdout + r.stderr
    th = np.fromfile(tmp_path / "out_theta.bin", np.float32)
    assert np.array_equal(th.view(np.uint32), o.get(oracle.THETA).view(np.uint32))
    mask = np.fromfile(tmp_path / "out_mask.bin", np.uint32)
    assert np.array_equal(mask, oracle.pack_bits(o.mask(0)))
    bbar = np.fromfile(tmp_path / "out_bbar.bin", np.float32)
    assert np.array_equal(bbar.view(np.uint32), o.sparse(-1)[1].view(np.uint32))
