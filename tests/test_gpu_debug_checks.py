"""The debug build of libscape (SCAPE_DEBUG_CHECKS): on valid input it gives
the release build's results bit for bit and records no failed check; fed a
mask whose chunks carry the wrong bit counts (one bit moved between two
middle chunks, so even an unchecked access would stay inside its buffer) it
records the failure instead of writing past a chunk's compact slots.
The corrupt mask is loaded with the test hook SCAPE_TEST_SKIP_MASK_CHECK."""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import types  # noqa: E402

import synth  # noqa: E402
from gpu_harness import OracleRun, compare, sample_chunks  # noqa: E402
from sparse_communication_distributed_gb300 import MASK, THETA, U, V, Scape  # noqa: E402
from sparse_communication_distributed_gb300 import build as pkg_build  # noqa: E402
from sparse_communication_distributed_gb300.scape import DEBUG_LIB_PATH  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def debug_lib():
    if not os.path.exists(DEBUG_LIB_PATH):
        pkg_build.build(debug_checks=True)
    return DEBUG_LIB_PATH


def _run(wl, density, lib_path, steps=3, mask=None):
    sc = Scape.for_workload(wl, density, lib_path=lib_path)
    dev = torch.device("cuda")
    th = torch.empty(wl.N, dtype=torch.float32, device=dev)
    synth.gpu().theta_into(wl, th)
    torch.cuda.synchronize()
    sc.load(THETA, th)
    if mask is not None:
        sc.load(MASK, mask)
    grads = [torch.empty(wl.N, dtype=torch.int16, device=dev) for _ in range(wl.W)]
    for t in range(steps):
        for w in range(wl.W):
            synth.gpu().grads_into(wl, w, t, grads[w])
        sc.step(grads)
    torch.cuda.synchronize()
    return sc


def test_debug_build_matches_release_and_records_nothing(debug_lib):
    wl = synth.tiny(5 * 4096 + 160, 3, 4096, 0.05, seed=81)
    from sparse_communication_distributed_gb300.scape import LIB_PATH
    rel = _run(wl, 0.05, LIB_PATH)
    dbg = _run(wl, 0.05, debug_lib)
    try:
        info = dbg._info()
        assert info["checks_compiled"] == 1 and info["check_count"] == 0
        assert rel._info()["checks_compiled"] == 0
        for f in (THETA, V, MASK):
            assert np.array_equal(dbg.read(f).view(np.uint32), rel.read(f).view(np.uint32))
        for w in range(wl.W):
            assert np.array_equal(dbg.read(U, w).view(np.uint32), rel.read(U, w).view(np.uint32))
    finally:
        rel.close()
        dbg.close()


def test_debug_build_records_a_corrupt_mask(debug_lib, monkeypatch):
    wl = synth.tiny(6 * 4096, 3, 4096, 0.05, seed=82)  # k = 204 per chunk
    bits = np.zeros(wl.N, np.uint8)
    for c in range(6):
        bits[c * 4096 + np.arange(204) * 17 % 4096] = 1
    # move one kept coordinate from chunk 1 to chunk 2: 203 and 205 bits
    one = np.nonzero(bits[4096:8192])[0][0]
    bits[4096 + one] = 0
    free = np.nonzero(bits[8192:12288] == 0)[0][0]
    bits[8192 + free] = 1
    assert bits.sum() == 6 * 204
    words = np.packbits(bits.reshape(-1, 32), axis=1, bitorder="little").view("<u4").ravel()
    monkeypatch.setenv("SCAPE_TEST_SKIP_MASK_CHECK", "1")
    sc = _run(wl, 0.05, debug_lib, steps=1, mask=words)
    try:
        info = sc._info()
        assert info["check_count"] > 0
        assert info["check_code"] in (1, 2, 3, 4, 5)
        assert 8192 <= info["check_where"] < 12288  # the chunk with one bit too many
    finally:
        sc.close()


def test_debug_build_full_size_records_nothing(debug_lib):
    # every guarded index at the benchmark layout's full size (1.8B
    # coordinates, 27091 chunks): no check fails, and the sampled chunks still
    # match the oracle bit for bit
    wl = synth.WORKLOADS["llama-1.8b-w4"]
    ids = sample_chunks(wl)
    sc = _run(wl, 0.01, debug_lib, steps=2)
    r = OracleRun(wl, 0.01, chunk_ids=ids)
    try:
        info = sc._info()
        assert info["checks_compiled"] == 1 and info["check_count"] == 0, info
        for _ in range(2):
            r.step()
        compare(types.SimpleNamespace(sc=sc, wl=wl), r, "debug build, after step 1")
    finally:
        sc.close()
        torch.cuda.empty_cache()

