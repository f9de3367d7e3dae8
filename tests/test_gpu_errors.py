"""Error paths of the C ABI on a GPU: every bad call returns its code and a
message before anything is enqueued, and the handle stays usable.  Failures
are made on the host (bad arguments, an injected allocation failure); nothing
here faults the GPU."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import synth  # noqa: E402
from gpu_harness import DeviceRun  # noqa: E402
from sparse_communication_distributed_gb300 import MASK, STEP, THETA, Scape, ScapeError  # noqa: E402
from sparse_communication_distributed_gb300.scape import (SCAPE_EINVAL, SCAPE_ENOMEM,  # noqa: E402
                                                          SCAPE_ESTATE)

pytestmark = pytest.mark.gpu


def test_injected_allocation_failure_leaks_nothing(monkeypatch):
    wl = synth.tiny(1 << 22, 4, 65536, 0.01)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for n in (1, 5, 9):
        monkeypatch.setenv("SCAPE_TEST_FAIL_ALLOC", str(n))
        with pytest.raises(ScapeError) as ei:
            Scape.for_workload(wl, 0.01)
        assert ei.value.code == SCAPE_ENOMEM
    monkeypatch.delenv("SCAPE_TEST_FAIL_ALLOC")
    free1, _ = torch.cuda.mem_get_info()
    assert abs(free1 - free0) < (64 << 20)
    sc = Scape.for_workload(wl, 0.01)  # a normal create still works
    sc.close()


def test_calls_before_the_first_step():
    wl = synth.tiny(8192, 2, 1024, 0.1)
    sc = Scape.for_workload(wl, 0.1)
    with pytest.raises(ScapeError) as ei:
        sc.mask()
    assert ei.value.code == SCAPE_ESTATE
    with pytest.raises(ScapeError) as ei:
        sc.sparse(0)
    assert ei.value.code == SCAPE_ESTATE
    with pytest.raises(ScapeError) as ei:
        sc.mask_stats()
    assert ei.value.code == SCAPE_ESTATE
    sc.close()


def test_bad_step_arguments_leave_the_handle_usable():
    wl = synth.tiny(8192, 2, 1024, 0.1)
    g = DeviceRun(wl, 0.1)
    try:
        buf = torch.empty(wl.N + 8, dtype=torch.int16, device="cuda")
        with pytest.raises(ScapeError) as ei:
            g.sc.step([buf[1:], buf[1:]])  # 2-byte offset: not 16-byte aligned
        assert ei.value.code == SCAPE_EINVAL and "aligned" in str(ei.value)
        assert int(g.sc.read(STEP)[0]) == 0
        with pytest.raises(ScapeError) as ei:
            g.sc.read(THETA, offset=wl.N - 10, count=11)
        assert ei.value.code == SCAPE_EINVAL
        g.step()  # still works
        assert int(g.sc.read(STEP)[0]) == 1
    finally:
        g.close()


def test_mask_load_is_validated_and_used():
    wl = synth.tiny(4096 + 64, 2, 1024, 0.05)  # k = 51 per full chunk, 3 in the last
    g = DeviceRun(wl, 0.05)
    try:
        words = np.zeros(g.sc.info["mask_words"], np.uint32)
        with pytest.raises(ScapeError) as ei:
            g.sc.load(MASK, words)  # no bits at all
        assert ei.value.code == SCAPE_EINVAL and "bits" in str(ei.value)
        bits = np.zeros(wl.N, np.uint8)
        for c0, k in ((0, 51), (1024, 51), (2048, 51), (3072, 51), (4096, 3)):
            bits[c0 + np.arange(k) * 7 % 1024 if c0 < 4096 else c0 + np.arange(k)] = 1
        packed = np.packbits(bits.reshape(-1, 32), axis=1, bitorder="little").view("<u4").ravel()
        bad = packed.copy()
        bad[-1] |= np.uint32(1 << 20)  # a 4th bit in the last chunk (k = 3)
        with pytest.raises(ScapeError):
            g.sc.load(MASK, bad)
        g.sc.load(MASK, packed)
        g.step()  # applies the loaded mask: no step-0 selection
        idx, _ = g.sc.sparse(-1)
        assert np.array_equal(idx, np.nonzero(bits)[0].astype(np.uint32))
    finally:
        g.close()
