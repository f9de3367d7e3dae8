"""Stream-ordered mask read-back (scape_mask_async): each step's M_t read on a
second stream while later steps run, checked word for word against the
oracle's mask after that step."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_harness import DeviceRun, OracleRun  # noqa: E402
from sparse_communication_distributed_gb300.scape import MASK, ScapeError  # noqa: E402

pytestmark = pytest.mark.gpu

STEPS = 5


def _oracle_masks(wl, density, steps):
    r = OracleRun(wl, density)
    out = []
    for _ in range(steps):
        r.step()
        out.append(oracle.pack_bits(r.o.mask(0)))
    return out


@pytest.mark.parametrize("delay_reads", [False, True])
def test_async_reads_while_later_steps_run(delay_reads):
    # Steps go back to back on one stream; after each, M_t is read on a second
    # stream into its own page-locked buffer.  Every second step reuses the
    # mask buffer being read.  With the reads held back behind a bounded
    # device sleep, a step that did not wait for the read would overwrite the
    # mask first and an earlier buffer would hold a later mask.
    wl = synth.tiny(4 * 4096 + 96, 4, 4096, 0.05, seed=73)
    ref = _oracle_masks(wl, 0.05, STEPS)
    g = DeviceRun(wl, 0.05)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    nwords = g.sc.info["mask_words"]
    outs = [torch.full((nwords,), -1, dtype=torch.int32).pin_memory() for _ in range(STEPS)]
    try:
        torch.cuda.synchronize()
        if delay_reads:
            with torch.cuda.stream(s2):
                torch.cuda._sleep(20_000_000)  # about 10 ms at 2 GHz
        with torch.cuda.stream(s1):
            for t in range(STEPS):
                g.step()
                g.sc.mask_into_async(outs[t], s2)
        torch.cuda.synchronize()
        for t in range(STEPS):
            got = outs[t].numpy().view(np.uint32)
            if not np.array_equal(got, ref[t]):
                bad = np.nonzero(got != ref[t])[0]
                raise AssertionError(f"step {t}: {bad.size} words differ, first {bad[0]}")
        # the synchronous reader agrees with the last async read
        assert np.array_equal(g.sc.mask(), ref[-1])
    finally:
        g.close()


def test_async_read_then_load_and_step():
    # a pending async read, then a mask load (host waits for the read) and a
    # step on another stream (waits on the GPU): the read keeps the old mask
    wl = synth.tiny(3 * 4096, 3, 4096, 0.1, seed=74)
    ref = _oracle_masks(wl, 0.1, 2)
    g = DeviceRun(wl, 0.1)
    s2 = torch.cuda.Stream()
    nwords = g.sc.info["mask_words"]
    out = torch.full((nwords,), -1, dtype=torch.int32).pin_memory()
    try:
        g.step()
        with torch.cuda.stream(s2):
            torch.cuda._sleep(10_000_000)
        g.sc.mask_into_async(out, s2)
        g.sc.load(MASK, torch.from_numpy(ref[1].view(np.int32)).cuda())  # a valid mask
        torch.cuda.synchronize()
        assert np.array_equal(out.numpy().view(np.uint32), ref[0])
        assert np.array_equal(g.sc.mask(), ref[1])
    finally:
        g.close()


def test_async_read_before_first_step_is_an_error():
    wl = synth.tiny(4096, 2, 4096, 0.1, seed=75)
    g = DeviceRun(wl, 0.1, theta0=False)
    out = torch.empty(g.sc.info["mask_words"], dtype=torch.int32).pin_memory()
    try:
        with pytest.raises(ScapeError):
            g.sc.mask_into_async(out, torch.cuda.current_stream())
    finally:
        g.close()
