"""Round trip of the compact buffers: what the step packs (coordinates and
values of b_w, and bbar) scatters back with scape_unpack into exactly the
oracle's dense sparse buffers (b_w = a_w on the applied mask, +0 elsewhere)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_harness import DeviceRun, OracleRun, assert_close_exact  # noqa: E402
from sparse_communication_distributed_gb300.scape import unpack  # noqa: E402

pytestmark = pytest.mark.gpu


def test_pack_unpack_round_trip():
    wl = synth.tiny(5 * 4096 + 160, 3, 4096, 0.07, seed=71)
    g, r = DeviceRun(wl, 0.07), OracleRun(wl, 0.07)
    dev = torch.device("cuda")
    try:
        for t in range(3):
            g.step()
            r.step()
            bad = torch.zeros(1, dtype=torch.int32, device=dev)
            for w in range(wl.W):
                idx, vals = g.sc.sparse(w)
                dense = torch.zeros(wl.N, dtype=torch.float32, device=dev)
                unpack(torch.from_numpy(idx.view(np.int32)).to(dev), torch.from_numpy(vals).to(dev),
                       dense, bad)
                assert_close_exact(f"b[{w}] step {t}", dense.cpu().numpy(), r.o.get(oracle.B, w))
            idx, bb = g.sc.sparse(-1)
            dense = torch.zeros(wl.N, dtype=torch.float32, device=dev)
            unpack(torch.from_numpy(idx.view(np.int32)).to(dev), torch.from_numpy(bb).to(dev), dense)
            ref = np.zeros(wl.N, np.float32)
            oidx, ob = r.o.sparse(-1)
            ref[oidx.astype(np.int64)] = ob
            assert_close_exact(f"bbar step {t}", dense.cpu().numpy(), ref)
            assert int(bad.item()) == 0
        # an out-of-range coordinate is skipped and counted
        dense = torch.zeros(16, dtype=torch.float32, device=dev)
        unpack(torch.tensor([3, 99, 5], dtype=torch.int32, device=dev),
               torch.tensor([1.0, 2.0, 3.0], device=dev), dense, bad)
        assert dense.cpu().numpy()[[3, 5]].tolist() == [1.0, 3.0] and int(bad.item()) == 1
    finally:
        g.close()
