"""scape_mask_stats against the oracle: mask size, overlap of consecutive masks,
and the union of every worker's own top-k over all chunks (the fill-in the
partitioned rule avoids), exact counts."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_harness import DeviceRun, OracleRun, compare  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("W,kind", [(3, synth.SYN_GAUSS), (4, synth.SYN_STUDENT_Q)])
def test_mask_stats_match_oracle(W, kind):
    wl = synth.tiny(6 * 1024 + 352, W, 1024, 0.1, kind=kind, seed=50 + W)
    g, r = DeviceRun(wl, 0.1), OracleRun(wl, 0.1)
    try:
        for t in range(4):
            g.step()
            r.step()
            compare(g, r, f"step {t}")
            st = g.sc.mask_stats()
            o = r.o
            m_new, m_used = o.mask(0).astype(bool), o.mask(1).astype(bool)
            union = np.zeros(o.n, bool)
            for w in range(W):
                a = o.get(oracle.A, w)
                for j in range(o.chunk_start.size):
                    s, ln, k = int(o.chunk_start[j]), int(o.chunk_len[j]), int(o.chunk_k[j])
                    union[s:s + ln] |= oracle.topk(a[s:s + ln], k).astype(bool)
            assert st["kept"] == int(m_new.sum())
            assert st["overlap_prev"] == int((m_new & m_used).sum())
            assert st["union_global_topk"] == int(union.sum())
            assert st["union_global_topk"] >= st["kept"]
    finally:
        g.close()
