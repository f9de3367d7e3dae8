"""scape_step_noalloc: the step on caller-owned buffers, with its scratch in a
static device array instead of memory from cudaMalloc.  It is meant for callers
whose device memory belongs to another allocator, or that must not allocate in
their step loop.  This file sorts last so that a run stopping at its first
failure has already run every other test.

The check: two steps in a row through the C ABI give the same state, masks and
compact buffers as scape_step on a handle (within the parity tolerance, and bit
for bit), on inputs where the first step needs the standalone-select fallback
(all keys tied) and the second does not.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import synth  # noqa: E402
from gpu_harness import assert_close_exact  # noqa: E402
from sparse_communication_distributed_gb300 import E, THETA, U, V, Scape  # noqa: E402
from sparse_communication_distributed_gb300.scape import step_noalloc  # noqa: E402

pytestmark = pytest.mark.gpu


def test_noalloc_step_matches_handle_step():
    wl = synth.tiny(3 * 4096 + 100, 3, 4096, 0.05, kind=synth.SYN_STUDENT_Q, seed=12)
    density = 0.05
    N, W = wl.N, wl.W
    dev = torch.device("cuda")
    sc = Scape.for_workload(wl, density)
    K, words = sc.K, sc.info["mask_words"]
    theta0 = synth.cpu().theta0(wl, np.arange(N))
    sc.load(THETA, theta0)

    stride = (N + 255) // 256 * 256
    buf = {
        "theta": torch.from_numpy(theta0).to(dev),
        "v": torch.zeros(N, dtype=torch.float32, device=dev),
        "u": torch.zeros(W * stride, dtype=torch.float32, device=dev),
        "e": torch.zeros(W * stride, dtype=torch.float32, device=dev),
        "vals": torch.zeros(W * K, dtype=torch.float32, device=dev),
        "bbar": torch.zeros(K, dtype=torch.float32, device=dev),
        "idx": torch.zeros(K, dtype=torch.int32, device=dev),
        "row_stride": stride,
        "vals_stride": K,
    }
    masks = [torch.zeros(words, dtype=torch.int32, device=dev) for _ in range(2)]
    hyper = (wl.beta1, wl.beta2, wl.lr, wl.wd, wl.eps)
    grads = [torch.empty(N, dtype=torch.int16, device=dev) for _ in range(W)]

    for t in range(2):
        if t == 0:  # every key in a chunk equal: the on-chip candidate list overflows
            bits = int(np.float32(0.001).view(np.uint32) >> 16)
            for g in grads:
                g.fill_(bits if bits < 32768 else bits - 65536)
        else:
            for w in range(W):
                synth.gpu().grads_into(wl, w, t, grads[w])
        sc.step(grads)
        buf["mask_prev"], buf["mask_next"] = masks[t % 2], masks[(t + 1) % 2]
        step_noalloc(wl.numel, wl.chunk, W, density, hyper, buf, grads, first_step=(t == 0))
        torch.cuda.synchronize()

        assert_close_exact(f"theta step {t}", buf["theta"].cpu().numpy(), sc.read(THETA))
        assert_close_exact(f"v step {t}", buf["v"].cpu().numpy(), sc.read(V))
        for w in range(W):
            row = slice(w * stride, w * stride + N)
            assert_close_exact(f"u[{w}] step {t}", buf["u"][row].cpu().numpy(), sc.read(U, w))
            assert_close_exact(f"e[{w}] step {t}", buf["e"][row].cpu().numpy(), sc.read(E, w))
            _, vals = sc.sparse(w)
            assert_close_exact(f"vals[{w}] step {t}",
                               buf["vals"][w * K:(w + 1) * K].cpu().numpy(), vals)
        idx, bbar = sc.sparse(-1)
        assert_close_exact(f"bbar step {t}", buf["bbar"].cpu().numpy(), bbar)
        assert np.array_equal(buf["idx"].cpu().numpy().view(np.uint32), idx)
        assert np.array_equal(buf["mask_next"].cpu().numpy().view(np.uint32), sc.mask())
        if t == 0:
            assert sc._info()["select_fallbacks"] > 0  # the fallback path ran
    sc.close()


def test_noalloc_rejects_too_many_chunks():
    dev = torch.device("cuda")
    z = torch.zeros(64, dtype=torch.float32, device=dev)
    buf = {k: z for k in ("theta", "v", "u", "e", "mask_prev", "vals", "bbar", "idx")}
    buf["mask_next"] = torch.zeros(64, dtype=torch.float32, device=dev)
    buf["row_stride"] = 65537 * 32
    buf["vals_stride"] = 1 << 30
    from sparse_communication_distributed_gb300.scape import ScapeError
    with pytest.raises(ScapeError, match="chunks exceed"):
        step_noalloc([65537 * 32], 32, 1, 0.5, (0.9, 0.95, 1e-3, 0.1, 1e-8), buf, [z],
                     first_step=True)
