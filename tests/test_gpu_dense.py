"""scape_dense_adams_step (the dense AdamS comparator) against the oracle's
dense AdamS, element by element: a ragged small size on every coordinate and
the 1.8B layout at full size on sampled coordinate ranges."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_harness import assert_close_exact  # noqa: E402
from sparse_communication_distributed_gb300.scape import dense_adams_step  # noqa: E402

pytestmark = pytest.mark.gpu


def _run(wl, steps, ranges):
    dev = torch.device("cuda")
    N, W = wl.N, wl.W
    th = torch.empty(N, dtype=torch.float32, device=dev)
    synth.gpu().theta_into(wl, th)
    m = torch.zeros(N, dtype=torch.float32, device=dev)
    v = torch.zeros(N, dtype=torch.float32, device=dev)
    grads = [torch.empty(N, dtype=torch.int16, device=dev) for _ in range(W)]
    idx = np.concatenate([np.arange(a, b) for a, b in ranges]).astype(np.uint64)
    oth = synth.cpu().theta0(wl, idx)
    om = np.zeros(idx.size, np.float32)
    ov = np.zeros(idx.size, np.float32)
    hyper = dict(beta1=wl.beta1, beta2=wl.beta2, lr=wl.lr, wd=wl.wd, eps=wl.eps)
    for t in range(steps):
        for w in range(W):
            synth.gpu().grads_into(wl, w, t, grads[w])
        dense_adams_step(th, m, v, grads, **hyper)
        g = np.stack([synth.cpu().grads(wl, w, t, idx=idx) for w in range(W)])
        oracle.dense_adams_step(oth, om, ov, g, **hyper)
        torch.cuda.synchronize()
        sel = torch.from_numpy(idx.astype(np.int64)).to(dev)
        for name, gpu, ref in (("theta", th, oth), ("m", m, om), ("v", v, ov)):
            assert_close_exact(f"dense {name} step {t}", gpu[sel].cpu().numpy(), ref)


def test_dense_small_every_coordinate():
    wl = synth.tiny(100003, 3, 1024, 1.0, seed=41)
    _run(wl, 4, [(0, wl.N)])


def test_dense_full_size_sampled():
    wl = synth.WORKLOADS["llama-1.8b-w4"]
    N = wl.N
    ranges = [(0, 8192), (N // 3, N // 3 + 4096), (N // 2 + 7, N // 2 + 4103), (N - 8192, N)]
    _run(wl, 3, ranges)
