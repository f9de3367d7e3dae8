"""scape_step_noalloc: the step on caller-owned buffers, with its scratch in a
static device array instead of memory from cudaMalloc.  It is meant for callers
whose device memory belongs to another allocator, or that must not allocate in
their step loop.  This file sorts last so that a run stopping at its first
failure has already run every other test.

The check: three steps in a row through the C ABI give the same state, masks
and compact buffers as scape_step on a handle and as the oracle (within the
parity tolerance, and bit for bit).  The first step either has every key of a
chunk tied (so the standalone select redoes the selection) or takes generic
gradients (so the step-0 mask comes from the standalone select here but from
the fused kernel's boot launch on the handle); u and e rows use the smallest
row stride the header allows or a padded one.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_harness import OracleRun, assert_close_exact  # noqa: E402
from sparse_communication_distributed_gb300 import E, THETA, U, V, Scape  # noqa: E402
from sparse_communication_distributed_gb300.scape import ScapeError, step_noalloc  # noqa: E402

pytestmark = pytest.mark.gpu


def _tied_bits() -> int:
    return int(np.float32(0.001).view(np.uint32) >> 16)


@pytest.mark.parametrize("first", ["tied", "generic"])
@pytest.mark.parametrize("stride_kind", ["smallest", "padded"])
def test_noalloc_step_matches_handle_and_oracle(first, stride_kind):
    wl = synth.tiny(3 * 4096 + 102, 3, 4096, 0.05, kind=synth.SYN_STUDENT_Q, seed=12)
    density = 0.05
    N, W = wl.N, wl.W
    dev = torch.device("cuda")
    sc = Scape.for_workload(wl, density)
    r = OracleRun(wl, density)
    K, words = sc.K, sc.info["mask_words"]
    theta0 = synth.cpu().theta0(wl, np.arange(N))
    sc.load(THETA, theta0)

    stride = (N + 3) // 4 * 4 if stride_kind == "smallest" else (N + 255) // 256 * 256
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

    try:
        for t in range(3):
            if t == 0 and first == "tied":  # every key of a chunk equal: the candidate list overflows
                host = np.full((W, N), _tied_bits(), np.uint16)
                for w in range(W):
                    grads[w].copy_(torch.from_numpy(host[w].view(np.int16)))
            else:
                for w in range(W):
                    synth.gpu().grads_into(wl, w, t, grads[w])
                host = r.grads(t)
            sc.step(grads)
            buf["mask_prev"], buf["mask_next"] = masks[t % 2], masks[(t + 1) % 2]
            step_noalloc(wl.numel, wl.chunk, W, density, hyper, buf, grads, first_step=(t == 0))
            r.step(host)
            torch.cuda.synchronize()

            o = r.o
            for name, got, hnd, ref in (
                    ("theta", buf["theta"], sc.read(THETA), o.get(oracle.THETA)),
                    ("v", buf["v"], sc.read(V), o.get(oracle.V))):
                got = got.cpu().numpy()
                assert_close_exact(f"{name} step {t} (handle)", got, hnd)
                assert_close_exact(f"{name} step {t} (oracle)", got, ref)
            oidx, _ = o.sparse(0)
            assert oidx.size == K
            for w in range(W):
                row = slice(w * stride, w * stride + N)
                for name, f, of in (("u", U, oracle.U), ("e", E, oracle.E)):
                    got = buf[name][row].cpu().numpy()
                    assert_close_exact(f"{name}[{w}] step {t} (handle)", got, sc.read(f, w))
                    assert_close_exact(f"{name}[{w}] step {t} (oracle)", got, o.get(of, w))
                got = buf["vals"][w * K:(w + 1) * K].cpu().numpy()
                assert_close_exact(f"vals[{w}] step {t} (handle)", got, sc.sparse(w)[1])
                assert_close_exact(f"vals[{w}] step {t} (oracle)", got, o.sparse(w)[1])
            got = buf["bbar"].cpu().numpy()
            hidx, hbbar = sc.sparse(-1)
            assert_close_exact(f"bbar step {t} (handle)", got, hbbar)
            assert_close_exact(f"bbar step {t} (oracle)", got, o.sparse(-1)[1])
            gidx = buf["idx"].cpu().numpy().view(np.uint32)
            assert np.array_equal(gidx, hidx), f"idx step {t} (handle)"
            assert np.array_equal(gidx.astype(np.uint64), oidx), f"idx step {t} (oracle)"
            gmask = buf["mask_next"].cpu().numpy().view(np.uint32)
            assert np.array_equal(gmask, sc.mask()), f"mask step {t} (handle)"
            assert np.array_equal(gmask, oracle.pack_bits(o.mask(0))), f"mask step {t} (oracle)"
            if t == 0 and first == "tied":
                assert sc._info()["select_fallbacks"] > 0  # the fallback path ran
    finally:
        sc.close()


def test_noalloc_rejects_too_many_chunks():
    dev = torch.device("cuda")
    z = torch.zeros(64, dtype=torch.float32, device=dev)
    buf = {k: z for k in ("theta", "v", "u", "e", "mask_prev", "vals", "bbar", "idx")}
    buf["mask_next"] = torch.zeros(64, dtype=torch.float32, device=dev)
    buf["row_stride"] = 65537 * 32
    buf["vals_stride"] = 1 << 30
    with pytest.raises(ScapeError, match="chunks exceed"):
        step_noalloc([65537 * 32], 32, 1, 0.5, (0.9, 0.95, 1e-3, 0.1, 1e-8), buf, [z],
                     first_step=True)


def test_noalloc_rejects_host_buffers_and_wrong_grad_count():
    # a page-locked host buffer in place of theta, or as a gradient: rejected
    # before anything is enqueued
    dev = torch.device("cuda")
    N, W = 1024, 2
    d = {k: torch.zeros(N, dtype=torch.float32, device=dev)
         for k in ("theta", "v", "vals", "bbar", "idx", "mask_prev", "mask_next")}
    d["u"] = torch.zeros(W * N, dtype=torch.float32, device=dev)
    d["e"] = torch.zeros(W * N, dtype=torch.float32, device=dev)
    d["row_stride"], d["vals_stride"] = N, N
    grads = [torch.zeros(N, dtype=torch.int16, device=dev) for _ in range(W)]
    hyper = (0.9, 0.95, 1e-3, 0.1, 1e-8)
    bad = dict(d, theta=torch.zeros(N, dtype=torch.float32).pin_memory())
    with pytest.raises(ScapeError, match="theta must be device memory"):
        step_noalloc([N], 1024, W, 0.1, hyper, bad, grads, first_step=True)
    host_g = [grads[0], torch.zeros(N, dtype=torch.int16).pin_memory()]
    with pytest.raises(ScapeError, match=r"grad_ptrs\[1\] must be device memory"):
        step_noalloc([N], 1024, W, 0.1, hyper, d, host_g, first_step=True)
    with pytest.raises(ValueError, match="gradient buffers"):
        step_noalloc([N], 1024, W, 0.1, hyper, d, grads[:1], first_step=True)
    torch.cuda.synchronize()
