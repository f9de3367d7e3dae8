"""libscape against the oracle, element by element, on the same seeded inputs.

- the 2^20 workload (W=4, density 0.10, chunk 4096, 5 steps) over every
  coordinate and every step;
- edge cases: ragged sizes (N not a multiple of 8, 32 or 256), the smallest
  chunk, W = 1 and odd W, density 1 and densities giving k = 0, all-equal
  accumulators, heavy ties in a 65536 chunk (more candidates than the
  shared-memory list holds), +-0;
- the full-size workloads in the launch configuration the bench times, on
  sampled whole chunks (both ends, every shard boundary, seeded others),
  plus properties over every chunk.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_harness import DeviceRun, OracleRun, check_full_mask, compare, sample_chunks  # noqa: E402
from sparse_communication_distributed_gb300 import E, MASK, STEP, THETA, U, V  # noqa: E402

pytestmark = pytest.mark.gpu


def _run_both(wl, density, steps, chunk_ids=None, every=True):
    g = DeviceRun(wl, density)
    r = OracleRun(wl, density, chunk_ids=chunk_ids)
    try:
        for t in range(steps):
            g.step()
            r.step()
            if every or t == steps - 1:
                compare(g, r, f"step {t}")
        check_full_mask(g)
    finally:
        g.close()


def test_flat_2p20_every_coordinate():
    wl = synth.WORKLOADS["flat-2^20-w4"]
    _run_both(wl, wl.densities[0], wl.steps)


@pytest.mark.parametrize("N,W,chunk,density", [
    (1000, 1, 32, 0.1),        # N % 8 != 0, k = 3, single worker
    (4099, 3, 96, 0.05),       # chunk not a power of two, ragged tail, odd W
    (70001, 5, 1024, 0.01),    # k = 10, last chunk 369 -> k = 3
    (3000, 2, 64, 0.01),       # k = 0 everywhere
    (2048 + 7, 4, 512, 1.0),   # density 1: every coordinate, dense AdamS
    (65536 * 2 + 160, 2, 65536, 0.3),  # large k in a full chunk, 160-coordinate last chunk
    (70001, 64, 1024, 0.05),   # the largest W
    (1, 1, 32, 1.0),           # one coordinate: one partial mask word, k = 1
    (31, 2, 32, 0.5),          # N below one word, two workers on one chunk
    (100, 7, 32, 0.25),        # 4 chunks, 7 workers: workers 4-6 own no chunk
    (65536 * 2, 2, 65536, 1.0),  # k = 65536: every coordinate of full-size chunks
    (16384 * 3 + 100, 3, 16384, 0.3),  # the largest chunk of the 512-thread shape
    (16416 * 2 + 50, 2, 16416, 0.05),  # the smallest chunk of the 1024-thread shape
])
def test_edge_shapes(N, W, chunk, density):
    wl = synth.tiny(N, W, chunk, density, seed=N)
    _run_both(wl, density, 4)


@pytest.mark.parametrize("chunk", [65536, 16384])
def test_heavy_ties_overflow_candidates(chunk):
    # Student-t means on a 2^-14 grid: |a| takes few hundred values, so the bin
    # holding the threshold exceeds the shared-memory candidate list (both
    # CTA shapes of the step kernel)
    wl = synth.tiny(chunk * 3, 3, chunk, 0.1, kind=synth.SYN_STUDENT_Q, seed=3)
    _run_both(wl, 0.1, 4)


def _const_grads(wl, value):
    bits = np.float32(value).view(np.uint32) >> 16
    return np.full((wl.W, wl.N), bits, np.uint16)


def test_all_equal_accumulators():
    # constant gradient: every |a| in a chunk is equal, the first k coordinates win
    wl = synth.tiny(8192 + 96, 2, 4096, 0.1)
    g, r = DeviceRun(wl, 0.1), OracleRun(wl, 0.1)
    try:
        for t in range(3):
            gr = _const_grads(wl, -0.0625)
            g.step(gr)
            r.step(gr)
            compare(g, r, f"step {t}")
            if t == 0:
                # the step-0 mask ranks equal keys only: the first k of each chunk
                idx, _ = g.sc.sparse(-1)
                ref = np.concatenate([np.arange(409), 4096 + np.arange(409), 8192 + np.arange(9)])
                assert np.array_equal(idx, ref)
    finally:
        g.close()


def test_loaded_residuals_select_exactly():
    # beta1 = 0 makes u = g; with zero gradients a = e, so both selections of a
    # step (step 0 and the new mask) rank the loaded e: +-0, ties, denormals.
    wl = synth.tiny(4 * 1024, 2, 1024, 0.25, beta1=0.0)
    rng = np.random.default_rng(5)
    e0 = (rng.integers(-8, 9, (2, wl.N)) * 0.5).astype(np.float32)
    e0[:, ::97] = -0.0
    e0[:, 5::131] = np.float32(1e-40)
    g, r = DeviceRun(wl, 0.25), OracleRun(wl, 0.25)
    try:
        for w in range(2):
            g.sc.load(E, e0[w], w)
            r.o.set(oracle.E, e0[w], w)
        zero = np.zeros((2, wl.N), np.uint16)
        for t in range(2):
            g.step(zero)
            r.step(zero)
            compare(g, r, f"step {t}")
    finally:
        g.close()


@pytest.mark.parametrize("chunk,density", [(65536, 0.01), (16384, 0.04)])
@pytest.mark.parametrize("n_high,n_tied,expect_fallback",
                         [(300, 400, False), (100, 1500, False), (100, 3000, True)])
def test_tied_bucket_paths(chunk, density, n_high, n_tied, expect_fallback):
    # Two chunks per worker with k = 655 (both CTA shapes of the step kernel):
    # n_high keys of 2.0 and n_tied keys of 1.0 (the rest 0.5); n_high < 655 <
    # n_high + n_tied puts the threshold inside the 16-bit bucket of 1.0, which
    # then holds n_tied tied keys.  400 -> ranked directly, 1500 -> radix among
    # the on-chip candidates, 3000 -> more than the on-chip list holds, redone
    # by the standalone select.
    wl = synth.tiny(chunk * 2, 2, chunk, density, beta1=0.0)
    assert int(np.floor(density * chunk)) == 655
    rng = np.random.default_rng(n_tied)
    e0 = np.full((2, wl.N), 0.5, np.float32)
    for w in range(2):
        for c in range(2):
            pos = c * chunk + rng.permutation(chunk)[: n_high + n_tied]
            e0[w, pos[:n_high]] = 2.0
            e0[w, pos[n_high:]] = -1.0
    g, r = DeviceRun(wl, density), OracleRun(wl, density)
    try:
        for w in range(2):
            g.sc.load(E, e0[w], w)
            r.o.set(oracle.E, e0[w], w)
        zero = np.zeros((2, wl.N), np.uint16)
        g.step(zero)
        r.step(zero)
        compare(g, r, "step 0")
        assert (g.sc._info()["select_fallbacks"] > 0) == expect_fallback
    finally:
        g.close()


def test_fallback_on_consecutive_steps():
    # 6000 residuals tied at |a| = 1.0 per chunk, zero gradients and b1 = 0:
    # every step keeps k = 655 of them, so the tied bucket stays above the
    # on-chip list for several steps and the standalone select redoes chunks
    # on every step (both slots of the step kernel's flagged-chunk counter).
    wl = synth.tiny(65536 * 2, 2, 65536, 0.01, beta1=0.0)
    rng = np.random.default_rng(77)
    e0 = np.full((2, wl.N), 0.5, np.float32)
    for w in range(2):
        for c in range(2):
            pos = c * 65536 + rng.permutation(65536)[:6100]
            e0[w, pos[:100]] = 2.0
            e0[w, pos[100:]] = -1.0
    g, r = DeviceRun(wl, 0.01), OracleRun(wl, 0.01)
    try:
        for w in range(2):
            g.sc.load(E, e0[w], w)
            r.o.set(oracle.E, e0[w], w)
        zero = np.zeros((2, wl.N), np.uint16)
        seen = 0
        for t in range(6):
            g.step(zero)
            r.step(zero)
            compare(g, r, f"step {t}")
            n = g.sc._info()["select_fallbacks"]
            assert n > seen, (t, n, seen)  # this step flagged chunks again
            seen = n
    finally:
        g.close()


def test_resume_is_bit_identical():
    wl = synth.tiny(3 * 4096 + 32, 3, 4096, 0.05, seed=8)
    a = DeviceRun(wl, 0.05)
    for _ in range(5):
        a.step()
    ref = {f: a.sc.read(f) for f in (THETA, V, MASK)}
    ref_u = [a.sc.read(U, w) for w in range(3)]
    a.close()
    b = DeviceRun(wl, 0.05)
    for _ in range(3):
        b.step()
    saved = {f: b.sc.read(f) for f in (THETA, V, MASK, STEP)}
    saved_ue = [(b.sc.read(U, w), b.sc.read(E, w)) for w in range(3)]
    b.close()
    c = DeviceRun(wl, 0.05, theta0=False)
    for f in (THETA, V, MASK, STEP):
        c.sc.load(f, saved[f])
    for w in range(3):
        c.sc.load(U, saved_ue[w][0], w)
        c.sc.load(E, saved_ue[w][1], w)
    c.t = 3
    for _ in range(2):
        c.step()
    try:
        for f in (THETA, V, MASK):
            assert np.array_equal(c.sc.read(f).view(np.uint32), ref[f].view(np.uint32)), f
        for w in range(3):
            assert np.array_equal(c.sc.read(U, w).view(np.uint32), ref_u[w].view(np.uint32))
        assert int(c.sc.read(STEP)[0]) == 5
    finally:
        c.close()


@pytest.mark.parametrize("memory", ["pinned", "pageable"])
def test_step_host_matches_step(memory):
    # pinned buffers are read in place by the kernel; pageable ones are staged
    wl = synth.tiny(20000, 2, 1024, 0.1, seed=4)
    a, b = DeviceRun(wl, 0.1), DeviceRun(wl, 0.1)
    try:
        for t in range(3):
            gr = np.stack([synth.cpu().grads(wl, w, t, n=wl.N) for w in range(2)])
            a.step(gr)
            if memory == "pinned":
                host = [torch.from_numpy(gr[w].view(np.int16)).pin_memory() for w in range(2)]
            else:
                host = [np.ascontiguousarray(gr[w]) for w in range(2)]
            b.sc.step_host(host)
        torch.cuda.synchronize()
        for f in (THETA, V, MASK):
            assert np.array_equal(a.sc.read(f).view(np.uint32), b.sc.read(f).view(np.uint32))
    finally:
        a.close()
        b.close()


def test_generator_gpu_equals_cpu():
    for name in ("flat-2^26-w8-ties", "gpt2-medium-w8", "llama-1.8b-w4"):
        wl = synth.WORKLOADS[name]
        n = 1 << 16
        for i0 in (0, wl.N // 2 + 5, wl.N - n):
            buf = torch.empty(n, dtype=torch.int16, device="cuda")
            synth.gpu().grads_into(wl, 1, 7, buf, i0=i0)
            ref = synth.cpu().grads(wl, 1, 7, i0=i0, n=n)
            assert np.array_equal(buf.cpu().numpy().view(np.uint16), ref), (name, i0)
        th = torch.empty(n, dtype=torch.float32, device="cuda")
        synth.gpu().theta_into(wl, th, i0=12345)
        ref = synth.cpu().theta0(wl, np.arange(12345, 12345 + n))
        assert np.array_equal(th.cpu().numpy().view(np.uint32), ref.view(np.uint32))


FULL = [("flat-2^26-w8-ties", 0.10), ("flat-2^26-w8-ties", 0.01), ("gpt2-medium-w8", 0.01),
        ("llama-500m-w8", 0.01), ("llama-500m-w8", 0.10), ("llama-1.8b-w4", 0.01)]


@pytest.mark.parametrize("name,density", FULL, ids=[f"{n}-d{d}" for n, d in FULL])
def test_full_size_sampled_chunks(name, density):
    wl = synth.WORKLOADS[name]
    ids = sample_chunks(wl)
    _run_both(wl, density, wl.steps, chunk_ids=ids)


def test_full_size_step_host_sampled():
    # the end-to-end path on the benchmark layout: page-locked host gradients
    # read in place by the step kernel over the CPU-GPU link
    wl = synth.WORKLOADS["llama-1.8b-w4"]
    ids = sample_chunks(wl)
    g = DeviceRun(wl, 0.01)
    r = OracleRun(wl, 0.01, chunk_ids=ids)
    host = [torch.empty(wl.N, dtype=torch.int16).pin_memory() for _ in range(wl.W)]
    try:
        for t in range(2):
            for w in range(wl.W):
                synth.gpu().grads_into(wl, w, t, g.grads[w])
                host[w].copy_(g.grads[w])
            torch.cuda.synchronize()
            g.sc.step_host(host)
            g.t += 1
            r.step()
            compare(g, r, f"step {t}")
        check_full_mask(g)
    finally:
        g.close()
        del host


# ---- variants: per-tensor chunks, residuals in host memory ---------------------------

from sparse_communication_distributed_gb300.scape import CHUNK_PER_TENSOR, RESIDUAL_HOST  # noqa: E402


def _per_tensor_run(wl, density, steps, chunk_ids=None):
    g = DeviceRun(wl, density, flags=CHUNK_PER_TENSOR)
    r = OracleRun(wl, density, chunk_ids=chunk_ids, per_tensor=True)
    try:
        assert g.sc.info["n_chunks"] == r.o.all_chunks()[0].size
        assert g.sc.K == int(r.o.all_chunks()[2].astype(np.int64).sum())
        for t in range(steps):
            g.step()
            r.step()
            compare(g, r, f"step {t}")
        check_full_mask(g, r)
    finally:
        g.close()


def test_per_tensor_chunks_small():
    # tensors of 96 .. 32000 coordinates (the last one ragged) cut separately
    numel = [96, 32000, 64, 3104, 1024, 4096 + 33]
    wl = synth.Workload("per-tensor", tuple((f"t{i}", (n,)) for i, n in enumerate(numel)), W=3,
                        chunk=1024, densities=(0.1,), steps=4, kind=synth.SYN_STUDENT_Q,
                        sigma=1e-3, seed=60)
    _per_tensor_run(wl, 0.1, 4)


def test_per_tensor_gpt2_full_size_sampled():
    wl = synth.WORKLOADS["gpt2-medium-w8"]
    probe = oracle.Oracle.for_workload(wl, 0.01, chunk_ids=[0], per_tensor=True)
    nch = probe.all_chunks()[0].size
    q = -(-nch // wl.W)
    ids = {0, 1, 2, nch - 2, nch - 1}
    for w in range(1, wl.W):
        ids |= {w * q - 1, w * q}
    ids |= set(int(x) for x in np.random.default_rng(1).integers(0, nch, 4))
    _per_tensor_run(wl, 0.01, 4, chunk_ids=sorted(ids))


def test_residuals_in_host_memory():
    wl = synth.tiny(3 * 4096 + 200, 3, 4096, 0.05, seed=61)
    g, r = DeviceRun(wl, 0.05, flags=RESIDUAL_HOST), OracleRun(wl, 0.05)
    try:
        assert g.sc.info["host_bytes"] >= 3 * wl.N * 4
        for t in range(3):
            g.step()
            r.step()
            compare(g, r, f"step {t}")
    finally:
        g.close()


def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    W = int(rng.integers(1, 10))
    C = 32 * int(rng.choice([1, 3, 8, 37, 128, 512, 2048]))
    density = float(rng.choice([0.003, 0.01, 0.05, 0.1, 0.37, 0.5, 1.0]))
    kind = int(rng.integers(0, 2))
    per_tensor = bool(rng.integers(0, 2))
    n_t = int(rng.integers(1, 6))
    numel = [32 * int(rng.integers(1, 3000)) for _ in range(n_t - 1)] + [int(rng.integers(1, 90000))]
    wl = synth.Workload(f"rand{seed}", tuple((f"t{i}", (n,)) for i, n in enumerate(numel)), W=W,
                        chunk=C, densities=(density,), steps=3, kind=kind, sigma=1e-3,
                        seed=seed)
    return wl, density, per_tensor


@pytest.mark.parametrize("seed", list(range(12)) + list(range(100, 112)))
def test_random_shapes(seed):
    wl, density, per_tensor = _random_case(seed)
    g = DeviceRun(wl, density, flags=CHUNK_PER_TENSOR if per_tensor else 0)
    r = OracleRun(wl, density, per_tensor=per_tensor)
    try:
        for t in range(3):
            g.step()
            r.step()
            compare(g, r, f"seed {seed} step {t}")
        check_full_mask(g, r)
    finally:
        g.close()


@pytest.mark.parametrize("seed", range(12, 18))
def test_random_shapes_host_residuals(seed):
    # the whole-sector access mapping of residuals in host memory, on ragged
    # chunk ends of every residue mod 4 and W from 1 to 9
    wl, density, per_tensor = _random_case(seed)
    flags = RESIDUAL_HOST | (CHUNK_PER_TENSOR if per_tensor else 0)
    g = DeviceRun(wl, density, flags=flags)
    r = OracleRun(wl, density, per_tensor=per_tensor)
    try:
        for t in range(3):
            g.step()
            r.step()
            compare(g, r, f"seed {seed} step {t}")
        check_full_mask(g, r)
    finally:
        g.close()


def test_largest_n():
    # N = 2^32 - 1, the largest N the uint32 coordinates allow: 65536 chunks of
    # 65536, the last one 65535 long; W = 2 (about 120 GB on the device).
    N = (1 << 32) - 1
    wl = synth.Workload("max-n", (("flat", (N,)),), W=2, chunk=65536, densities=(0.001,),
                        steps=2, sigma=1e-3, seed=90)
    nch = -(-N // 65536)
    ids = [0, 1, nch // 2 - 1, nch // 2, nch - 2, nch - 1]
    _run_both(wl, 0.001, 2, chunk_ids=ids)


def test_full_size_host_residuals_sampled():
    # the whole-sector mapping at full size: 17.8 GB of residuals in host memory
    wl = synth.WORKLOADS["llama-500m-w8"]
    ids = sample_chunks(wl)
    g = DeviceRun(wl, 0.01, flags=RESIDUAL_HOST)
    r = OracleRun(wl, 0.01, chunk_ids=ids)
    try:
        assert g.sc.info["host_bytes"] >= wl.W * wl.N * 4
        for t in range(3):
            g.step()
            r.step()
            compare(g, r, f"step {t}")
        check_full_mask(g)
    finally:
        g.close()


def test_per_tensor_with_host_residuals_and_mask_stats():
    # both options at once, and the mask diagnostics on per-tensor chunks
    numel = [96, 20000 * 32, 64, 4096 + 33]
    wl = synth.Workload("pt-host", tuple((f"t{i}", (n,)) for i, n in enumerate(numel)), W=3,
                        chunk=2048, densities=(0.05,), steps=3, sigma=1e-3, seed=62)
    g = DeviceRun(wl, 0.05, flags=CHUNK_PER_TENSOR | RESIDUAL_HOST)
    r = OracleRun(wl, 0.05, per_tensor=True)
    try:
        for t in range(3):
            g.step()
            r.step()
            compare(g, r, f"step {t}")
        st = g.sc.mask_stats()
        o = r.o
        m_new, m_used = o.mask(0).astype(bool), o.mask(1).astype(bool)
        union = np.zeros(o.n, bool)
        for w in range(wl.W):
            a = o.get(oracle.A, w)
            for j in range(o.chunk_start.size):
                s0, ln, k = int(o.chunk_start[j]), int(o.chunk_len[j]), int(o.chunk_k[j])
                union[s0:s0 + ln] |= oracle.topk(a[s0:s0 + ln], k).astype(bool)
        assert st["kept"] == int(m_new.sum())
        assert st["overlap_prev"] == int((m_new & m_used).sum())
        assert st["union_global_topk"] == int(union.sum())
    finally:
        g.close()
