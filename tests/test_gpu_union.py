"""The non-partitioned variant (SCAPE_UNION_MASK: every worker's own top-k in
every chunk, OR-ed) against the oracle's union mode, bit for bit: every
coordinate on small layouts of both kernel shapes, sampled chunks at full
size, the tied-bucket fallback, mask loads and the mask diagnostics."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_harness import (DeviceRun, OracleRun, compare_all, compare_by_coordinate,  # noqa: E402
                         sample_chunks)
from sparse_communication_distributed_gb300 import E, MASK, THETA, U, V  # noqa: E402
from sparse_communication_distributed_gb300.scape import (CHUNK_PER_TENSOR, RESIDUAL_HOST,  # noqa: E402
                                                          UNION_MASK, ScapeError)

pytestmark = pytest.mark.gpu


def _run(wl, density, steps, flags=UNION_MASK, chunk_ids=None, per_tensor=False):
    g = DeviceRun(wl, density, flags=flags)
    r = OracleRun(wl, density, chunk_ids=chunk_ids, per_tensor=per_tensor, union_mask=True)
    ks = []
    try:
        for t in range(steps):
            g.step()
            r.step()
            if r.o.n == wl.N:
                compare_all(g, r, f"step {t}")
            else:
                compare_by_coordinate(g, r, f"step {t}")
            ks.append(g.sc.K)
    finally:
        g.close()
    return ks


@pytest.mark.parametrize("N,W,chunk,density", [
    (5 * 4096 + 160, 3, 4096, 0.05),       # 512-thread shape, ragged last chunk
    (3 * 65536 + 96, 4, 65536, 0.01),      # 1024-thread shape
    (70001, 5, 1024, 0.02),                # odd sizes
    (4099, 9, 96, 0.2),                    # W * k_c above the chunk length: capped at len
    (2048 + 7, 4, 512, 1.0),               # density 1: every worker keeps everything
])
def test_union_every_coordinate(N, W, chunk, density):
    ks = _run(synth.tiny(N, W, chunk, density, seed=N), density, 4)
    k_sum = sum(int(np.floor(density * min(chunk, N - c))) for c in range(0, N, chunk))
    assert all(k >= k_sum for k in ks)
    if density < 1.0:
        assert max(ks) > k_sum  # the union fills in
    else:
        assert ks == [N] * len(ks)


def test_union_single_worker_equals_partitioned():
    wl = synth.tiny(3 * 4096 + 64, 1, 4096, 0.05, seed=31)
    a, b = DeviceRun(wl, 0.05), DeviceRun(wl, 0.05, flags=UNION_MASK)
    try:
        for _ in range(4):
            a.step()
            b.step()
        for f in (THETA, V, MASK):
            assert np.array_equal(a.sc.read(f).view(np.uint32), b.sc.read(f).view(np.uint32))
        for f in (U, E):
            assert np.array_equal(a.sc.read(f, 0).view(np.uint32), b.sc.read(f, 0).view(np.uint32))
        assert a.sc.K == b.sc.K
    finally:
        a.close()
        b.close()


def test_union_per_tensor_and_host_residuals():
    numel = [96, 20000 * 32, 64, 4096 + 33]
    wl = synth.Workload("union-pt", tuple((f"t{i}", (n,)) for i, n in enumerate(numel)), W=3,
                        chunk=2048, densities=(0.05,), steps=3, sigma=1e-3, seed=63)
    _run(wl, 0.05, 3, flags=UNION_MASK | CHUNK_PER_TENSOR | RESIDUAL_HOST, per_tensor=True)


@pytest.mark.parametrize("chunk,density", [(65536, 0.01), (16384, 0.04)])
def test_union_tied_bucket_fallback(chunk, density):
    # worker 1's accumulator holds 3000 keys tied at |a| = 1.0 per chunk: its
    # selection overflows the on-chip list and the standalone select redoes
    # the chunk as the union of both workers' selections
    wl = synth.tiny(chunk * 2, 2, chunk, density, beta1=0.0)
    rng = np.random.default_rng(5)
    e0 = np.full((2, wl.N), 0.5, np.float32)
    e0[0] = rng.standard_normal(wl.N).astype(np.float32)
    for c in range(2):
        pos = c * chunk + rng.permutation(chunk)[:3100]
        e0[1, pos[:100]] = 2.0
        e0[1, pos[100:]] = -1.0
    g, r = DeviceRun(wl, density, flags=UNION_MASK), OracleRun(wl, density, union_mask=True)
    try:
        for w in range(2):
            g.sc.load(E, e0[w], w)
            r.o.set(oracle.E, e0[w], w)
        zero = np.zeros((2, wl.N), np.uint16)
        for t in range(3):
            g.step(zero)
            r.step(zero)
            compare_all(g, r, f"step {t}")
        assert g.sc._info()["select_fallbacks"] > 0
    finally:
        g.close()


def test_union_full_size_sampled():
    wl = synth.WORKLOADS["llama-500m-w8"]
    _run(wl, 0.01, 3, chunk_ids=sample_chunks(wl))


def test_union_mask_load_and_diagnostics():
    wl = synth.tiny(4 * 4096, 3, 4096, 0.05, seed=41)
    g = DeviceRun(wl, 0.05, flags=UNION_MASK)
    r = OracleRun(wl, 0.05, union_mask=True)
    try:
        for t in range(2):
            g.step()
            r.step()
        # the mask diagnostics: M_t is itself the union of the workers' top-k
        st = g.sc.mask_stats()
        m_new = r.o.mask(0).astype(bool)
        assert st["kept"] == int(m_new.sum()) == st["union_global_topk"]
        assert st["overlap_prev"] == int((m_new & r.o.mask(1).astype(bool)).sum())
        # a loaded union mask drives the next step exactly like the oracle's
        m = oracle.pack_bits(r.o.mask(0))
        g.sc.load(MASK, m)
        g.step()
        r.step()
        compare_all(g, r, "after the load")
        # fewer than k_c bits in a chunk is not a union of top-k selections
        bad = m.copy()
        bad[: 4096 // 32] = 0
        with pytest.raises(ScapeError):
            g.sc.load(MASK, bad)
    finally:
        g.close()


@pytest.mark.parametrize("seed", list(range(18, 24)) + list(range(200, 206)))
def test_union_random_shapes(seed):
    rng = np.random.default_rng(2000 + seed)
    W = int(rng.integers(1, 10))
    C = 32 * int(rng.choice([1, 3, 8, 37, 128, 512, 2048]))
    density = float(rng.choice([0.003, 0.01, 0.05, 0.1, 0.37]))
    n_t = int(rng.integers(1, 5))
    numel = [32 * int(rng.integers(1, 3000)) for _ in range(n_t - 1)] + [int(rng.integers(1, 90000))]
    per_tensor = bool(rng.integers(0, 2))
    wl = synth.Workload(f"urand{seed}", tuple((f"t{i}", (n,)) for i, n in enumerate(numel)), W=W,
                        chunk=C, densities=(density,), steps=3, kind=int(rng.integers(0, 2)),
                        sigma=1e-3, seed=seed)
    _run(wl, density, 3, flags=UNION_MASK | (CHUNK_PER_TENSOR if per_tensor else 0),
         per_tensor=per_tensor)


def test_union_debug_build_records_nothing():
    # the debug build's guards bound every compact slot by the chunk's count in
    # M_{t-1} (the union's capacity): on valid input none fires and the result
    # equals the release build's bit for bit
    import os
    from sparse_communication_distributed_gb300 import build as pkg_build
    from sparse_communication_distributed_gb300.scape import DEBUG_LIB_PATH, Scape
    if not os.path.exists(DEBUG_LIB_PATH):
        pkg_build.build(debug_checks=True)
    wl = synth.tiny(3 * 65536 + 96, 4, 65536, 0.01, seed=77)
    dev = torch.device("cuda")
    out = []
    for lib in (None, DEBUG_LIB_PATH):
        kw = {} if lib is None else {"lib_path": lib}
        sc = Scape.for_workload(wl, 0.01, flags=UNION_MASK, **kw)
        grads = [torch.empty(wl.N, dtype=torch.int16, device=dev) for _ in range(wl.W)]
        for t in range(3):
            for w in range(wl.W):
                synth.gpu().grads_into(wl, w, t, grads[w])
            sc.step(grads)
        torch.cuda.synchronize()
        info = sc._info()
        out.append((sc.read(THETA).view(np.uint32), sc.read(MASK), sc.sparse(-1)[1].view(np.uint32),
                    info))
        sc.close()
    (th_r, m_r, b_r, _), (th_d, m_d, b_d, info_d) = out
    assert info_d["checks_compiled"] == 1 and info_d["check_count"] == 0, info_d
    assert np.array_equal(th_r, th_d) and np.array_equal(m_r, m_d) and np.array_equal(b_r, b_d)

