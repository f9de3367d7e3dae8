"""Pins of the SCAPE oracle against facts that do not come from the oracle.

Each ``pin_*`` takes the path of a compiled oracle library and raises
AssertionError when the oracle breaks the fact it checks.  The test suite runs
them against the real oracle (``test_oracle_pins.py``) and against copies of it
with planted mistakes (``test_oracle_mutants.py``), which must each fail at
least one pin.

Sources of the facts (SCAPE, arXiv 2607.01678: abstract; gist.science technical
summary §2 and §3), stated in the oracle header:
  - at density 1 every coordinate is sent, so the step is dense AdamS on the
    mean first moment; by linearity of the momentum recurrence that equals one
    momentum run on the mean gradient (checked in fp64);
  - error feedback: a = b + e, and what is sent plus what is left equals
    what was accumulated;
  - delayed mask usage: the mask applied at step t is the one built at t-1,
    and step 0, which has no earlier mask, applies the selection of its own
    accumulators (recomputed here from loaded nonzero state);
  - partitioned top-k: every chunk keeps exactly floor(density*len) entries,
    the largest |a| of its owner, ties to the lower index (checked by its
    characterisation and against numpy's sort);
  - coordinates never sent only decay: theta *= (1 - lr*wd), v *= b2;
  - the non-partitioned alternative (technical summary §2, "Partitioned Mask
    Synchronization") keeps the union of every worker's own top-k per chunk.
"""
from __future__ import annotations

import math

import numpy as np

import oracle
import synth

SO = oracle.SO


def _f32_from_bf16(g: np.ndarray) -> np.ndarray:
    return (g.astype(np.uint32) << 16).view(np.float32)


def _key(a: np.ndarray) -> np.ndarray:
    return a.view(np.uint32) & np.uint32(0x7FFFFFFF)


def _run(o: oracle.Oracle, wl, steps: int, t0: int = 0, grads=None):
    gen = synth.cpu()
    for t in range(t0, t0 + steps):
        g = grads(t) if grads else np.stack([gen.grads(wl, w, t, idx=o.index) for w in range(o.W)])
        o.step(g)


# ---------------------------------------------------------------- density 1

def pin_dense_adams(lib: str = SO) -> None:
    """Density 1.0: every chunk keeps every coordinate, so theta and v follow
    dense AdamS driven by the mean gradient (one fp64 momentum)."""
    for W, eps in ((1, 1e-8), (3, 1e-8), (4, 1e-4)):
        wl = synth.tiny(3000, W, 256, 1.0, seed=11 + W, eps=eps)
        o = oracle.Oracle.for_workload(wl, 1.0, lib_path=lib)
        gen = synth.cpu()
        th0 = gen.theta0(wl, o.index)
        o.set(oracle.THETA, th0)
        m = np.zeros(o.n)
        v = np.zeros(o.n)
        th = th0.astype(np.float64)
        b1, b2, lr, wd = wl.beta1, wl.beta2, wl.lr, wl.wd
        for t in range(6):
            g = np.stack([gen.grads(wl, w, t, idx=o.index) for w in range(W)])
            o.step(g)
            gbar = _f32_from_bf16(g).astype(np.float64).mean(axis=0)
            m = b1 * m + (1 - b1) * gbar
            v = b2 * v + (1 - b2) * m * m
            th = th - lr * (m / (np.sqrt(v) + eps) + wd * th)
            assert o.mask(1).all(), "density 1 must apply every coordinate"
        np.testing.assert_allclose(o.get(oracle.V), v, rtol=2e-5, atol=1e-20)
        np.testing.assert_allclose(o.get(oracle.THETA), th, rtol=0, atol=5e-8)
        for w in range(W):
            assert not o.get(oracle.E, w).any(), "density 1 leaves no residual"


def pin_single_worker_identity(lib: str = SO) -> None:
    """W = 1: the synchronized buffer is worker 0's sparse buffer itself
    (mean of one term), at any density."""
    for d in (1.0, 0.25):
        wl = synth.tiny(2048, 1, 512, d, seed=5)
        o = oracle.Oracle.for_workload(wl, d, lib_path=lib)
        _run(o, wl, 3)
        i0, v0 = o.sparse(0)
        ib, vb = o.sparse(-1)
        assert np.array_equal(i0, ib)
        assert np.array_equal(v0.view(np.uint32), vb.view(np.uint32))


def pin_momentum_closed_form(lib: str = SO) -> None:
    """Constant gradient c on every worker and step, density 1:
    u_t = (1 - b1^(t+1)) c (geometric series) and bbar = u_t."""
    W, n = 2, 512
    wl = synth.tiny(n, W, 128, 1.0)
    o = oracle.Oracle.for_workload(wl, 1.0, lib_path=lib)
    c = np.float32(0.0078125)  # exactly representable in bf16
    gbits = np.full((W, o.n), (c.view(np.uint32) >> 16), dtype=np.uint16)
    for t in range(8):
        o.step(gbits)
        expect = (1 - wl.beta1 ** (t + 1)) * float(c)
        np.testing.assert_allclose(o.get(oracle.U, 1), expect, rtol=3e-6)
        _, bb = o.sparse(-1)
        np.testing.assert_allclose(bb, expect, rtol=3e-6)


def pin_fixed_sum_order(lib: str = SO) -> None:
    """bbar sums workers left to right, 0..W-1: with worker values 2^24, 1,
    -2^24 the fp32 sum is (2^24 + 1) - 2^24 = 0 (2^24+1 rounds to 2^24),
    whereas any order that adds 1 last gives 1/3."""
    W = 3
    wl = synth.tiny(64, W, 32, 1.0, beta1=1.0)  # b1 = 1: c1 = 0, u keeps its value
    o = oracle.Oracle.for_workload(wl, 1.0, lib_path=lib)
    for w, val in enumerate((16777216.0, 1.0, -16777216.0)):
        o.set(oracle.U, np.full(o.n, val, np.float32), w)
    o.step(np.zeros((W, o.n), np.uint16))
    _, bb = o.sparse(-1)
    assert np.all(bb == 0.0), bb[:4]


# ---------------------------------------------------------- error feedback

def pin_accumulator_split(lib: str = SO) -> None:
    """a_w = b_w + e_w exactly; b_w = a_w on the applied mask and +0 off it."""
    wl = synth.tiny(8192, 3, 1024, 0.05, seed=3)
    o = oracle.Oracle.for_workload(wl, 0.05, lib_path=lib)
    for t in range(4):
        _run(o, wl, 1, t0=t)
        m = o.mask(1).astype(bool)
        for w in range(3):
            a, b, e = o.get(oracle.A, w), o.get(oracle.B, w), o.get(oracle.E, w)
            assert np.array_equal((b + e).view(np.uint32) & 0x7FFFFFFF, a.view(np.uint32) & 0x7FFFFFFF)
            assert np.array_equal(b[m], a[m]) and not b[~m].any() and not e[m].any()
            assert np.array_equal(e[~m], a[~m])


def pin_error_feedback_conservation(lib: str = SO) -> None:
    """sum_s b_{w,s} + e_{w,T} = sum_s u_{w,s}, up to fp32 rounding of a."""
    W, T = 2, 6
    wl = synth.tiny(4096, W, 512, 0.02, seed=9)
    o = oracle.Oracle.for_workload(wl, 0.02, lib_path=lib)
    sb = np.zeros((W, o.n))
    su = np.zeros((W, o.n))
    amax = np.zeros((W, o.n))
    for t in range(T):
        _run(o, wl, 1, t0=t)
        for w in range(W):
            sb[w] += o.get(oracle.B, w)
            su[w] += o.get(oracle.U, w)
            amax[w] = np.maximum(amax[w], np.abs(o.get(oracle.A, w)))
    for w in range(W):
        lhs = sb[w] + o.get(oracle.E, w)
        tol = T * amax[w] * 2.0 ** -23 + 1e-30
        assert np.all(np.abs(lhs - su[w]) <= tol), np.abs(lhs - su[w]).max()


# ------------------------------------------------------------ delayed mask

def pin_delayed_mask(lib: str = SO) -> None:
    """The mask applied at step t (t >= 1) is the one built at step t-1, and
    the compact buffers hold exactly its coordinates, ascending."""
    wl = synth.tiny(6144, 2, 1024, 0.03, seed=21)
    o = oracle.Oracle.for_workload(wl, 0.03, lib_path=lib)
    prev = None
    for t in range(4):
        _run(o, wl, 1, t0=t)
        used = o.mask(1)
        if prev is not None:
            assert np.array_equal(used, prev)
        idx, _ = o.sparse(0)
        assert np.array_equal(idx, o.index[used.astype(bool)])
        assert np.all(np.diff(idx.astype(np.int64)) > 0)
        prev = o.mask(0)


# ------------------------------------------------------------ step-0 mask

def pin_bootstrap_mask(lib: str = SO) -> None:
    """Step 0 has no earlier mask, so the mask it applies (M_{-1}) is the
    selection run on the step-0 accumulators a_w = e_w + (b1*u_w + (1-b1)*g_w)
    before anything is written.  The state is loaded with nonzero u_w and e_w
    first, so every term of a_w matters; a_w is recomputed here in numpy fp32
    (one rounding per operation, as the rule states), and each chunk of the
    applied mask must equal numpy's lexsort top-k_c of the owner's a_w, or,
    in the non-partitioned variant, the union of every worker's top-k_c."""
    for union in (False, True):
        for kind in (synth.SYN_GAUSS, synth.SYN_STUDENT_Q):
            wl = synth.tiny(5 * 1024 + 352, 3, 1024, 0.1, kind=kind, seed=14, sigma=2e-3)
            o = oracle.Oracle.for_workload(wl, 0.1, lib_path=lib, union_mask=union)
            rng = np.random.default_rng(40 + kind)
            u0 = (rng.standard_normal((wl.W, o.n)) * 3e-3).astype(np.float32)
            e0 = (rng.standard_normal((wl.W, o.n)) * 2e-3).astype(np.float32)
            for w in range(wl.W):
                o.set(oracle.U, u0[w], w)
                o.set(oracle.E, e0[w], w)
            g = np.stack([synth.cpu().grads(wl, w, 0, idx=o.index) for w in range(wl.W)])
            o.step(g)
            b1 = np.float32(wl.beta1)
            c1 = np.float32(1.0) - b1
            a0 = e0 + ((b1 * u0) + (c1 * _f32_from_bf16(g)))
            used = o.mask(1).astype(bool)
            for j in range(o.chunk_start.size):
                s, ln = int(o.chunk_start[j]), int(o.chunk_len[j])
                k = math.floor(0.1 * ln)
                rows = a0[:, s:s + ln] if union else a0[int(o.chunk_owner[j])][None, s:s + ln]
                ref = _union_ref(rows, k)
                assert np.array_equal(used[s:s + ln], ref), (union, kind, j)


# --------------------------------------------------------------- selection

def _check_topk_flags(a: np.ndarray, keep: np.ndarray, k: int) -> None:
    keep = keep.astype(bool)
    assert keep.sum() == k
    if k == 0 or k == a.size:
        return
    key = _key(a).astype(np.int64)
    kmin, umax = key[keep].min(), key[~keep].max()
    assert kmin >= umax
    if kmin == umax:  # ties at the threshold: kept ones come first
        tie = np.nonzero(key == kmin)[0]
        assert np.all(np.diff(keep[tie].astype(np.int8)) <= 0)


def pin_partitioned_topk(lib: str = SO) -> None:
    """Every chunk's next mask is the top-k_c of its owner's |a|, ties to the
    lower index; k_c = floor(density*len) (ragged last chunk included)."""
    for kind in (synth.SYN_GAUSS, synth.SYN_STUDENT_Q):
        wl = synth.tiny(5 * 1024 + 352, 3, 1024, 0.1, kind=kind, seed=4, sigma=2e-3)
        o = oracle.Oracle.for_workload(wl, 0.1, lib_path=lib)
        for t in range(3):
            _run(o, wl, 1, t0=t)
            m = o.mask(0)
            for j in range(o.chunk_start.size):
                s = int(o.chunk_start[j])
                ln = int(o.chunk_len[j])
                k = math.floor(0.1 * ln)
                assert o.chunk_k[j] == k
                a = o.get(oracle.A, int(o.chunk_owner[j]))[s:s + ln]
                _check_topk_flags(a, m[s:s + ln], k)


def pin_topk_against_sort(lib: str = SO) -> None:
    """The selection agrees with numpy's stable lexicographic sort on
    (|a| descending, index ascending), 64..4096 elements, heavy ties, +-0,
    k in {0, 1, random, len}; all-equal input keeps the first k."""
    rng = np.random.default_rng(1)
    for n in (64, 100, 1000, 4096):
        for kind in range(3):
            if kind == 0:
                a = rng.standard_normal(n).astype(np.float32)
            elif kind == 1:
                a = (rng.integers(-6, 7, n) * 0.25).astype(np.float32)
                a[rng.integers(0, n, 5)] = -0.0
            else:
                a = np.full(n, -1.5, np.float32)
            for k in (0, 1, int(rng.integers(0, n + 1)), n):
                keep = oracle.topk(a, k, lib_path=lib)
                order = np.lexsort((np.arange(n), -_key(a).astype(np.int64)))
                ref = np.zeros(n, np.uint8)
                ref[order[:k]] = 1
                assert np.array_equal(keep, ref), (n, kind, k)
                if kind == 2:
                    assert keep[:k].all() and not keep[k:].any()


def pin_shard_geometry(lib: str = SO) -> None:
    """Chunk counts, k and shard ownership on the five workload layouts:
    q = ceil(n_ch/W) chunks per worker, the last worker takes the rest;
    K for 2^20 at density 0.1, chunk 4096 is 256 * floor(409.6) = 104704."""
    expect = {  # name: (chunks, last chunk len, chunks of the last worker)
        "flat-2^20-w4": (256, 4096, 64),
        "flat-2^26-w8-ties": (1024, 65536, 128),
        "gpt2-medium-w8": (5415, 354823168 - 5414 * 65536, 5415 - 7 * 677),
        "llama-500m-w8": (8511, 557774080 - 8510 * 65536, 8511 - 7 * 1064),
        "llama-1.8b-w4": (27091, 1775372288 - 27090 * 65536, 27091 - 3 * 6773),
    }
    for name, (nch, last, nlast) in expect.items():
        wl = synth.WORKLOADS[name]
        ids = [0, nch - 1]
        o = oracle.Oracle.for_workload(wl, wl.densities[0], chunk_ids=ids, lib_path=lib)
        assert int(o.chunk_len[1]) == last
        assert int(o.chunk_owner[1]) == wl.W - 1 and int(o.chunk_owner[0]) == 0
        q = -(-nch // wl.W)
        assert nch - (wl.W - 1) * q == nlast
        assert int(o.chunk_k[0]) == math.floor(wl.densities[0] * wl.chunk)
    o = oracle.Oracle.for_workload(synth.WORKLOADS["flat-2^20-w4"], 0.1, lib_path=lib)
    assert int(o.chunk_k.astype(np.int64).sum()) == 104704


def pin_per_tensor_chunks(lib: str = SO) -> None:
    """Per-tensor chunking: every tensor is cut into ceil(n_t / C) chunks that
    start at the tensor's offset, k_c = floor(density * len_c), shards stay
    contiguous over the chunk list, and the top-k characterisation holds in
    every such chunk (ties included)."""
    numel = [96, 1000 * 32, 64, 3 * 1024 + 32, 32]
    C, W, d = 1024, 3, 0.1
    starts = np.concatenate([[0], np.cumsum(numel)])
    expect = [int(starts[t]) + x for t, n in enumerate(numel) for x in range(0, n, C)]
    wl = synth.Workload("pt", tuple((f"t{i}", (n,)) for i, n in enumerate(numel)), W=W, chunk=C,
                        densities=(d,), steps=1, kind=synth.SYN_STUDENT_Q, sigma=2e-3, seed=6)
    o = oracle.Oracle.for_workload(wl, d, lib_path=lib, per_tensor=True)
    assert o.chunk_start.astype(np.int64).tolist() == expect
    q = -(-len(expect) // W)
    assert o.chunk_owner.tolist() == [j // q for j in range(len(expect))]
    for t in range(3):
        _run(o, wl, 1, t0=t)
        m = o.mask(0)
        for j in range(o.chunk_start.size):
            s0, ln = int(o.chunk_start[j]), int(o.chunk_len[j])
            k = math.floor(d * ln)
            assert int(o.chunk_k[j]) == k
            _check_topk_flags(o.get(oracle.A, int(o.chunk_owner[j]))[s0:s0 + ln], m[s0:s0 + ln], k)


# -------------------------------------------------------------- off the mask

def pin_offmask_decay(lib: str = SO) -> None:
    """A coordinate that is never sent only decays: theta_T = theta_0 (1 - lr
    wd)^T and v_T = b2^T v_0 (fp64 closed forms)."""
    W, T, n = 2, 5, 2048
    wl = synth.tiny(n, W, 1024, 0.01, seed=2)
    o = oracle.Oracle.for_workload(wl, 0.01, lib_path=lib)
    th0 = synth.cpu().theta0(wl, o.index)
    v0 = np.full(n, 3e-7, np.float32)
    o.set(oracle.THETA, th0)
    o.set(oracle.V, v0)
    # coordinates >= 64 of each chunk get zero gradient; the rest are large,
    # so k = 10 per chunk is always drawn from the first 64
    def grads(t):
        g = np.zeros((W, n), np.uint16)
        base = synth.cpu().grads(wl, 0, t, idx=o.index)
        for s in (0, 1024):
            g[:, s:s + 64] = base[s:s + 64]
        return g
    ever = np.zeros(n, bool)
    for t in range(T):
        _run(o, wl, 1, t0=t, grads=grads)
        ever |= o.mask(1).astype(bool)
    never = ~ever
    assert never.sum() > 1800
    th_ref = th0.astype(np.float64) * (1 - wl.lr * wl.wd) ** T
    np.testing.assert_allclose(o.get(oracle.THETA)[never], th_ref[never], rtol=2e-6)
    np.testing.assert_allclose(o.get(oracle.V)[never], (v0.astype(np.float64) * wl.beta2 ** T)[never],
                               rtol=2e-6)


# ---------------------------------------------------------------- dense AdamS

def pin_dense_adams_single_worker(lib: str = SO) -> None:
    """Dense AdamS with W = 1 is the SCAPE step at W = 1, density 1, bit for
    bit: gbar = g, m = u, bbar = u (1/W = 1 is exact)."""
    wl = synth.tiny(2048, 1, 512, 1.0, seed=31)
    o = oracle.Oracle.for_workload(wl, 1.0, lib_path=lib)
    th0 = synth.cpu().theta0(wl, o.index)
    o.set(oracle.THETA, th0)
    th, m, v = th0.copy(), np.zeros(o.n, np.float32), np.zeros(o.n, np.float32)
    for t in range(4):
        g = np.stack([synth.cpu().grads(wl, 0, t, idx=o.index)])
        o.step(g)
        oracle.dense_adams_step(th, m, v, g, wl.beta1, wl.beta2, wl.lr, wl.wd, wl.eps, lib_path=lib)
    assert np.array_equal(th.view(np.uint32), o.get(oracle.THETA).view(np.uint32))
    assert np.array_equal(v.view(np.uint32), o.get(oracle.V).view(np.uint32))
    assert np.array_equal(m.view(np.uint32), o.get(oracle.U, 0).view(np.uint32))


def pin_dense_adams_matches_scape_density1(lib: str = SO) -> None:
    """W = 4: the mean of per-worker momenta (SCAPE at density 1) equals the
    momentum of the mean gradient (dense AdamS) up to fp32 rounding."""
    wl = synth.tiny(4096, 4, 1024, 1.0, seed=32)
    o = oracle.Oracle.for_workload(wl, 1.0, lib_path=lib)
    th0 = synth.cpu().theta0(wl, o.index)
    o.set(oracle.THETA, th0)
    th, m, v = th0.copy(), np.zeros(o.n, np.float32), np.zeros(o.n, np.float32)
    for t in range(5):
        g = np.stack([synth.cpu().grads(wl, w, t, idx=o.index) for w in range(4)])
        o.step(g)
        oracle.dense_adams_step(th, m, v, g, wl.beta1, wl.beta2, wl.lr, wl.wd, wl.eps, lib_path=lib)
    np.testing.assert_allclose(v, o.get(oracle.V), rtol=2e-5, atol=1e-20)
    np.testing.assert_allclose(th, o.get(oracle.THETA), rtol=0, atol=5e-8)


def pin_dense_adams_constant_gradient(lib: str = SO) -> None:
    """Constant gradient c: m_t = (1 - b1^(t+1)) c, v_t = sum_s b2^(t-s) (1-b2) m_s^2."""
    n, W = 256, 3
    c = np.float32(0.0078125)
    g = np.full((W, n), c.view(np.uint32) >> 16, np.uint16)
    th, m, v = np.zeros(n, np.float32), np.zeros(n, np.float32), np.zeros(n, np.float32)
    vr = 0.0
    for t in range(6):
        oracle.dense_adams_step(th, m, v, g, lib_path=lib)
        mr = (1 - 0.9 ** (t + 1)) * float(c)
        vr = 0.95 * vr + 0.05 * mr * mr
        np.testing.assert_allclose(m, mr, rtol=3e-6)
        np.testing.assert_allclose(v, vr, rtol=1e-5)


def _union_ref(rows: np.ndarray, k: int) -> np.ndarray:
    """Union over the rows of each row's top-k by (|a| descending, index
    ascending), from numpy's lexicographic sort."""
    n = rows.shape[1]
    ref = np.zeros(n, bool)
    for a in rows:
        order = np.lexsort((np.arange(n), -_key(a).astype(np.int64)))
        ref[order[:k]] = True
    return ref


def pin_union_mask(lib: str = SO) -> None:
    """The non-partitioned variant: each chunk's next mask is the union over
    workers of each worker's own top-k_c (computed here with numpy's sort), so
    it keeps between k_c and min(len, W*k_c) coordinates and somewhere more
    than k_c (fill-in); it is applied one step later, and the compact list
    holds exactly the applied mask's coordinates, ascending."""
    for kind in (synth.SYN_GAUSS, synth.SYN_STUDENT_Q):
        wl = synth.tiny(5 * 1024 + 352, 3, 1024, 0.1, kind=kind, seed=5, sigma=2e-3)
        o = oracle.Oracle.for_workload(wl, 0.1, lib_path=lib, union_mask=True)
        prev = None
        grew = False
        for t in range(3):
            _run(o, wl, 1, t0=t)
            m = o.mask(0).astype(bool)
            used = o.mask(1).astype(bool)
            if prev is not None:
                assert np.array_equal(used, prev)
            idx, _ = o.sparse(0)
            assert np.array_equal(idx, o.index[used])
            for j in range(o.chunk_start.size):
                s, ln = int(o.chunk_start[j]), int(o.chunk_len[j])
                k = math.floor(0.1 * ln)
                rows = np.stack([o.get(oracle.A, w)[s:s + ln] for w in range(wl.W)])
                ref = _union_ref(rows, k)
                assert np.array_equal(m[s:s + ln], ref), (kind, t, j)
                cnt = int(ref.sum())
                assert k <= cnt <= min(ln, wl.W * k)
                grew |= cnt > k
            prev = m
        assert grew


def pin_union_single_worker(lib: str = SO) -> None:
    """With one worker the union is that worker's own top-k: the
    non-partitioned variant equals the partitioned rule bit for bit."""
    wl = synth.tiny(3 * 1024 + 96, 1, 1024, 0.05, seed=9)
    a = oracle.Oracle.for_workload(wl, 0.05, lib_path=lib)
    b = oracle.Oracle.for_workload(wl, 0.05, lib_path=lib, union_mask=True)
    for o in (a, b):
        o.set(oracle.THETA, synth.cpu().theta0(wl, o.index))
        _run(o, wl, 4)
    for f in (oracle.THETA, oracle.V, oracle.U, oracle.E):
        assert np.array_equal(a.get(f).view(np.uint32), b.get(f).view(np.uint32)), f
    assert np.array_equal(a.mask(0), b.mask(0))


ALL_PINS = [
    pin_dense_adams, pin_single_worker_identity, pin_momentum_closed_form, pin_fixed_sum_order,
    pin_accumulator_split, pin_error_feedback_conservation, pin_delayed_mask,
    pin_bootstrap_mask,
    pin_partitioned_topk, pin_topk_against_sort, pin_shard_geometry, pin_per_tensor_chunks,
    pin_offmask_decay,
    pin_dense_adams_single_worker, pin_dense_adams_matches_scape_density1,
    pin_dense_adams_constant_gradient, pin_union_mask, pin_union_single_worker,
]
