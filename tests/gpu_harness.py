"""Helpers of the GPU parity tests: run libscape and the oracle on the same
seeded inputs and compare them over whole chunks.

Tolerance for floats (theta, v, u, e, kept values, bbar):
    |gpu - oracle| <= 1e-6 * |oracle| + 1e-12
and, because both sides evaluate the same fp32 expressions in the same order
without fused multiply-adds, the tests also require bit equality.  Masks,
coordinate lists and counts must be bit-exact.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import synth
from sparse_communication_distributed_gb300 import E, MASK, THETA, U, V, Scape
from sparse_communication_distributed_gb300.scape import DEBUG_LIB_PATH

RTOL, ATOL = 1e-6, 1e-12


def assert_close_exact(name: str, got: np.ndarray, ref: np.ndarray) -> None:
    got = np.asarray(got, np.float32)
    ref = np.asarray(ref, np.float32)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    err = np.abs(got.astype(np.float64) - ref.astype(np.float64))
    bad = err > RTOL * np.abs(ref.astype(np.float64)) + ATOL
    if bad.any():
        i = int(np.nonzero(bad)[0][0])
        raise AssertionError(f"{name}: {int(bad.sum())} values outside tolerance; first at {i}: "
                             f"gpu {got[i]!r} oracle {ref[i]!r}")
    neq = got.view(np.uint32) != ref.view(np.uint32)
    if neq.any():
        i = int(np.nonzero(neq)[0][0])
        raise AssertionError(f"{name}: {int(neq.sum())} values within tolerance but not bit-equal; "
                             f"first at {i}: gpu {got[i]!r} oracle {ref[i]!r}")


class DeviceRun:
    """libscape on a workload, inputs from the GPU build of the generator."""

    def __init__(self, wl, density: float, theta0: bool = True, flags: int = 0):
        self.wl = wl
        # SCAPE_TEST_LIB=debug runs the suite on libscape_debug.so, whose kernels
        # check every mask-dependent index; close() then asserts none failed
        self.debug = os.environ.get("SCAPE_TEST_LIB") == "debug"
        lib = {"lib_path": DEBUG_LIB_PATH} if self.debug else {}
        self.sc = Scape.for_workload(wl, density, flags=flags, **lib)
        self.dev = torch.device("cuda")
        self.grads = [torch.empty(wl.N, dtype=torch.int16, device=self.dev) for _ in range(wl.W)]
        if theta0:
            th = torch.empty(wl.N, dtype=torch.float32, device=self.dev)
            synth.gpu().theta_into(wl, th)
            torch.cuda.synchronize()
            self.sc.load(THETA, th)
            del th
        self.t = 0

    def step(self, grads=None) -> None:
        if grads is None:
            for w in range(self.wl.W):
                synth.gpu().grads_into(self.wl, w, self.t, self.grads[w])
        else:
            for w in range(self.wl.W):
                self.grads[w].copy_(torch.from_numpy(grads[w].view(np.int16)))
        self.sc.step(self.grads)
        self.t += 1

    def close(self):
        if self.debug:
            info = self.sc._info()
            assert info["checks_compiled"] == 1 and info["check_count"] == 0, info
        self.sc.close()
        self.grads = None
        torch.cuda.empty_cache()


class OracleRun:
    """The oracle over a set of whole chunks, inputs from the CPU build of the
    generator."""

    def __init__(self, wl, density: float, chunk_ids=None, theta0: bool = True,
                 per_tensor: bool = False, union_mask: bool = False):
        self.wl = wl
        self.o = oracle.Oracle.for_workload(wl, density, chunk_ids=chunk_ids,
                                            per_tensor=per_tensor, union_mask=union_mask)
        if theta0:
            self.o.set(oracle.THETA, synth.cpu().theta0(wl, self.o.index))
        self.t = 0

    def grads(self, t: int) -> np.ndarray:
        return np.stack([synth.cpu().grads(self.wl, w, t, idx=self.o.index)
                         for w in range(self.wl.W)])

    def step(self, grads=None) -> None:
        self.o.step(self.grads(self.t) if grads is None else grads)
        self.t += 1


def compare(g: DeviceRun, r: OracleRun, what: str = "") -> None:
    """Compare the GPU state with the oracle over the oracle's chunks."""
    if r.o.n == g.wl.N:
        return compare_all(g, r, what)
    o, sc, W = r.o, g.sc, g.wl.W
    m_gen = o.mask(0)
    m_used = o.mask(1)
    all_start, _, all_k = o.all_chunks()
    all_base = np.concatenate([[0], np.cumsum(all_k.astype(np.int64))])
    pos = 0
    for j in range(o.chunk_start.size):
        s, ln, k = int(o.chunk_start[j]), int(o.chunk_len[j]), int(o.chunk_k[j])
        c = int(np.searchsorted(all_start, s))
        sl = slice(pos, pos + ln)
        tag = f"{what} chunk {c}"
        assert_close_exact(f"theta {tag}", sc.read(THETA, offset=s, count=ln), o.get(oracle.THETA)[sl])
        assert_close_exact(f"v {tag}", sc.read(V, offset=s, count=ln), o.get(oracle.V)[sl])
        for w in range(W):
            assert_close_exact(f"u[{w}] {tag}", sc.read(U, w, offset=s, count=ln),
                               o.get(oracle.U, w)[sl])
            assert_close_exact(f"e[{w}] {tag}", sc.read(E, w, offset=s, count=ln),
                               o.get(oracle.E, w)[sl])
        # next mask (bit-exact), words of this chunk
        nw = (ln + 31) // 32
        words = sc.read(MASK, offset=s // 32, count=nw)
        ref = oracle.pack_bits(m_gen[sl])
        if not np.array_equal(words, ref):
            bad = np.nonzero(words != ref)[0]
            raise AssertionError(f"mask {tag}: {bad.size} words differ, first word {bad[0]}")
        # compact buffers of this chunk: packed positions [base_c, base_c + k)
        base = int(all_base[c])
        kept_local = np.nonzero(m_used[sl])[0]
        assert kept_local.size == k, (tag, kept_local.size, k)
        if k:
            oidx, _ = o.sparse(0)
            start = int(np.count_nonzero(m_used[:pos]))
            for w in list(range(W)) + [-1]:
                gi, gv = sc.sparse(w, offset=base, count=k)
                _, ov = o.sparse(w)
                assert np.array_equal(gi.astype(np.uint64), oidx[start:start + k]), f"idx {tag}"
                assert_close_exact(f"vals[{w}] {tag}", gv, ov[start:start + k])
        pos += ln


def compare_all(g: DeviceRun, r: OracleRun, what: str = "") -> None:
    """compare() when the oracle covers every coordinate: whole arrays at once."""
    o, sc, W = r.o, g.sc, g.wl.W
    assert_close_exact(f"theta {what}", sc.read(THETA), o.get(oracle.THETA))
    assert_close_exact(f"v {what}", sc.read(V), o.get(oracle.V))
    for w in range(W):
        assert_close_exact(f"u[{w}] {what}", sc.read(U, w), o.get(oracle.U, w))
        assert_close_exact(f"e[{w}] {what}", sc.read(E, w), o.get(oracle.E, w))
    words = sc.mask()
    ref = oracle.pack_bits(o.mask(0))
    if not np.array_equal(words, ref):
        bad = np.nonzero(words != ref)[0]
        raise AssertionError(f"mask {what}: {bad.size} words differ, first word {bad[0]}")
    oidx, _ = o.sparse(0)
    assert oidx.size == sc.K, (what, oidx.size, sc.K)
    if sc.K:
        for w in list(range(W)) + [-1]:
            gi, gv = sc.sparse(w)
            _, ov = o.sparse(w)
            assert np.array_equal(gi.astype(np.uint64), oidx), f"idx {what}"
            assert_close_exact(f"vals[{w}] {what}", gv, ov)


def compare_by_coordinate(g: DeviceRun, r: OracleRun, what: str = "") -> None:
    """compare() for layouts whose packed positions depend on every chunk (the
    union variant): state and mask words chunk by chunk over the oracle's
    chunks, and each chunk's compact entries located through the device's own
    coordinate list."""
    o, sc, W = r.o, g.sc, g.wl.W
    m_gen = o.mask(0)
    K = sc.K
    gidx, _ = sc.sparse(0, count=K)
    gidx = gidx.astype(np.uint64)
    assert np.all(np.diff(gidx.astype(np.int64)) > 0), f"idx not ascending {what}"
    g_vals = [sc.sparse(w, count=K)[1] for w in list(range(W)) + [-1]]
    oidx, _ = o.sparse(0)
    o_vals = [o.sparse(w)[1] for w in list(range(W)) + [-1]]
    pos = 0
    for j in range(o.chunk_start.size):
        s, ln = int(o.chunk_start[j]), int(o.chunk_len[j])
        sl = slice(pos, pos + ln)
        tag = f"{what} chunk at {s}"
        assert_close_exact(f"theta {tag}", sc.read(THETA, offset=s, count=ln), o.get(oracle.THETA)[sl])
        assert_close_exact(f"v {tag}", sc.read(V, offset=s, count=ln), o.get(oracle.V)[sl])
        for w in range(W):
            assert_close_exact(f"u[{w}] {tag}", sc.read(U, w, offset=s, count=ln),
                               o.get(oracle.U, w)[sl])
            assert_close_exact(f"e[{w}] {tag}", sc.read(E, w, offset=s, count=ln),
                               o.get(oracle.E, w)[sl])
        nw = (ln + 31) // 32
        words = sc.read(MASK, offset=s // 32, count=nw)
        ref = oracle.pack_bits(m_gen[sl])
        if not np.array_equal(words, ref):
            bad = np.nonzero(words != ref)[0]
            raise AssertionError(f"mask {tag}: {bad.size} words differ, first word {bad[0]}")
        ga, gb = np.searchsorted(gidx, [s, s + ln])
        oa, ob = np.searchsorted(oidx, [s, s + ln])
        assert np.array_equal(gidx[ga:gb], oidx[oa:ob]), f"idx {tag}"
        for gv, ov, w in zip(g_vals, o_vals, list(range(W)) + [-1]):
            assert_close_exact(f"vals[{w}] {tag}", gv[ga:gb], ov[oa:ob])
        pos += ln


def sample_chunks(wl, n_extra: int = 4, seed: int = 0) -> list[int]:
    """Chunks at both ends, at every shard boundary and a few seeded others."""
    nch = -(-wl.N // wl.chunk)
    q = -(-nch // wl.W)
    ids = {0, 1, nch - 2, nch - 1}
    for w in range(1, wl.W):
        if w * q < nch:
            ids |= {w * q - 1, w * q}
    rng = np.random.default_rng(seed)
    ids |= set(int(x) for x in rng.integers(0, nch, n_extra))
    return sorted(i for i in ids if 0 <= i < nch)


_POPC8 = np.array([bin(i).count("1") for i in range(256)], np.uint8)


def check_full_mask(g: DeviceRun, r: OracleRun | None = None) -> None:
    """Properties over the full size: every chunk of the next mask carries
    exactly k_c bits, none past N; the last step's coordinate list is strictly
    increasing and has K entries.  Chunk boundaries come from the oracle's
    layout table when given (per-tensor chunks), else from C."""
    sc, wl = g.sc, g.wl
    info = sc.info
    words = sc.mask()
    C, N = wl.chunk, wl.N
    nch = info["n_chunks"]
    if N % 32:
        assert (int(words[-1]) >> (N % 32)) == 0, "bits past N"
    per_byte = _POPC8[words.view(np.uint8)]
    if r is not None:
        st, ln, k = r.o.all_chunks()
        assert st.size == nch
        cum = np.concatenate([[0], np.cumsum(per_byte, dtype=np.int64)])
        # chunk starts are multiples of 32, so chunk bit counts are byte sums
        # except a ragged last chunk, which ends at N (no bits past it)
        ends = np.minimum((st + ln + 7) // 8, per_byte.size).astype(np.int64)
        counts = cum[ends] - cum[(st // 8).astype(np.int64)]
        assert np.array_equal(counts, k.astype(np.int64)), "a chunk with the wrong bit count"
    else:
        full = (per_byte[: (nch - 1) * (C // 8)].reshape(nch - 1, C // 8).sum(axis=1, dtype=np.int64)
                if nch > 1 else np.zeros(0))
        assert np.all(full == info["k_full"]), "a full chunk with the wrong bit count"
        assert int(per_byte[(nch - 1) * (C // 8):].sum(dtype=np.int64)) == info["k_last"]
    idx, _ = sc.sparse(-1)
    assert idx.size == info["K"]
    assert np.all(np.diff(idx.astype(np.int64)) > 0)
