"""Every chunk of the full-size layouts against the oracle, bit for bit.

The sampled full-size tests compare a few whole chunks; this file compares all
of them.  The GPU runs the layout's whole step count in the launch
configuration the bench times, reading M_t back after every step.  The oracle
then runs over groups of consecutive whole chunks: its domain restriction (the
rule touches one coordinate across workers, the selection one chunk) makes a
group's run give, chunk for chunk, what a run over the whole layout gives.
Many groups run at once, each an independent single-threaded oracle instance
in its own thread (the C++ oracle releases the GIL), fed the same gradient
bytes: the GPU build of the seeded generator fills the group's coordinate
range (the generator's two builds are checked equal in test_gpu_parity, and
again here on a slice of every group).

Compared, for every chunk: the new mask M_t after every step; after the last
step theta, v, u_w and e_w, every worker's compact values, bbar and the
coordinate list.  Besides the six config/density cases of the partitioned rule
on flat chunks, three variants run at full size: per-tensor chunks, residuals
in host memory and the non-partitioned union (whose compact entries are
located by coordinate, since their packed positions depend on every chunk).
Host time is printed per case (run pytest with -rP).
"""
import os
import threading
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle  # noqa: E402
import synth  # noqa: E402
from gpu_harness import DeviceRun, OracleRun, assert_close_exact, check_full_mask  # noqa: E402
from sparse_communication_distributed_gb300 import E, THETA, U, V  # noqa: E402
from sparse_communication_distributed_gb300.scape import (CHUNK_PER_TENSOR, RESIDUAL_HOST,  # noqa: E402
                                                          UNION_MASK)

pytestmark = pytest.mark.gpu

FULL = [("flat-2^26-w8-ties", 0.10, 0), ("flat-2^26-w8-ties", 0.01, 0), ("gpt2-medium-w8", 0.01, 0),
        ("llama-500m-w8", 0.01, 0), ("llama-500m-w8", 0.10, 0), ("llama-1.8b-w4", 0.01, 0),
        # the variants at full size: per-tensor chunks, residuals in host memory, the
        # non-partitioned union (on the heavy-ties layout, where its fallback can fire)
        ("gpt2-medium-w8", 0.01, CHUNK_PER_TENSOR), ("llama-500m-w8", 0.01, RESIDUAL_HOST),
        ("flat-2^26-w8-ties", 0.10, UNION_MASK)]
FLAG_NAMES = {0: "", CHUNK_PER_TENSOR: "-per-tensor", RESIDUAL_HOST: "-host-residuals",
              UNION_MASK: "-union"}

GROUP_COORDS = 1 << 22  # coordinates per oracle group (whole chunks)


def _bits_equal(name: str, got: np.ndarray, ref: np.ndarray) -> None:
    if got.shape != ref.shape or not np.array_equal(got.view(np.uint32), ref.view(np.uint32)):
        assert_close_exact(name, got, ref)  # reports the first difference


@pytest.mark.parametrize("name,density,flags", FULL,
                         ids=[f"{n}-d{d}{FLAG_NAMES[f]}" for n, d, f in FULL])
def test_full_size_every_chunk(name, density, flags):
    wl = synth.WORKLOADS[name]
    W, steps = wl.W, wl.steps
    per_tensor = bool(flags & CHUNK_PER_TENSOR)
    union = bool(flags & UNION_MASK)
    t_start = time.perf_counter()
    g = DeviceRun(wl, density, flags=flags)
    lock = threading.Lock()  # one thread at a time on the GPU and the handle
    try:
        masks = []
        for _ in range(steps):
            g.step()
            masks.append(g.sc.mask())
        probe = oracle.Oracle.for_workload(wl, density, chunk_ids=[0], per_tensor=per_tensor,
                                           union_mask=union)
        st_all, ln_all, k_all = (a.astype(np.int64) for a in probe.all_chunks())
        del probe
        n_ch = st_all.size
        assert n_ch == g.sc.info["n_chunks"]
        if not (per_tensor or union):
            check_full_mask(g)
        base_all = np.concatenate([[0], np.cumsum(k_all)])
        if union:  # packed positions depend on every chunk: locate entries by coordinate
            K = g.sc.K
            gidx = g.sc.sparse(0, count=K)[0].astype(np.uint64)
            assert np.all(np.diff(gidx.astype(np.int64)) > 0)
            gvals = {w: g.sc.sparse(w, count=K)[1] for w in list(range(W)) + [-1]}
        t_gpu = time.perf_counter() - t_start

        def gpu_range(fill, n, dtype):
            buf = torch.empty(n, dtype=dtype, device="cuda")
            fill(buf)
            return buf.cpu().numpy()

        def run_group(ids):
            r = OracleRun(wl, density, chunk_ids=ids, theta0=False, per_tensor=per_tensor,
                          union_mask=union)
            o = r.o
            s0, n = int(o.chunk_start[0]), o.n
            assert int(o.index[-1]) == s0 + n - 1  # consecutive chunks: one coordinate range
            with lock:
                th = gpu_range(lambda b: synth.gpu().theta_into(wl, b, i0=s0), n, torch.float32)
            o.set(oracle.THETA, th)
            w0, nw = s0 // 32, (n + 31) // 32
            for t in range(steps):
                with lock:
                    gr = np.stack([gpu_range(lambda b, w=w: synth.gpu().grads_into(wl, w, t, b, i0=s0),
                                             n, torch.int16).view(np.uint16) for w in range(W)])
                if t == 0:  # the generator's GPU build against its CPU build on a slice
                    m = min(n, 2048)
                    assert np.array_equal(gr[W - 1, :m], synth.cpu().grads(wl, W - 1, 0, i0=s0, n=m))
                o.step(gr)
                ref = oracle.pack_bits(o.mask(0))
                got = masks[t][w0:w0 + nw]
                if not np.array_equal(got, ref):
                    bad = int(np.nonzero(got != ref)[0][0])
                    raise AssertionError(f"{name} step {t}: mask word {w0 + bad} differs "
                                         f"(coordinate {(w0 + bad) * 32})")
            oidx, _ = o.sparse(0)
            with lock:
                dev = {"theta": g.sc.read(THETA, offset=s0, count=n),
                       "v": g.sc.read(V, offset=s0, count=n)}
                for w in range(W):
                    dev[f"u{w}"] = g.sc.read(U, w, offset=s0, count=n)
                    dev[f"e{w}"] = g.sc.read(E, w, offset=s0, count=n)
                if not union:
                    base, cnt = int(base_all[ids[0]]), int(k_all[ids].sum())
                    sp = {w: g.sc.sparse(w, offset=base, count=cnt) for w in list(range(W)) + [-1]}
            if union:
                ga, gb = np.searchsorted(gidx, [s0, s0 + n])
                sp = {w: (gidx[ga:gb], gvals[w][ga:gb]) for w in list(range(W)) + [-1]}
            else:
                assert oidx.size == cnt
            tag = f"{name} chunks {ids[0]}..{ids[-1]}"
            _bits_equal(f"theta {tag}", dev["theta"], o.get(oracle.THETA))
            _bits_equal(f"v {tag}", dev["v"], o.get(oracle.V))
            for w in range(W):
                _bits_equal(f"u[{w}] {tag}", dev[f"u{w}"], o.get(oracle.U, w))
                _bits_equal(f"e[{w}] {tag}", dev[f"e{w}"], o.get(oracle.E, w))
            for w in list(range(W)) + [-1]:
                gi, gv = sp[w]
                assert np.array_equal(gi.astype(np.uint64), oidx), f"idx {tag}"
                _bits_equal(f"vals[{w}] {tag}", gv, o.sparse(w)[1])
            return n

        per = max(1, GROUP_COORDS // wl.chunk)
        groups = [list(range(c, min(c + per, n_ch))) for c in range(0, n_ch, per)]
        threads = len(os.sched_getaffinity(0))
        t1 = time.perf_counter()
        with ThreadPoolExecutor(threads) as ex:
            covered = sum(ex.map(run_group, groups))
        t_oracle = time.perf_counter() - t1
        assert covered == wl.N  # every coordinate, so every chunk, was compared
        print(f"\n{name} density {density}{FLAG_NAMES[flags]}: {n_ch} chunks in {len(groups)} "
              f"oracle groups on {threads} threads, {steps} steps; GPU run + mask reads "
              f"{t_gpu:.1f} s, oracle and comparison {t_oracle:.1f} s, total "
              f"{time.perf_counter() - t_start:.1f} s")
    finally:
        g.close()
