"""SCAPE oracle: plain single-threaded C++ CPU reference of the optimizer step.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline and reference legs of ``bench.py`` may import this package.  It shares no code
with the CUDA path (``sparse_communication_distributed_gb300``) and imports
nothing from it; its only shared input is the seeded generator in ``synth``.

The rule it follows, the readings of the points the SCAPE pages leave open and
the domain restriction (whole chunks) are stated in the header of
``scape_oracle.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "scape_oracle.cpp")
SO = os.path.join(HERE, "libscape_oracle.so")

THETA, V, U, E, A, B = 0, 1, 2, 3, 4, 5


def build_command(src: str = SRC, out: str = SO):
    return ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", "-Wall", "-o", out, src]


def build(src: str = SRC, out: str = SO) -> None:
    r = subprocess.run(build_command(src, out), capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"oracle build failed:\n{r.stdout}{r.stderr}")


_u64p = ctypes.POINTER(ctypes.c_uint64)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f32p = ctypes.POINTER(ctypes.c_float)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)

_libs: dict = {}


def load(path: str = SO):
    """Load (building on first use) an oracle library and declare its ABI."""
    if path in _libs:
        return _libs[path]
    if path == SO and not os.path.exists(SO):
        build()
    lib = ctypes.CDLL(path)
    lib.oracle_create.argtypes = [_u64p, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int,
                                  ctypes.c_double, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                  ctypes.c_float, ctypes.c_float, _u64p, ctypes.c_uint64,
                                  ctypes.c_int]
    lib.oracle_create.restype = ctypes.c_void_p
    lib.oracle_destroy.argtypes = [ctypes.c_void_p]
    lib.oracle_domain_size.argtypes = [ctypes.c_void_p]
    lib.oracle_domain_size.restype = ctypes.c_uint64
    lib.oracle_step_count.argtypes = [ctypes.c_void_p]
    lib.oracle_step_count.restype = ctypes.c_long
    lib.oracle_domain_index.argtypes = [ctypes.c_void_p, _u64p]
    lib.oracle_chunks.argtypes = [ctypes.c_void_p, _u64p, _u32p, _u32p, _i32p]
    lib.oracle_chunks.restype = ctypes.c_uint64
    lib.oracle_step.argtypes = [ctypes.c_void_p, _u16p]
    lib.oracle_all_chunks.argtypes = [ctypes.c_void_p, _u64p, _u64p, _u64p]
    lib.oracle_all_chunks.restype = ctypes.c_uint64
    lib.oracle_get.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, _f32p]
    lib.oracle_set.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, _f32p]
    lib.oracle_get_mask.argtypes = [ctypes.c_void_p, ctypes.c_int, _u8p]
    lib.oracle_set_mask.argtypes = [ctypes.c_void_p, _u8p, ctypes.c_long]
    lib.oracle_get_sparse.argtypes = [ctypes.c_void_p, ctypes.c_int, _f32p, _u64p]
    lib.oracle_get_sparse.restype = ctypes.c_uint64
    lib.oracle_topk.argtypes = [_f32p, ctypes.c_uint32, ctypes.c_uint32, _u8p]
    lib.oracle_dense_adams_step.argtypes = [_f32p, _f32p, _f32p, _u16p, ctypes.c_uint64,
                                            ctypes.c_int, ctypes.c_float, ctypes.c_float,
                                            ctypes.c_float, ctypes.c_float, ctypes.c_float]
    _libs[path] = lib
    return lib


def _p(a, t):
    return a.ctypes.data_as(t)


class Oracle:
    """One oracle instance over a domain of whole chunks (all chunks by default)."""

    def __init__(self, numel, chunk: int, W: int, density: float, beta1=0.9, beta2=0.95,
                 lr=1e-3, wd=0.1, eps=1e-8, chunk_ids=None, lib_path: str = SO,
                 per_tensor: bool = False, union_mask: bool = False):
        self.lib = load(lib_path)
        numel = np.ascontiguousarray(numel, dtype=np.uint64)
        ids = (np.zeros(0, np.uint64) if chunk_ids is None
               else np.ascontiguousarray(chunk_ids, dtype=np.uint64))
        self.h = self.lib.oracle_create(_p(numel, _u64p), numel.size, chunk, W, density, beta1,
                                        beta2, lr, wd, eps, _p(ids, _u64p), ids.size,
                                        (1 if per_tensor else 0) | (2 if union_mask else 0))
        if not self.h:
            raise ValueError("oracle_create rejected its arguments")
        self.W = W
        self.n = int(self.lib.oracle_domain_size(self.h))
        self.index = np.empty(self.n, np.uint64)
        self.lib.oracle_domain_index(self.h, _p(self.index, _u64p))
        nc = int(self.lib.oracle_chunks(self.h, None, None, None, None))
        self.chunk_start = np.empty(nc, np.uint64)
        self.chunk_len = np.empty(nc, np.uint32)
        self.chunk_k = np.empty(nc, np.uint32)
        self.chunk_owner = np.empty(nc, np.int32)
        self.lib.oracle_chunks(self.h, _p(self.chunk_start, _u64p), _p(self.chunk_len, _u32p),
                               _p(self.chunk_k, _u32p), _p(self.chunk_owner, _i32p))

    def all_chunks(self):
        """(start, len, k) of every chunk of the layout, as uint64 arrays."""
        n = int(self.lib.oracle_all_chunks(self.h, None, None, None))
        st, ln, k = (np.empty(n, np.uint64) for _ in range(3))
        self.lib.oracle_all_chunks(self.h, _p(st, _u64p), _p(ln, _u64p), _p(k, _u64p))
        return st, ln, k

    @classmethod
    def for_workload(cls, wl, density: float, chunk_ids=None, lib_path: str = SO,
                     per_tensor: bool = False, union_mask: bool = False):
        return cls(wl.numel, wl.chunk, wl.W, density, wl.beta1, wl.beta2, wl.lr, wl.wd, wl.eps,
                   chunk_ids=chunk_ids, lib_path=lib_path, per_tensor=per_tensor,
                   union_mask=union_mask)

    def __del__(self):
        if getattr(self, "h", None):
            self.lib.oracle_destroy(self.h)
            self.h = None

    @property
    def t(self) -> int:
        return int(self.lib.oracle_step_count(self.h))

    def step(self, grads: np.ndarray) -> None:
        """grads: uint16 bf16 bit patterns, shape (W, n)."""
        g = np.ascontiguousarray(grads, dtype=np.uint16)
        assert g.shape == (self.W, self.n)
        if self.lib.oracle_step(self.h, _p(g, _u16p)) != 0:
            raise RuntimeError("oracle_step failed")

    def get(self, which: int, w: int = 0) -> np.ndarray:
        out = np.empty(self.n, np.float32)
        if self.lib.oracle_get(self.h, which, w, _p(out, _f32p)) != 0:
            raise ValueError("bad field")
        return out

    def set(self, which: int, values: np.ndarray, w: int = 0) -> None:
        v = np.ascontiguousarray(values, dtype=np.float32)
        assert v.size == self.n
        if self.lib.oracle_set(self.h, which, w, _p(v, _f32p)) != 0:
            raise ValueError("bad field")

    def mask(self, which: int = 0) -> np.ndarray:
        """which=0: mask generated by the last step; 1: mask applied in it."""
        out = np.empty(self.n, np.uint8)
        self.lib.oracle_get_mask(self.h, which, _p(out, _u8p))
        return out

    def set_mask(self, m: np.ndarray, t: int) -> None:
        m = np.ascontiguousarray(m, dtype=np.uint8)
        self.lib.oracle_set_mask(self.h, _p(m, _u8p), t)

    def sparse(self, w: int):
        """(flat indices, values) of the last step's compact buffer of worker w
        (w = -1: the synchronized buffer)."""
        cnt = int(self.lib.oracle_get_sparse(self.h, w, None, None))
        vals = np.empty(cnt, np.float32)
        idx = np.empty(cnt, np.uint64)
        self.lib.oracle_get_sparse(self.h, w, _p(vals, _f32p), _p(idx, _u64p))
        return idx, vals


def topk(a: np.ndarray, k: int, lib_path: str = SO) -> np.ndarray:
    """The oracle's selection on one array: uint8 keep-flags."""
    lib = load(lib_path)
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.size, np.uint8)
    if lib.oracle_topk(_p(a, _f32p), a.size, k, _p(out, _u8p)) != 0:
        raise ValueError("oracle_topk rejected its arguments")
    return out


def dense_adams_step(theta: np.ndarray, m: np.ndarray, v: np.ndarray, grads: np.ndarray,
                     beta1=0.9, beta2=0.95, lr=1e-3, wd=0.1, eps=1e-8, lib_path: str = SO) -> None:
    """The oracle's dense AdamS step, in place on fp32 theta, m, v; grads (W, n) bf16 bits."""
    lib = load(lib_path)
    g = np.ascontiguousarray(grads, dtype=np.uint16)
    W, n = g.shape
    for a in (theta, m, v):
        assert a.dtype == np.float32 and a.flags.c_contiguous and a.size == n
    if lib.oracle_dense_adams_step(_p(theta, _f32p), _p(m, _f32p), _p(v, _f32p), _p(g, _u16p), n,
                                   W, beta1, beta2, lr, wd, eps) != 0:
        raise ValueError("oracle_dense_adams_step rejected its arguments")


def pack_bits(m: np.ndarray) -> np.ndarray:
    """0/1 bytes -> uint32 words, bit j of word i = element 32*i + j."""
    m = np.asarray(m, dtype=np.uint8)
    pad = (-m.size) % 32
    if pad:
        m = np.concatenate([m, np.zeros(pad, np.uint8)])
    return np.packbits(m.reshape(-1, 32), axis=1, bitorder="little").view("<u4").ravel()
