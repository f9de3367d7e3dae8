"""Python binding of libscape (argument marshalling only).

Every step of the optimizer runs in the CUDA kernels of ``libscape.so``; this
module only loads the library, converts arguments and raises on error codes.
There is no CPU path: if the library is missing, importing the binding fails.
Function names follow the C ABI in ``include/scape.h``.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libscape.so")
DEBUG_LIB_PATH = os.path.join(HERE, "libscape_debug.so")

SCAPE_OK, SCAPE_EINVAL, SCAPE_ENOMEM, SCAPE_ECUDA, SCAPE_ESTATE = 0, -1, -2, -3, -4
THETA, V, U, E, MASK, STEP = 0, 1, 2, 3, 4, 5
PHASES = ("select_boot", "step", "select_fallback", "h2d")

# Symbols declared in include/scape.h (checked by the ABI test).
CHUNK_PER_TENSOR, RESIDUAL_HOST, UNION_MASK = 1, 2, 4
EXPORTS = ("scape_create", "scape_create_ex", "scape_step", "scape_step_host", "scape_mask",
           "scape_mask_async", "scape_destroy",
           "scape_info", "scape_read_state", "scape_load_state", "scape_read_sparse",
           "scape_last_error", "scape_profile", "scape_profile_read", "scape_step_noalloc",
           "scape_dense_adams_step", "scape_mask_stats", "scape_unpack")


class ScapeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class _Layout(ctypes.Structure):
    _fields_ = [("n_tensors", ctypes.c_uint32), ("numel", ctypes.POINTER(ctypes.c_uint64)),
                ("chunk", ctypes.c_uint32)]


class _Info(ctypes.Structure):
    _fields_ = [("N", ctypes.c_uint64), ("W", ctypes.c_uint32), ("chunk", ctypes.c_uint32),
                ("n_chunks", ctypes.c_uint64), ("chunks_per_worker", ctypes.c_uint64),
                ("k_full", ctypes.c_uint32), ("k_last", ctypes.c_uint32), ("K", ctypes.c_uint64),
                ("mask_words", ctypes.c_uint64), ("step", ctypes.c_int64),
                ("device_bytes", ctypes.c_uint64), ("select_fallbacks", ctypes.c_uint64),
                ("flags", ctypes.c_uint32), ("host_bytes", ctypes.c_uint64),
                ("checks_compiled", ctypes.c_uint32), ("check_code", ctypes.c_uint32),
                ("check_count", ctypes.c_uint32), ("check_where", ctypes.c_uint64)]


class StepBuffers(ctypes.Structure):
    """scape_step_buffers: caller-owned state for scape_step_noalloc."""
    _fields_ = [("layout", ctypes.POINTER(_Layout)), ("W", ctypes.c_int),
                ("density", ctypes.c_double), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("lr", ctypes.c_float), ("wd", ctypes.c_float),
                ("eps", ctypes.c_float), ("theta", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("u", ctypes.c_void_p), ("e", ctypes.c_void_p), ("row_stride", ctypes.c_uint64),
                ("mask_prev", ctypes.c_void_p), ("mask_next", ctypes.c_void_p),
                ("vals", ctypes.c_void_p), ("vals_stride", ctypes.c_uint64),
                ("bbar", ctypes.c_void_p), ("idx", ctypes.c_void_p), ("first_step", ctypes.c_int)]


_lib = None
_libs: dict = {}


def load_library(path: str = LIB_PATH):
    """Load libscape (or another build of it, e.g. DEBUG_LIB_PATH) once."""
    global _lib
    if path == LIB_PATH and _lib is not None:
        return _lib
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m sparse_communication_distributed_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, u64, i32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int
    lib.scape_create.argtypes = [ctypes.POINTER(_Layout), i32, ctypes.c_double, ctypes.c_float,
                                 ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                 ctypes.POINTER(vp)]
    lib.scape_create_ex.argtypes = [ctypes.POINTER(_Layout), i32, ctypes.c_double,
                                    ctypes.c_float, ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                    ctypes.c_float, ctypes.c_uint32, ctypes.POINTER(vp)]
    lib.scape_step.argtypes = [vp, ctypes.POINTER(vp), vp]
    lib.scape_step_host.argtypes = [vp, ctypes.POINTER(vp), vp]
    lib.scape_mask.argtypes = [vp, vp]
    lib.scape_mask_async.argtypes = [vp, vp, vp]
    lib.scape_destroy.argtypes = [vp]
    lib.scape_destroy.restype = None
    lib.scape_info.argtypes = [vp, ctypes.POINTER(_Info)]
    lib.scape_read_state.argtypes = [vp, i32, i32, vp, u64, u64]
    lib.scape_load_state.argtypes = [vp, i32, i32, vp, u64, u64]
    lib.scape_read_sparse.argtypes = [vp, i32, vp, vp, u64, u64, ctypes.POINTER(u64)]
    lib.scape_last_error.argtypes = [vp]
    lib.scape_last_error.restype = ctypes.c_char_p
    lib.scape_profile.argtypes = [vp, i32]
    lib.scape_profile_read.argtypes = [vp, ctypes.POINTER(ctypes.c_double),
                                       ctypes.POINTER(ctypes.c_uint32)]
    lib.scape_step_noalloc.argtypes = [ctypes.POINTER(StepBuffers), ctypes.POINTER(vp), vp]
    lib.scape_mask_stats.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64 * 3)]
    lib.scape_unpack.argtypes = [vp, vp, u64, vp, u64, vp, vp]
    f32 = ctypes.c_float
    lib.scape_dense_adams_step.argtypes = [vp, vp, vp, ctypes.POINTER(vp), i32, u64, f32, f32, f32,
                                           f32, f32, vp]
    _libs[path] = lib
    if path == LIB_PATH:
        _lib = lib
    return lib


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(stream, int):
        return stream or None
    return stream.cuda_stream or None


def _ptr(x) -> int:
    """Address of a torch tensor or a numpy array."""
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


class Scape:
    """One SCAPE optimizer instance (a libscape handle)."""

    def __init__(self, numel, chunk: int, W: int, density: float, beta1: float = 0.9,
                 beta2: float = 0.95, lr: float = 1e-3, wd: float = 0.1, eps: float = 1e-8,
                 flags: int = 0, lib_path: str = LIB_PATH):
        self.lib = load_library(lib_path)
        arr = np.ascontiguousarray(numel, dtype=np.uint64)
        lay = _Layout(arr.size, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), chunk)
        h = ctypes.c_void_p()
        rc = self.lib.scape_create_ex(ctypes.byref(lay), W, density, beta1, beta2, lr, wd, eps,
                                      flags, ctypes.byref(h))
        if rc != SCAPE_OK:
            raise ScapeError(rc, self.lib.scape_last_error(None).decode())
        self.h = h
        self.info = self._info()

    @classmethod
    def for_workload(cls, wl, density: float, flags: int = 0, lib_path: str = LIB_PATH) -> "Scape":
        return cls(wl.numel, wl.chunk, wl.W, density, wl.beta1, wl.beta2, wl.lr, wl.wd, wl.eps,
                   flags=flags, lib_path=lib_path)

    def _check(self, rc: int) -> None:
        if rc != SCAPE_OK:
            raise ScapeError(rc, self.lib.scape_last_error(self.h).decode())

    def _info(self) -> dict:
        inf = _Info()
        self._check(self.lib.scape_info(self.h, ctypes.byref(inf)))
        return {f: getattr(inf, f) for f, _ in _Info._fields_}

    def close(self) -> None:
        if getattr(self, "h", None):
            self.lib.scape_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def N(self) -> int:
        return self.info["N"]

    @property
    def K(self) -> int:
        """Compact values per worker of the last step (fixed unless UNION_MASK)."""
        if self.info["flags"] & UNION_MASK:
            return self._info()["K"]
        return self.info["K"]

    @property
    def step_count(self) -> int:
        return self._info()["step"]

    def step(self, grads, stream=None) -> None:
        """grads: W device tensors of N bf16 (16-byte aligned)."""
        arr = (ctypes.c_void_p * len(grads))(*[_ptr(g) for g in grads])
        self._check(self.lib.scape_step(self.h, arr, _stream_handle(stream)))

    def step_host(self, grads, stream=None) -> None:
        """grads: W host buffers (numpy uint16 or pinned torch tensors) of N bf16."""
        arr = (ctypes.c_void_p * len(grads))(*[_ptr(g) for g in grads])
        self._check(self.lib.scape_step_host(self.h, arr, _stream_handle(stream)))

    def mask_into(self, out) -> None:
        self._check(self.lib.scape_mask(self.h, _ptr(out)))

    def mask_into_async(self, out, stream) -> None:
        """Stream-ordered copy of M_t into out (pinned host or device tensor of
        mask_words int32); out is written when `stream` reaches the copy."""
        self._check(self.lib.scape_mask_async(self.h, _ptr(out), _stream_handle(stream)))

    def mask(self) -> np.ndarray:
        out = np.empty(self.info["mask_words"], np.uint32)
        self.mask_into(out)
        return out

    def read_into(self, which: int, out, w: int = 0, offset: int = 0) -> None:
        n = out.size if isinstance(out, np.ndarray) else out.numel()
        self._check(self.lib.scape_read_state(self.h, which, w, _ptr(out), offset, n))

    def read(self, which: int, w: int = 0, offset: int = 0, count: int | None = None) -> np.ndarray:
        if which == STEP:
            out = np.empty(1, np.int64)
            self._check(self.lib.scape_read_state(self.h, STEP, 0, out.ctypes.data, 0, 1))
            return out
        total = self.info["mask_words"] if which == MASK else self.N
        count = total - offset if count is None else count
        out = np.empty(count, np.uint32 if which == MASK else np.float32)
        self._check(self.lib.scape_read_state(self.h, which, w, out.ctypes.data, offset, count))
        return out

    def load(self, which: int, src, w: int = 0, offset: int = 0) -> None:
        if isinstance(src, np.ndarray):
            dt = {MASK: np.uint32, STEP: np.int64}.get(which, np.float32)
            src = np.ascontiguousarray(src, dtype=dt)
            n = src.size
        else:
            n = src.numel()
        self._check(self.lib.scape_load_state(self.h, which, w, _ptr(src), offset, n))

    def sparse(self, w: int, offset: int = 0, count: int | None = None):
        """(idx uint32, vals fp32) of the last step's compact buffer of worker
        w (w = -1: the synchronized buffer)."""
        count = self.K - offset if count is None else count
        idx = np.empty(count, np.uint32)
        vals = np.empty(count, np.float32)
        tot = ctypes.c_uint64()
        self._check(self.lib.scape_read_sparse(self.h, w, idx.ctypes.data, vals.ctypes.data,
                                               offset, count, ctypes.byref(tot)))
        return idx, vals

    def mask_stats(self) -> dict:
        """kept, overlap_prev, union_global_topk of the last step (scape_mask_stats)."""
        out = (ctypes.c_uint64 * 3)()
        self._check(self.lib.scape_mask_stats(self.h, ctypes.byref(out)))
        return {"kept": out[0], "overlap_prev": out[1], "union_global_topk": out[2]}

    def profile(self, enable: bool) -> None:
        self._check(self.lib.scape_profile(self.h, 1 if enable else 0))

    def profile_read(self) -> dict:
        ms = (ctypes.c_double * len(PHASES))()
        n = (ctypes.c_uint32 * len(PHASES))()
        self._check(self.lib.scape_profile_read(self.h, ms, n))
        return {p: (ms[i], n[i]) for i, p in enumerate(PHASES)}


def step_noalloc(numel, chunk: int, W: int, density: float, hyper, buffers: dict, grads,
                 first_step: bool, stream=None) -> None:
    """scape_step_noalloc on caller-owned device tensors.  ``hyper`` is
    (beta1, beta2, lr, wd, eps); ``buffers`` maps theta, v, u, e, mask_prev,
    mask_next, vals, bbar, idx to tensors and row_stride, vals_stride to ints."""
    lib = load_library()
    if len(grads) != W:
        raise ValueError(f"step_noalloc: {len(grads)} gradient buffers for W={W}")
    arr = np.ascontiguousarray(numel, dtype=np.uint64)
    lay = _Layout(arr.size, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), chunk)
    b1, b2, lr, wd, eps = hyper
    sb = StepBuffers(ctypes.pointer(lay), W, density, b1, b2, lr, wd, eps,
                     *[_ptr(buffers[k]) for k in ("theta", "v", "u", "e")], buffers["row_stride"],
                     _ptr(buffers["mask_prev"]), _ptr(buffers["mask_next"]), _ptr(buffers["vals"]),
                     buffers["vals_stride"], _ptr(buffers["bbar"]), _ptr(buffers["idx"]),
                     1 if first_step else 0)
    gp = (ctypes.c_void_p * len(grads))(*[_ptr(g) for g in grads])
    rc = lib.scape_step_noalloc(ctypes.byref(sb), gp, _stream_handle(stream))
    if rc != SCAPE_OK:
        raise ScapeError(rc, lib.scape_last_error(None).decode())


def dense_adams_step(theta, m, v, grads, beta1=0.9, beta2=0.95, lr=1e-3, wd=0.1, eps=1e-8,
                     stream=None) -> None:
    """scape_dense_adams_step on device tensors (theta, m, v fp32; grads W x bf16)."""
    lib = load_library()
    gp = (ctypes.c_void_p * len(grads))(*[_ptr(g) for g in grads])
    rc = lib.scape_dense_adams_step(_ptr(theta), _ptr(m), _ptr(v), gp, len(grads), theta.numel(),
                                    beta1, beta2, lr, wd, eps, _stream_handle(stream))
    if rc != SCAPE_OK:
        raise ScapeError(rc, lib.scape_last_error(None).decode())


def unpack(idx, vals, dense, bad_count=None, stream=None) -> None:
    """scape_unpack on device tensors: dense[idx[r]] = vals[r]."""
    lib = load_library()
    rc = lib.scape_unpack(_ptr(idx), _ptr(vals), idx.numel(), _ptr(dense), dense.numel(),
                          _ptr(bad_count) if bad_count is not None else None,
                          _stream_handle(stream))
    if rc != SCAPE_OK:
        raise ScapeError(rc, lib.scape_last_error(None).decode())
