"""The C ABI without a GPU: libscape.so loads, exports every entry point that
include/scape.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import sparse_communication_distributed_gb300 as pkg
from sparse_communication_distributed_gb300 import build, scape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(scape.LIB_PATH):
        build.build()
    return scape.load_library()


def declared():
    txt = open(os.path.join(ROOT, "include", "scape.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|void|const char\*)\s+(scape_\w+)\(", txt, re.M)))


def test_header_matches_binding():
    assert declared() == sorted(scape.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in declared():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", scape.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r" T (scape_\w+)$", out, re.M))
    assert exported == set(declared()), exported ^ set(declared())


def _create(lib, numel, chunk, W, density, eps=1e-8):
    arr = np.asarray(numel, np.uint64)
    lay = scape._Layout(arr.size, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), chunk)
    h = ctypes.c_void_p(1234)
    rc = lib.scape_create(ctypes.byref(lay), W, density, 0.9, 0.95, 1e-3, 0.1, eps, ctypes.byref(h))
    return rc, h


@pytest.mark.parametrize("numel,chunk,W,density,eps,what", [
    ([1024], 1024, 0, 0.1, 1e-8, "W=0"),
    ([1024], 1024, 65, 0.1, 1e-8, "W=65"),
    ([1024], 1024, 2, 0.0, 1e-8, "density"),
    ([1024], 1024, 2, 1.5, 1e-8, "density"),
    ([1024], 48, 2, 0.1, 1e-8, "chunk"),
    ([1024], 131072, 2, 0.1, 1e-8, "chunk"),
    ([0], 1024, 2, 0.1, 1e-8, "N="),
    ([1 << 31, 1 << 31], 1024, 2, 0.1, 1e-8, "N="),
    ([1024], 1024, 2, 0.1, 0.0, "eps"),
    ([1024], 1024, 2, float("nan"), 1e-8, "density"),
    ([1024], 1024, 2, 0.1, float("nan"), "eps"),
    ([1024], 1024, 2, 0.1, float("inf"), "hyper-parameters"),
])
def test_create_rejects_bad_arguments(lib, numel, chunk, W, density, eps, what):
    rc, h = _create(lib, numel, chunk, W, density, eps)
    assert rc == scape.SCAPE_EINVAL
    assert not h.value
    assert what in lib.scape_last_error(None).decode()


def test_null_handles(lib):
    lib.scape_destroy(None)
    assert lib.scape_step(None, None, None) == scape.SCAPE_EINVAL
    assert lib.scape_mask(None, None) == scape.SCAPE_EINVAL
    assert lib.scape_mask_async(None, None, None) == scape.SCAPE_EINVAL
    assert lib.scape_info(None, None) == scape.SCAPE_EINVAL
    assert lib.scape_read_sparse(None, 0, None, None, 0, 0, None) == scape.SCAPE_EINVAL


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(scape, "_lib", None)
    with pytest.raises(ImportError):
        scape.load_library(str(tmp_path / "missing.so"))
    assert pkg.Scape is scape.Scape


def test_create_ex_rejects_bad_flags(lib):
    arr = np.asarray([100, 64], np.uint64)
    lay = scape._Layout(arr.size, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), 64)
    h = ctypes.c_void_p()
    assert lib.scape_create_ex(ctypes.byref(lay), 2, 0.1, 0.9, 0.95, 1e-3, 0.1, 1e-8, 8,
                               ctypes.byref(h)) == scape.SCAPE_EINVAL
    assert "unknown flags" in lib.scape_last_error(None).decode()
    # per-tensor chunks: a tensor before the last that is not a multiple of 32
    assert lib.scape_create_ex(ctypes.byref(lay), 2, 0.1, 0.9, 0.95, 1e-3, 0.1, 1e-8,
                               scape.CHUNK_PER_TENSOR, ctypes.byref(h)) == scape.SCAPE_EINVAL
    assert "multiple of 32" in lib.scape_last_error(None).decode()


def test_injected_allocation_failure_is_reported(lib, monkeypatch):
    # the first device allocation of scape_create fails: no CUDA call is made,
    # the handle is not returned and the error says what happened
    monkeypatch.setenv("SCAPE_TEST_FAIL_ALLOC", "0")
    rc, h = _create(lib, [4096], 1024, 2, 0.1)
    assert rc == scape.SCAPE_ENOMEM
    assert not h.value
    assert "allocation" in lib.scape_last_error(None).decode()


def _noalloc(lib, numel, hyper=(0.9, 0.95, 1e-3, 0.1, 1e-8), chunk=1024, W=2, density=0.1):
    # every argument check of scape_step_noalloc runs before any CUDA call, so
    # null buffers are fine here: the call must fail on the argument first
    arr = np.asarray(numel, np.uint64)
    lay = scape._Layout(arr.size, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), chunk)
    b1, b2, lr, wd, eps = hyper
    sb = scape.StepBuffers(ctypes.pointer(lay), W, density, b1, b2, lr, wd, eps,
                           None, None, None, None, 0, None, None, None, 0, None, None, 1)
    return lib.scape_step_noalloc(ctypes.byref(sb), None, None)


@pytest.mark.parametrize("numel,hyper,what", [
    ([(1 << 64) - 1, 2], (0.9, 0.95, 1e-3, 0.1, 1e-8), "tensor too large"),
    ([1 << 32, 1 << 32], (0.9, 0.95, 1e-3, 0.1, 1e-8), "N must be"),
    ([1024], (float("nan"), 0.95, 1e-3, 0.1, 1e-8), "hyper-parameters"),
    ([1024], (0.9, 0.95, float("inf"), 0.1, 1e-8), "hyper-parameters"),
    ([1024], (0.9, 0.95, 1e-3, 0.1, 0.0), "eps"),
])
def test_noalloc_rejects_bad_arguments(lib, numel, hyper, what):
    assert _noalloc(lib, numel, hyper) == scape.SCAPE_EINVAL
    assert what in lib.scape_last_error(None).decode()


@pytest.mark.parametrize("hyper", [(float("nan"), 0.95, 1e-3, 0.1, 1e-8),
                                   (0.9, 0.95, 1e-3, float("inf"), 1e-8),
                                   (0.9, 0.95, 1e-3, 0.1, 0.0)])
def test_dense_rejects_bad_hyper_parameters(lib, hyper):
    # aligned placeholder addresses: the call must fail on the hyper-parameters
    # before anything touches them or launches
    fake = ctypes.c_void_p(1 << 20)
    grads = (ctypes.c_void_p * 2)(1 << 21, 1 << 22)
    b1, b2, lr, wd, eps = hyper
    rc = lib.scape_dense_adams_step(fake, fake, fake, grads, 2, 1024, b1, b2, lr, wd, eps, None)
    assert rc == scape.SCAPE_EINVAL
    assert "hyper-parameters" in lib.scape_last_error(None).decode()



def test_noalloc_rejects_host_buffers(lib):
    # host memory in every buffer (aligned, non-null): rejected as not device
    # memory before anything is enqueued; without a GPU the pointer query
    # itself fails, which is reported the same way
    N, W = 1024, 2
    raw = np.zeros(N * 16 + 16, np.float32)
    off = (-raw.ctypes.data % 16) // 4
    host = raw[off:off + N * 16]
    p = host.ctypes.data
    arr = np.asarray([N], np.uint64)
    lay = scape._Layout(1, arr.ctypes.data_as(ctypes.POINTER(ctypes.c_uint64)), 1024)
    sb = scape.StepBuffers(ctypes.pointer(lay), W, 0.1, 0.9, 0.95, 1e-3, 0.1, 1e-8,
                           p, p + 4096, p + 8192, p + 16384, N, p + 24576, p + 28672,
                           p + 32768, N, p + 40960, p + 45056, 1)
    grads = (ctypes.c_void_p * W)(p + 49152, p + 53248)
    assert lib.scape_step_noalloc(ctypes.byref(sb), grads, None) == scape.SCAPE_EINVAL
    assert "device" in lib.scape_last_error(None).decode()
