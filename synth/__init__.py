"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

``synth_core.h`` defines the generator once; ``libscape_synth_cpu.so`` (gcc)
and ``libscape_synth_gpu.so`` (nvcc) are its two builds.  The CPU build feeds
the oracle, the GPU build fills device buffers for the CUDA path, and a GPU
test checks that the two agree bit for bit.  This package computes no part of
the optimizer.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .layouts import BENCH_WORKLOAD, SYN_GAUSS, SYN_STUDENT_Q, WORKLOADS, Workload, tiny

HERE = os.path.dirname(os.path.abspath(__file__))
CPU_SO = os.path.join(HERE, "libscape_synth_cpu.so")
GPU_SO = os.path.join(HERE, "libscape_synth_gpu.so")

__all__ = ["Workload", "WORKLOADS", "BENCH_WORKLOAD", "SYN_GAUSS", "SYN_STUDENT_Q", "tiny",
           "build", "cpu", "gpu"]


def build_commands(nvcc: str = "nvcc"):
    """The compile commands of both builds (argument lists)."""
    cpu = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-o", CPU_SO, os.path.join(HERE, "synth_cpu.c"), "-lm"]
    gpu = [nvcc, "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
           "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
           "-Xcompiler", "-fPIC", "-shared", "-o", GPU_SO, os.path.join(HERE, "synth_gpu.cu")]
    return cpu, gpu


def build(gpu_lib: bool = True) -> None:
    cmds = build_commands()
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
             for c in (cmds if gpu_lib else cmds[:1])]
    for c, p in zip(cmds, procs):
        out, _ = p.communicate()
        if p.returncode != 0:
            raise RuntimeError(f"synth build failed: {' '.join(c)}\n{out.decode()}")


_u64p = ctypes.POINTER(ctypes.c_uint64)
_f32p = ctypes.POINTER(ctypes.c_float)
_u16p = ctypes.POINTER(ctypes.c_uint16)


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


class _Cpu:
    def __init__(self):
        if not os.path.exists(CPU_SO):
            build(gpu_lib=False)
        lib = ctypes.CDLL(CPU_SO)
        lib.syn_cpu_grads_range.argtypes = [ctypes.c_int, ctypes.c_uint64, _u64p, _f32p,
                                            ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                            ctypes.c_uint64, ctypes.c_uint64, _u16p]
        lib.syn_cpu_grads_list.argtypes = [ctypes.c_int, ctypes.c_uint64, _u64p, _f32p,
                                           ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                           _u64p, ctypes.c_uint64, _u16p]
        lib.syn_cpu_theta_list.argtypes = [ctypes.c_uint64, _u64p, ctypes.c_uint64, _f32p]
        lib.syn_cpu_normals.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32,
                                        ctypes.c_uint32, ctypes.c_uint64, ctypes.c_uint64, _f32p]
        lib.syn_cpu_logf.argtypes = [ctypes.c_float]
        lib.syn_cpu_logf.restype = ctypes.c_float
        self.lib = lib

    def grads(self, wl: Workload, w: int, t: int, idx: np.ndarray | None = None,
              i0: int = 0, n: int | None = None) -> np.ndarray:
        """bf16 bits (uint16) of worker w's gradient at step t, for the listed
        coordinates (``idx``) or the range [i0, i0+n)."""
        starts, sig = wl.starts(), wl.sigmas()
        if idx is not None:
            idx = np.ascontiguousarray(idx, dtype=np.uint64)
            out = np.empty(idx.size, dtype=np.uint16)
            rc = self.lib.syn_cpu_grads_list(wl.kind, wl.seed, _ptr(starts, _u64p), _ptr(sig, _f32p),
                                             len(sig), w, t, _ptr(idx, _u64p), idx.size,
                                             _ptr(out, _u16p))
        else:
            n = wl.N - i0 if n is None else n
            out = np.empty(n, dtype=np.uint16)
            rc = self.lib.syn_cpu_grads_range(wl.kind, wl.seed, _ptr(starts, _u64p), _ptr(sig, _f32p),
                                              len(sig), w, t, i0, n, _ptr(out, _u16p))
        if rc != 0:
            raise RuntimeError("syn_cpu_grads failed")
        return out

    def theta0(self, wl: Workload, idx: np.ndarray) -> np.ndarray:
        idx = np.ascontiguousarray(idx, dtype=np.uint64)
        out = np.empty(idx.size, dtype=np.float32)
        if self.lib.syn_cpu_theta_list(wl.seed, _ptr(idx, _u64p), idx.size, _ptr(out, _f32p)) != 0:
            raise RuntimeError("syn_cpu_theta_list failed")
        return out

    def normals(self, seed: int, stream: int, w: int, t: int, i0: int, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.float32)
        self.lib.syn_cpu_normals(seed, stream, w, t, i0, n, _ptr(out, _f32p))
        return out

    def logf(self, x: float) -> float:
        return float(self.lib.syn_cpu_logf(x))


class _Gpu:
    """Fills torch CUDA tensors; the tensor table lives on the device."""

    def __init__(self):
        if not os.path.exists(GPU_SO):
            raise RuntimeError(f"{GPU_SO} is missing: run synth.build() (or __graft_entry__.build())")
        lib = ctypes.CDLL(GPU_SO)
        vp = ctypes.c_void_p
        lib.syn_gpu_grads_range.argtypes = [ctypes.c_int, ctypes.c_uint64, vp, vp, ctypes.c_uint32,
                                            ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint64,
                                            ctypes.c_uint64, vp, vp]
        lib.syn_gpu_theta_range.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, vp, vp]
        self.lib = lib
        self._tables = {}

    def _table(self, wl: Workload, device):
        import torch
        key = (wl.name, wl.tensors, str(device))
        if key not in self._tables:
            starts = torch.from_numpy(wl.starts().view(np.int64)).to(device)
            sig = torch.from_numpy(wl.sigmas()).to(device)
            self._tables[key] = (starts, sig)
        return self._tables[key]

    def grads_into(self, wl: Workload, w: int, t: int, out, i0: int = 0, stream=None) -> None:
        """Write worker w's step-t gradient for [i0, i0+out.numel()) into the
        CUDA tensor ``out`` (any 2-byte dtype, contiguous)."""
        import torch
        assert out.is_cuda and out.element_size() == 2 and out.is_contiguous()
        starts, sig = self._table(wl, out.device)
        s = stream if stream is not None else torch.cuda.current_stream(out.device).cuda_stream
        rc = self.lib.syn_gpu_grads_range(wl.kind, wl.seed, starts.data_ptr(), sig.data_ptr(),
                                          len(wl.tensors), w, t, i0, out.numel(), out.data_ptr(), s)
        if rc != 0:
            raise RuntimeError(f"syn_gpu_grads_range failed ({rc})")

    def theta_into(self, wl: Workload, out, i0: int = 0, stream=None) -> None:
        import torch
        assert out.is_cuda and out.dtype == torch.float32 and out.is_contiguous()
        s = stream if stream is not None else torch.cuda.current_stream(out.device).cuda_stream
        if self.lib.syn_gpu_theta_range(wl.seed, i0, out.numel(), out.data_ptr(), s) != 0:
            raise RuntimeError("syn_gpu_theta_range failed")


_cpu = None
_gpu = None


def cpu() -> _Cpu:
    global _cpu
    if _cpu is None:
        _cpu = _Cpu()
    return _cpu


def gpu() -> _Gpu:
    global _gpu
    if _gpu is None:
        _gpu = _Gpu()
    return _gpu
