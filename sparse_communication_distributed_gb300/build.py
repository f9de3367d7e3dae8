"""Compile libscape.so in-tree for sm_103a (nvcc, one process per source file).

    python -m sparse_communication_distributed_gb300.build [--ptxas-verbose]
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libscape.so")
DEBUG_LIB = os.path.join(HERE, "libscape_debug.so")
SOURCES = ["scape_api.cu", "k_fused.cu", "k_select.cu", "k_dense.cu", "k_maskops.cu",
           "scape_noalloc.cu"]

NVCC_FLAGS = [
    "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
    # IEEE fp32 everywhere: no contraction into FMA, correctly rounded / and sqrt,
    # denormals kept.  The step must reproduce the plain fp32 rule bit for bit.
    "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(ptxas_verbose: bool = False, out: str = LIB, debug_checks: bool = False) -> str:
    """Compile libscape.so; debug_checks builds libscape_debug.so, whose
    kernels check mask-dependent indexes (SCAPE_DEBUG_CHECKS)."""
    if debug_checks and out == LIB:
        out = DEBUG_LIB
    bdir = os.path.join(BUILD, "debug" if debug_checks else "release")
    os.makedirs(bdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if debug_checks:
        extra += ["-DSCAPE_DEBUG_CHECKS"]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    logs = []
    for cmd, p in procs:
        o, _ = p.communicate()
        logs.append(o.decode())
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{o.decode()}")
    link = [nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", out] + objs
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}{r.stderr}")
    if ptxas_verbose:
        print("\n".join(logs))
    return out


if __name__ == "__main__":
    print(build(ptxas_verbose="--ptxas-verbose" in sys.argv,
                debug_checks="--debug-checks" in sys.argv))
