"""SCAPE sparse-communication optimizer step on one GB300 (sm_103a).

The CUDA kernels and the C ABI live in ``csrc/`` and build into
``libscape.so`` (``python -m sparse_communication_distributed_gb300.build``);
``scape.Scape`` is the thin ctypes binding over ``include/scape.h``.
"""
from .scape import (E, MASK, PHASES, STEP, THETA, U, V, Scape, ScapeError, load_library)

__all__ = ["Scape", "ScapeError", "load_library", "THETA", "V", "U", "E", "MASK", "STEP", "PHASES"]
