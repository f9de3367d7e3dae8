"""Parameter layouts and synthetic-gradient recipes of the SCAPE workloads.

The SCAPE pages train GPT-345M (GPT-2-medium) and Llama-style 500M / 1.8B
models under data parallelism ("SCAPE: Accurate and Efficient LLM Training with
Extreme Sparse Communication", abstract; gist.science technical summary, §4).
No dataset or trained weight is used here: each workload is the model's flat
parameter layout (the concatenation of its tensors, in order) with seeded
gradients drawn by ``synth_core.h``.  Nothing in this module computes any part
of the optimizer.

Shapes follow the PyTorch ``[out_features, in_features]`` convention, so the
per-tensor scale ``sigma = 0.02 / sqrt(fan_in)`` takes ``fan_in`` as the last
dimension (the length, for 1-D tensors).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SYN_GAUSS = 0
SYN_STUDENT_Q = 1


@dataclass(frozen=True)
class Workload:
    name: str
    tensors: tuple  # ((name, shape), ...)
    W: int
    chunk: int
    densities: tuple
    steps: int
    kind: int = SYN_GAUSS
    sigma: float | None = None  # one sigma for every tensor; None -> 0.02/sqrt(fan_in)
    seed: int = 0
    beta1: float = 0.9
    beta2: float = 0.95
    lr: float = 1e-3
    wd: float = 0.1
    eps: float = 1e-8
    description: str = field(default="", compare=False)

    @property
    def numel(self) -> list[int]:
        return [int(np.prod(s)) for _, s in self.tensors]

    @property
    def N(self) -> int:
        return sum(self.numel)

    def starts(self) -> np.ndarray:
        """uint64[n_tensors + 1]: flat offset of each tensor, then N."""
        return np.concatenate([[0], np.cumsum(self.numel)]).astype(np.uint64)

    def sigmas(self) -> np.ndarray:
        """float32[n_tensors]: the gradient scale of each tensor."""
        if self.sigma is not None:
            return np.full(len(self.tensors), self.sigma, dtype=np.float32)
        return np.array([0.02 / math.sqrt(s[-1]) for _, s in self.tensors], dtype=np.float32)


def _gpt2_medium():
    d, ff, vocab, ctx, layers = 1024, 4096, 50257, 1024, 24
    t = [("wte", (vocab, d)), ("wpe", (ctx, d))]
    for l in range(layers):
        p = f"h{l}."
        t += [
            (p + "ln1.w", (d,)), (p + "ln1.b", (d,)),
            (p + "c_attn.w", (3 * d, d)), (p + "c_attn.b", (3 * d,)),
            (p + "c_proj.w", (d, d)), (p + "c_proj.b", (d,)),
            (p + "ln2.w", (d,)), (p + "ln2.b", (d,)),
            (p + "c_fc.w", (ff, d)), (p + "c_fc.b", (ff,)),
            (p + "c_proj2.w", (d, ff)), (p + "c_proj2.b", (d,)),
        ]
    t += [("ln_f.w", (d,)), ("ln_f.b", (d,))]
    return tuple(t)


def _llama(d, ff, layers, vocab=32000):
    t = [("emb", (vocab, d))]
    for l in range(layers):
        p = f"l{l}."
        t += [
            (p + "attn_norm", (d,)),
            (p + "q", (d, d)), (p + "k", (d, d)), (p + "v", (d, d)), (p + "o", (d, d)),
            (p + "mlp_norm", (d,)),
            (p + "gate", (ff, d)), (p + "up", (ff, d)), (p + "down", (d, ff)),
        ]
    t += [("final_norm", (d,)), ("lm_head", (vocab, d))]
    return tuple(t)


WORKLOADS = {
    "flat-2^20-w4": Workload(
        "flat-2^20-w4", (("flat", (1 << 20,)),), W=4, chunk=4096, densities=(0.10,), steps=5,
        sigma=1e-3,
        description="one fp32 tensor of 2^20, W=4, density 0.10, chunk 4096, 5 steps"),
    "flat-2^26-w8-ties": Workload(
        "flat-2^26-w8-ties", (("flat", (1 << 26,)),), W=8, chunk=65536, densities=(0.10, 0.01),
        steps=20, kind=SYN_STUDENT_Q, sigma=1e-3,
        description="one fp32 tensor of 2^26, W=8, densities 0.10/0.01, chunk 65536, "
                    "Student-t(3) means, grads on a 2^-14 grid (heavy ties), 20 steps"),
    "gpt2-medium-w8": Workload(
        "gpt2-medium-w8", _gpt2_medium(), W=8, chunk=65536, densities=(0.01,), steps=10,
        description="GPT-2-medium layout (354.8M params, 292 tensors), W=8, density 0.01, "
                    "chunk 65536, 10 steps"),
    "llama-500m-w8": Workload(
        "llama-500m-w8", _llama(1280, 3456, 24), W=8, chunk=65536, densities=(0.01, 0.10),
        steps=10,
        description="Llama-style 557.8M layout (219 tensors), W=8, densities 0.01/0.10, "
                    "chunk 65536, 10 steps"),
    "llama-1.8b-w4": Workload(
        "llama-1.8b-w4", _llama(2048, 5632, 32), W=4, chunk=65536, densities=(0.01,), steps=10,
        description="Llama-style 1775.4M layout (291 tensors), W=4, density 0.01 (99% sparsity), "
                    "chunk 65536, 10 steps"),
}

# A small flat layout for profiler captures: state and gradients ~2 GB on the
# device (well above L2), same per-worker shape as the 1.8B layout.
WORKLOADS["profile-2^25-w4"] = Workload(
    "profile-2^25-w4", (("flat", (1 << 25,)),), W=4, chunk=65536, densities=(0.01,), steps=3,
    sigma=1e-3, description="one tensor of 2^25, W=4, density 0.01, chunk 65536 (profiling case)")

# Half of it: a second capture point, to show the kernel's DRAM bytes per
# coordinate do not change with the size.
WORKLOADS["profile-2^24-w4"] = Workload(
    "profile-2^24-w4", (("flat", (1 << 24,)),), W=4, chunk=65536, densities=(0.01,), steps=3,
    sigma=1e-3, description="one tensor of 2^24, W=4, density 0.01, chunk 65536 (profiling case)")

# The workload the throughput line is quoted on.
BENCH_WORKLOAD = "llama-1.8b-w4"


def tiny(N: int, W: int, chunk: int, density: float, kind: int = SYN_GAUSS, seed: int = 0,
         sigma: float = 1e-3, **hyper) -> Workload:
    """A one-tensor workload for unit and edge-case tests."""
    return Workload(f"tiny-{N}-w{W}", (("flat", (N,)),), W=W, chunk=chunk, densities=(density,),
                    steps=1, kind=kind, sigma=sigma, seed=seed, **hyper)
