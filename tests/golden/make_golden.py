"""Writes tests/golden/oracle_regression.json from the oracle alone.

A regression fixture, not a pin: the SCAPE pages print no worked example, so
these values come from the oracle (which the pins in tests/oracle_pins.py tie
to facts outside it).  The fixture makes any later change to the oracle's
arithmetic visible; such a change must name, in its commit message, the
passage of the pages or the reading that justifies it, and regenerate this
file with:

    python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

CASES = [  # (N, W, chunk, density, generator kind, seed, steps)
    (3 * 1024 + 96, 3, 1024, 0.05, synth.SYN_GAUSS, 1, 4),
    (4096, 2, 512, 0.25, synth.SYN_STUDENT_Q, 2, 3),
    (2048 + 7, 4, 512, 1.0, synth.SYN_GAUSS, 3, 3),
]


def digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def run_case(N, W, chunk, density, kind, seed, steps):
    wl = synth.tiny(N, W, chunk, density, kind=kind, seed=seed)
    o = oracle.Oracle.for_workload(wl, density)
    o.set(oracle.THETA, synth.cpu().theta0(wl, o.index))
    for t in range(steps):
        o.step(np.stack([synth.cpu().grads(wl, w, t, idx=o.index) for w in range(W)]))
    out = {"case": [N, W, chunk, density, kind, seed, steps],
           "theta": digest(o.get(oracle.THETA)), "v": digest(o.get(oracle.V)),
           "mask": digest(o.mask(0)), "bbar": digest(o.sparse(-1)[1]),
           "theta_first4": [float(x) for x in o.get(oracle.THETA)[:4]],
           "kept_coordinates_first8": [int(x) for x in o.sparse(-1)[0][:8]]}
    for w in range(W):
        out[f"u{w}"] = digest(o.get(oracle.U, w))
        out[f"e{w}"] = digest(o.get(oracle.E, w))
    return out


def main():
    data = {"about": "SHA-256 of the oracle's state after a few steps on tiny seeded layouts; "
                     "written by tests/golden/make_golden.py (oracle only)",
            "cases": [run_case(*c) for c in CASES]}
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as f:
        json.dump(data, f, indent=1)


if __name__ == "__main__":
    main()
