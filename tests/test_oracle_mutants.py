"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
the pins catch every one of them.  A mutant no pin catches would mean the
oracle's arithmetic at that spot is not pinned to anything outside itself."""
from __future__ import annotations

import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

# (name, original text, planted mistake); each original occurs exactly once.
MUTANTS = [
    ("momentum uses beta2", "o.u[x] = (o.b1 * o.u[x]) + (c1 * g);",
     "o.u[x] = (o.b2 * o.u[x]) + (c1 * g);"),
    ("momentum weight is beta1", "const float c1 = 1.0f - o.b1;", "const float c1 = o.b1;"),
    ("error feedback dropped", "float a = o.e[x] + o.u[x];", "float a = o.u[x];"),
    ("residual sign flipped", "o.e[x] = a - b;", "o.e[x] = b - a;"),
    ("residual keeps everything", "o.e[x] = a - b;", "o.e[x] = a;"),
    ("mean misses 1/W", "o.bbar[p] = s * invW;", "o.bbar[p] = s;"),
    ("workers summed in reverse", "for (int w = 1; w < W; w++) s = s + o.vals[w][p];",
     "s = o.vals[W - 1][p]; for (int w = W - 2; w >= 0; w--) s = s + o.vals[w][p];"),
    ("second moment not squared", "(c2 * (bb * bb))", "(c2 * bb)"),
    ("second moment uses beta1", "o.v[i] = (o.b2 * o.v[i])", "o.v[i] = (o.b1 * o.v[i])"),
    ("eps inside the sqrt", "bb / (std::sqrt(o.v[i]) + o.eps)", "bb / std::sqrt(o.v[i] + o.eps)"),
    ("weight decay dropped", "(o.lr * (q + (o.wd * o.theta[i])))", "(o.lr * q)"),
    ("bbar applied off the mask", "if (o.mask_prev[i]) bb = o.bbar[p++];",
     "if (p < o.bbar.size()) bb = o.bbar[p++];"),
    ("top-k keeps the smallest", "if (kx != ky) return kx > ky;", "if (kx != ky) return kx < ky;"),
    ("ties go to the higher index", "return x < y;", "return x > y;"),
    ("key keeps the sign bit", "return bits & 0x7fffffffu;", "return bits;"),
    ("every chunk owned by worker 0", "ch.owner = (int)(c / q);", "ch.owner = 0;"),
    ("k rounded up", "ch.k = (uint32_t)std::floor(density * (double)ch.len);",
     "ch.k = (uint32_t)std::ceil(density * (double)ch.len);"),
    ("mask not delayed", "if (o.t == 0) {", "if (true) {"),
    ("step-0 mask from zero accumulators (first k of every chunk)", "a0[x] = o.e[x] + un;",
     "a0[x] = 0.0f;"),
    ("step-0 mask drops e + b1*u", "a0[x] = o.e[x] + un;", "a0[x] = c1 * g;"),
    ("step-0 mask drops the residual", "a0[x] = o.e[x] + un;", "a0[x] = un;"),
    ("bias correction added", "float q = bb / (std::sqrt(o.v[i]) + o.eps);",
     "float q = (bb / (1.0f - std::pow(o.b1, (float)(o.t + 1)))) / (std::sqrt(o.v[i]) + o.eps);"),
    ("per-tensor chunks ignore tensor boundaries", "  if (per_tensor) {", "  if (false) {"),
    ("union: every worker ranks the owner's accumulator",
     "select_topk(a.data() + (uint64_t)w * o.n + c.dom0, c.len, c.k, keep.data());",
     "select_topk(a.data() + (uint64_t)c.owner * o.n + c.dom0, c.len, c.k, keep.data());"),
    ("union: the last worker's selection overwrites", "m[i] |= keep[i];", "m[i] = keep[i];"),
    ("union: stale bits not cleared", "for (uint32_t i = 0; i < c.len; i++) m[i] = 0;", ""),
    ("union flag ignored", "if (o.union_mask) union_select(o, a, mask);",
     "if (false) union_select(o, a, mask);"),
    ("dense: mean misses 1/W", "const float gbar = s * invW;", "const float gbar = s;"),
    ("dense: second moment from the gradient", "v[i] = (b2 * v[i]) + (c2 * (m[i] * m[i]));",
     "v[i] = (b2 * v[i]) + (c2 * (gbar * gbar));"),
    ("dense: momentum uses beta2", "m[i] = (b1 * m[i]) + (c1 * gbar);",
     "m[i] = (b2 * m[i]) + (c1 * gbar);"),
    ("dense: weight decay dropped", "theta[i] = theta[i] - (lr * (q + (wd * theta[i])));",
     "theta[i] = theta[i] - (lr * q);"),
]


@pytest.fixture(scope="module")
def mutant_libs(tmp_path_factory):
    src = open(oracle.SRC).read()
    d = tmp_path_factory.mktemp("mutants")
    jobs = []
    for j, (name, old, new) in enumerate(MUTANTS):
        assert src.count(old) == 1, f"mutant '{name}': anchor text not unique in the oracle"
        path = os.path.join(d, f"m{j}.cpp")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        so = os.path.join(d, f"libm{j}.so")
        jobs.append((name, so, subprocess.Popen(oracle.build_command(path, so),
                                                stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    libs = {}
    for name, so, p in jobs:
        out, _ = p.communicate()
        assert p.returncode == 0, f"mutant '{name}' failed to build:\n{out.decode()}"
        libs[name] = so
    return libs


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_catch_mutant(mutant_libs, name):
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mutant_libs[name])
        except AssertionError:
            caught.append(pin.__name__)
            break
    assert caught, f"no pin catches the planted mistake '{name}'"
