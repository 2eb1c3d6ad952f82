"""The oracle's pins catch plausible mistakes in it.

Each case below plants one mistake in a copy of the oracle's C source (a
flipped sign, swapped gate/up halves, a dropped routing weight, a transposed
or wrong index, a missing SwiGLU-grad term, an unstable permutation), builds
the copy on the CPU, puts it in the oracle's place and runs the pins of
``test_oracle_pins.py`` against it: at least one pin must fail for every
mistake.  The committed oracle is untouched; every mutant keeps its memory
accesses inside the arrays it is given.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests import test_oracle_pins as pins

# (name, text in hmm_oracle.c, replacement)
MUTANTS = [
    ("sigmoid sign",
     "return 1.0 / (1.0 + exp(-z));",
     "return 1.0 / (1.0 + exp(z));"),
    ("gate and up swapped",
     "double g = h[j], u = h[I + j];\n    a[j] = g * sigma(g) * u;",
     "double g = h[I + j], u = h[j];\n    a[j] = g * sigma(g) * u;"),
    ("routing weight dropped at combine",
     "yt[c] += wk * o[c];",
     "yt[c] += o[c];"),
    ("down_proj read transposed",
     "o[c] += aj * ld(W2, row + c, dt);",
     "o[c] += aj * ld(W2, w2_off + c * I + j, dt);"),
    ("dgate without the sigma' term",
     "(1.0 + g * (1.0 - sg))",
     "(1.0 + g * sg)"),
    ("dup without g",
     "dH[I + j] = dA[j] * g * sg;",
     "dH[I + j] = dA[j] * sg;"),
    ("dx without the up half",
     "for (int64_t j = 0; j < 2 * I; ++j) acc += dH[j] * ld(W1, row + j, dt);",
     "for (int64_t j = 0; j < I; ++j) acc += dH[j] * ld(W1, row + j, dt);"),
    ("d_topk_weights scaled by the weight",
     "d += ld(dy, t * H + c, dt) * o[c];",
     "d += ld(w, t * K + k, dt) * ld(dy, t * H + c, dt) * o[c];"),
    ("W2Grad without the routing weight",
     "dW2_e[j * H + c] += aj * DO[r * H + c];",
     "dW2_e[j * H + c] += aj * ld(dy, (slots[r] / K) * H + c, dt);"),
    ("W1Grad with the wrong token row",
     "double xi = ld(x, (slots[r] / K) * H + i, dt);",
     "double xi = ld(x, (slots[r] % T) * H + i, dt);"),
    ("permutation not stable inside an expert",
     "slot2row[s] = offsets[e] + seen[e];",
     "slot2row[s] = offsets[e] + (counts[e] - 1 - seen[e]);"),
    ("shared expert's dx from the gate half only",
     "acc += DH[t * 2 * I + j] * ld(Ws1, i * 2 * I + j, dt);",
     "acc += (j < I ? DH[t * 2 * I + j] : 0.0) * ld(Ws1, i * 2 * I + j, dt);"),
    ("shared expert's dWs2 with a transposed output",
     "dWs2[j * H + c] += aj * ld(dy, t * H + c, dt);",
     "dWs2[c * I + j] += aj * ld(dy, t * H + c, dt);"),
    ("up_proj rows read with the stride of I",
     "int64_t row = w1_off + i * 2 * I;",
     "int64_t row = w1_off + i * I;"),
    ("act_grad without the routing weight",
     "acc += dO[c] * ld(W2, row + c, dt);",
     "acc += ld(dy, dy_off + c, dt) * ld(W2, row + c, dt);"),
    ("weight gradients with slot s read as token s mod T",
     "int64_t s = slots[r], t = s / K;",
     "int64_t s = slots[r], t = s % T;"),
]


def _pin_checks():
    """The pins, with their arguments; each raises on a mismatch."""
    return [
        ("route brute force", lambda: pins.test_route_brute_force_sort(300, 6, 64, 3)),
        ("route brute force, repeats", lambda: pins.test_route_brute_force_sort(50, 4, 3, 4)),
        ("dense formulation", lambda: pins.test_forward_matches_dense_formulation(True, 0)),
        ("dense formulation, repeats",
         lambda: pins.test_forward_matches_dense_formulation(False, 1)),
        ("E=1 K=1 torch forward", pins.test_forward_E1_K1_is_plain_swiglu_ffn_torch),
        ("signature probe", pins.test_forward_closed_form_signature_probe),
        ("finite differences", lambda: pins.test_backward_finite_differences(True)),
        ("finite differences, repeats", lambda: pins.test_backward_finite_differences(False)),
        ("E=1 K=1 torch autograd", pins.test_backward_E1_K1_torch_autograd),
        ("d_topk_weights linear response", pins.test_backward_dw_is_exact_linear_response),
        ("shared expert: torch forward", pins.test_shared_forward_is_a_dense_swiglu_ffn_torch),
        ("shared expert: torch autograd", pins.test_shared_backward_matches_torch_autograd),
        ("shared expert: finite differences", pins.test_shared_backward_finite_differences),
        ("shared expert = unit-weight routed expert",
         pins.test_shared_expert_equals_a_routed_expert_with_unit_weight),
    ]


def _build_mutant(tmp_path, old, new):
    with open(os.path.join(os.path.dirname(oracle.__file__), "hmm_oracle.c")) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    c = tmp_path / "mutant.c"
    c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so),
                    str(c), "-lm"], check=True)
    return oracle._configure(ctypes.CDLL(str(so)))


def test_pins_pass_on_the_oracle():
    for name, check in _pin_checks():
        check()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, name, old, new):
    monkeypatch.setattr(oracle, "_lib", _build_mutant(tmp_path, old, new))
    caught = []
    for pin, check in _pin_checks():
        try:
            with np.errstate(all="ignore"):
                check()
        except Exception:  # a failed assertion (or a shape the mutant broke)
            caught.append(pin)
    assert caught, f"no pin catches the mistake: {name}"
