"""The pins catch plausible mistakes: each test plants one mistake in a copy of
oracle.c (on the CPU, in a temporary directory), builds it, and requires that
at least one pin from tests/oracle_pins.py fails on it."""
import functools
import os

import pytest

import oracle
from tests import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "residual_sign": ("const double d = p[v] - qv;",
                      "const double d = qv - p[v];"),
    "test_uses_sample_uniform": ("if ((double)u[i] * qx < px)", "if ((double)u[K] * qx < px)"),
    "ratio_transposed": ("if ((double)u[i] * qx < px)", "if ((double)u[i] * px < qx)"),
    "accept_inverted": ("if ((double)u[i] * qx < px)", "if ((double)u[i] * qx > px)"),
    "no_break_at_rejection": ("        j = i;\n        break;", "        j = i;"),
    "bonus_from_wrong_row": ("lbase + (size_t)K * (size_t)V * esz",
                             "lbase + (size_t)(K - 1) * (size_t)V * esz"),
    "temperature_dropped": ("double e = exp(logit_at(row, dtype, v) / T - m);",
                            "double e = exp(logit_at(row, dtype, v) - m);"),
    "unnormalised_p": ("        p[v] /= s;", "        p[v] /= 1.0;"),
    "sample_uses_test_uniform": ("draw_inverse_cdf(w, V, S, (double)u[K]",
                                 "draw_inverse_cdf(w, V, S, (double)u[0]"),
    "residual_from_wrong_q_row": ("const float* qj = dlog ? 0 : q + (size_t)j * (size_t)V;",
                                  "const float* qj = dlog ? 0 : q + (size_t)(j ? j - 1 : 0) * (size_t)V;"),
    "accept_len_off_by_one": ("*len = j + 1;", "*len = j;"),
    "cdf_non_strict": ("if (run > t) {", "if (run >= t && w[v] >= 0.0 && v > 0) {"),
}


@functools.lru_cache(maxsize=None)
def _mutant_lib(name, tmpdir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = os.path.join(tmpdir, f"oracle_{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    return oracle.load_variant(path, os.path.join(tmpdir, f"lib_{name}.so"))


def _pins(verify):
    """A fast subset of the pins, run in order until one fails."""
    pins.check_output_law(verify, 5, 2, 0.8, seed=2, M=4000, tol=1.5e-3)
    pins.check_chisq(verify, 6, 3, 1.0, seed=33, trials=40000)
    pins.check_mean_tokens(verify, 0.6, 3, V=48, B=32, rounds=100)


def test_pins_pass_on_the_oracle():
    _pins(oracle.verify)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path_factory):
    tmpdir = str(tmp_path_factory.getbasetemp())
    lib = _mutant_lib(name, tmpdir)
    verify = functools.partial(oracle.verify, lib=lib)
    with pytest.raises((pins.PinFailure, ValueError, IndexError)):
        _pins(verify)
