"""Mutation check of the error-bound pins.

Each case takes the source of ``oracle.error_bound``, plants one plausible
mistake (the beta term dropped, a signed scalar, no floor on K, the wrong
constant, C swapped for |A||B|, the bias left out), and runs the
hand-computed pins of test_oracle.py against the mutant, which must fail
them; the unmodified function passes the same pins.
"""
import inspect
import textwrap

import numpy as np
import pytest

import oracle
from tests.test_oracle import check_bound_pins

SRC = textwrap.dedent(inspect.getsource(oracle.error_bound))

MUTANTS = {
    "drops_beta_term": (
        "        bound = bound + np.abs(beta) * np.abs(np.asarray(C, dtype=np.float64))\n",
        "        pass\n"),
    "signed_beta": ("np.abs(beta) *", "beta *"),
    "signed_alpha": ("np.abs(alpha) * absprod", "alpha * absprod"),
    "no_k_floor": ("max(int(K), 4 if bias is not None else 3)", "int(K)"),
    "same_floor_with_bias": ("4 if bias is not None else 3", "3"),
    "factor_one": ("return 2.0 * keff * u * bound", "return keff * u * bound"),
    "unit_roundoff_2e-23": ("u = 2.0 ** -24", "u = 2.0 ** -23"),
    "absprod_for_c": ("np.abs(np.asarray(C, dtype=np.float64))",
                      "np.abs(np.asarray(absprod, dtype=np.float64))"),
    "drops_bias": (
        "        bound = bound + np.abs(np.asarray(bias, dtype=np.float64))[None, :]\n",
        "        pass\n"),
    "bias_by_row": ("[None, :]", "[:, None]"),
}


def _compile(src):
    ns = {"np": np}
    exec(compile(src, "<error_bound mutant>", "exec"), ns)
    return ns["error_bound"]


def test_unmodified_bound_passes_the_pins():
    check_bound_pins(_compile(SRC))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_bound_mutant(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant = _compile(SRC.replace(old, new))
    with pytest.raises((AssertionError, ValueError, IndexError)):
        check_bound_pins(mutant)
