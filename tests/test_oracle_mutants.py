"""Mutation check of the oracle pins.

Each case copies the oracle source, plants one plausible mistake in the copy
(a dropped k term, a wrong sign, a transposed operand, the wrong scalar on C,
an ignored leading dimension, a signed |A||B|), builds it on the CPU and runs
the pin suite against it in a separate process.  The pins must reject every
mutant; the unmodified oracle passes the same suite (test_oracle.py).
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle_sgemm.c")

MUTANTS = {
    "drop_last_k": ("for (int64_t k = 0; k < job->K; ++k)",
                    "for (int64_t k = 0; k < job->K - 1; ++k)"),
    "wrong_sign": ("acc[j] += a * b;", "acc[j] -= a * b;"),
    "transposed_a": ("job->A[i * job->lda + k]", "job->A[k * job->lda + i]"),
    "alpha_on_c": ("v += job->beta * (double)job->C", "v += job->alpha * (double)job->C"),
    "ignores_ldb": ("job->B + k * job->ldb", "job->B + k * job->N"),
    "signed_absprod": ("abs_acc[j] += abs_a * fabs(b);", "abs_acc[j] += a * b;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mutant_src = tmp_path / "oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    oracle.compile_oracle(str(mutant_src), str(lib))
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(lib))
    proc = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle.py")],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert proc.returncode != 0, f"mutant {name} passed every pin:\n{proc.stdout[-2000:]}"
