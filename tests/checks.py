"""Comparison helpers shared by the test files (no GEMM arithmetic here)."""
from __future__ import annotations

import numpy as np


def first_mismatch(got, want, bound, label=""):
    """None if |got - want| <= bound everywhere (and got is finite where want
    is), else a message naming the first offending element, in the style of a
    checker that prints the case, row and column of the first mismatch."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    bound = np.asarray(bound, dtype=np.float64)
    err = np.abs(got - want)
    bad = ~(err <= bound)
    bad |= np.isfinite(want) & ~np.isfinite(got)
    if not bad.any():
        return None
    idx = np.argwhere(bad)[0]
    i = tuple(int(v) for v in idx)
    return (f"{label}: {int(bad.sum())} elements outside the bound; first at "
            f"{i}: got {got[i]!r} want {want[i]!r} |err| {err[i]!r} "
            f"bound {np.broadcast_to(bound, got.shape)[i]!r}")


def assert_within(got, want, bound, label=""):
    msg = first_mismatch(got, want, bound, label)
    assert msg is None, msg
