"""The oracle's result for each whole benchmark workload, computed once per
test process and shared by the test files that compare a GPU product with it
element by element (about 15 s of host time for all of them on 16 cores)."""
from __future__ import annotations

import functools

import datagen
import oracle


@functools.lru_cache(maxsize=None)
def workload_reference(name: str):
    """(cfg, A, B, C, ref, bound) for workload `name`: ref and bound are
    M x N float64 arrays, bound the elementwise FP32 bound."""
    cfg, A, B, C = datagen.config_inputs(name)
    M, N, K, alpha, beta = cfg["M"], cfg["N"], cfg["K"], cfg["alpha"], cfg["beta"]
    ref, absprod = oracle.sgemm_ref_flat(M, N, K, alpha, A, K, B, N, beta,
                                         C if beta != 0 else None, N)
    Cm = C.reshape(M, N) if beta != 0 else None
    bound = oracle.error_bound(absprod, Cm, alpha, beta, K)
    del absprod
    return cfg, A, B, C, ref, bound
