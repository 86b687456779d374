"""CPU reference (oracle) for C = alpha * A * B + beta * C in double precision.

TEST INFRASTRUCTURE ONLY.  Only the test-suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline arm import this package.  The CUDA library and its
Python binding never import it, and it imports nothing from them.

The arithmetic lives in ``oracle_sgemm.c`` (plain C, no CUDA header): the
textbook triple loop of "Optimizing Matrix Multiply on CUDA, Part 1" (section
"Counting the Work") and the row-major naive kernel of "GEMM from Scratch"
(Module 02), widened to double as "Optimizing CUDA matmul, steps 4 to 6"
(section "Five paths, one table") prescribes for its checker.

Every function here is pinned by tests against values the pages and the
mathematics fix (all-ones inputs, identity and permutation matrices, alpha/beta
closed forms, exact integer brute force, dot products, |A||B|), not against
itself.  Parity pinned: yes, for both outputs (Cref and absprod).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_sgemm.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_sgemm.so")

_lib = None
_lock = threading.Lock()


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the C oracle into a shared library with gcc (host only).

    Plain -O2: no -ffast-math, so the double sums keep IEEE semantics.
    """
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           *extra_flags, "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build() -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        compile_oracle()
    return _LIB_PATH


def load_library(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    lib.oracle_sgemm_rows.restype = ctypes.c_int
    lib.oracle_sgemm_rows.argtypes = [
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double,
        ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_default_threads.restype = ctypes.c_int
    lib.oracle_default_threads.argtypes = []
    return lib


def _library() -> ctypes.CDLL:
    """The oracle library; ORACLE_LIB_OVERRIDE names another build of it (the
    mutation tests load deliberately broken copies this way)."""
    global _lib
    with _lock:
        if _lib is None:
            override = os.environ.get("ORACLE_LIB_OVERRIDE")
            _lib = load_library(override if override else build())
        return _lib


def default_threads() -> int:
    """Threads the oracle uses when ``threads=0`` (all online host cores)."""
    return int(_library().oracle_default_threads())


def _as_f32(x, name):
    if x is None:
        return None
    arr = np.asarray(x)
    if arr.dtype != np.float32:
        raise TypeError(f"{name} must be float32, got {arr.dtype}")
    return arr


def _ptr(a):
    return None if a is None else a.ctypes.data


def sgemm_ref_flat(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, rows=None,
                   threads=0, want_absprod=True, lib=None):
    """Reference rows of alpha*A*B + beta*C on flat float32 buffers.

    ``A``, ``B`` and ``C`` are 1-D float32 arrays holding row-major matrices
    with leading dimensions ``lda``, ``ldb``, ``ldc`` (elements).  ``rows`` is
    an iterable of row indices (default: all M rows).  Returns
    ``(Cref, absprod)`` as float64 arrays of shape (len(rows), N); absprod is
    None when ``want_absprod`` is false.
    """
    lib = lib or _library()
    A = _as_f32(A, "A")
    B = _as_f32(B, "B")
    C = _as_f32(C, "C")
    for name, arr in (("A", A), ("B", B), ("C", C)):
        if arr is not None and not arr.flags.c_contiguous:
            raise ValueError(f"{name} must be contiguous")
    rows_arr = (np.arange(M, dtype=np.int64) if rows is None
                else np.ascontiguousarray(np.asarray(rows, dtype=np.int64)))
    out = np.empty((rows_arr.size, N), dtype=np.float64)
    absprod = (np.empty((rows_arr.size, N), dtype=np.float64)
               if want_absprod else None)
    rc = lib.oracle_sgemm_rows(
        int(M), int(N), int(K), float(alpha),
        _ptr(A), int(lda), _ptr(B), int(ldb),
        float(beta), _ptr(C), int(ldc),
        rows_arr.ctypes.data, int(rows_arr.size),
        out.ctypes.data, _ptr(absprod), int(threads))
    if rc != 0:
        raise RuntimeError(f"oracle_sgemm_rows failed with code {rc}")
    return out, absprod


def sgemm_ref(A, B, C=None, alpha=1.0, beta=0.0, rows=None, threads=0,
              want_absprod=True):
    """Reference for 2-D float32 arrays (copied to row-major contiguous form).

    For leading dimensions larger than the row length use ``sgemm_ref_flat``.
    """
    A = np.ascontiguousarray(_as_f32(A, "A"))
    B = np.ascontiguousarray(_as_f32(B, "B"))
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    Cf = None
    if beta != 0.0:
        if C is None:
            raise ValueError("C is required when beta != 0")
        Cf = np.ascontiguousarray(_as_f32(C, "C"))
        if Cf.shape != (M, N):
            raise ValueError("C has the wrong shape")
        Cf = Cf.reshape(-1)
    return sgemm_ref_flat(M, N, K, alpha, A.reshape(-1), max(1, K),
                          B.reshape(-1), max(1, N), beta, Cf, max(1, N),
                          rows=rows, threads=threads, want_absprod=want_absprod)


def error_bound(absprod, C, alpha, beta, K, bias=None):
    """Elementwise FP32 bound 2*K*2^-24*(|alpha|*(|A||B|)_ij + |beta|*|C_ij|).

    K is taken as max(K, 3).  A K-term FP32 dot product followed by the
    epilogue passes each product through at most K + 2 roundings, an error of
    at most gamma_{K+2} = (K+2)u/(1-(K+2)u) relative to |alpha|(|A||B|)_ij,
    and the beta term through at most two.  2*K*u covers gamma_{K+2} for every
    K >= 3 (u = 2^-24), so smaller K use the K = 3 constant.

    With a bias (a length-N vector added to every row) each term passes
    through one more rounding, so |bias_j| joins the sum and K is taken as
    max(K, 4) (2*K*u covers gamma_{K+3} for K >= 4).  ReLU is 1-Lipschitz and
    exact, so the same bound holds after it.
    """
    keff = max(int(K), 4 if bias is not None else 3)
    u = 2.0 ** -24
    bound = np.abs(alpha) * absprod
    if beta != 0.0 and C is not None:
        bound = bound + np.abs(beta) * np.abs(np.asarray(C, dtype=np.float64))
    if bias is not None:
        bound = bound + np.abs(np.asarray(bias, dtype=np.float64))[None, :]
    return 2.0 * keff * u * bound


ACT_NONE, ACT_RELU = 0, 1


def apply_epilogue(ref, bias=None, activation=ACT_NONE):
    """act(ref + bias) in double, on an oracle result ref (rows x N).

    "GEMM from Scratch", end of Module 08 ("When to just call the library"):
    fusing an epilogue or activation into the product is the reason given for
    writing one's own GEMM.  The pages name no activation; ReLU is taken as
    x < 0 ? 0 : x, so NaN passes through.  The bias is a vector of N values,
    bias[j] added to every row's column j.
    """
    out = np.array(ref, dtype=np.float64, copy=True)
    if bias is not None:
        out = out + np.asarray(bias, dtype=np.float64)[None, :]
    if activation == ACT_RELU:
        out = np.where(out < 0.0, 0.0, out)
    elif activation != ACT_NONE:
        raise ValueError(f"unknown activation {activation}")
    return out
