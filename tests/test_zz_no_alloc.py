"""sgemm_run_skinny_noalloc: the skinny-M product for callers that cannot call
cudaMalloc (code running under a framework allocator that owns the device
memory, loops that must not allocate after start-up).  Its partial sums and
tickets live in a fixed buffer compiled into the library instead of a
workspace allocated on first use.

Checked through the C ABI against the CPU oracle, element by element, within
the FP32 bound the other tests use, on calls in a row (each later call sees
the buffer exactly as the one before left it); then its limits, its quick
return for alpha == 0 and K == 0, and its timeout report
(sgemm_skinny_noalloc_status), with the next call checked again.  This file
is collected last so that a run stopping at the first failure has already run
every other test.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen
import dense_fp32_sgemm_gb300 as sg
import oracle
from tests.checks import assert_within

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT, INVALID_ARG, TIMEOUT = 8, 1, 5


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.build()
    sg.set_plan_override(-1, 0)
    sg.set_wait_timeout_ns(0, -1)
    yield
    sg.set_wait_timeout_ns(0, -1)


def stream():
    return torch.cuda.current_stream().cuda_stream


def noalloc_case(M, N, K, alpha, beta, seed):
    """One call on seeded inputs; returns nothing, asserts the oracle bound."""
    lib = sg.library()
    A = datagen.matrix("uniform", seed, "A", M, K)
    B = datagen.matrix("uniform", seed, "B", K, N)
    C = datagen.matrix("uniform", seed, "C", M, N)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C).cuda() if beta != 0 else torch.full((M * N,), float("nan"),
                                                                 device="cuda")
    st = lib.sgemm_run_skinny_noalloc(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                                      dC.data_ptr(), N, stream())
    assert st == 0, sg.status_string(st)
    assert lib.sgemm_skinny_noalloc_status(stream()) == 0
    got = dC.cpu().numpy().reshape(M, N)
    ref, absprod = oracle.sgemm_ref_flat(M, N, K, alpha, A, K, B, N, beta,
                                         C if beta != 0 else None, N)
    bound = oracle.error_bound(absprod, C.reshape(M, N) if beta != 0 else None, alpha, beta, K)
    assert np.isfinite(got).all()
    assert_within(got, ref, bound, f"noalloc {M}x{N}x{K}")


def test_noalloc_matches_the_oracle_on_calls_in_a_row():
    noalloc_case(16, 8192, 4096, 1.0, 0.0, 2001)
    noalloc_case(7, 3000, 1000, 0.5, 2.0, 2002)
    noalloc_case(1, 8192, 8192, 1.0, 0.0, 2003)
    noalloc_case(16, 8192, 4096, -1.0, 0.5, 2004)


def test_noalloc_quick_return_alpha_zero_and_k_zero():
    lib = sg.library()
    M, N, K = 8, 1000, 300
    C = datagen.matrix("uniform", 2010, "C", M, N)
    for alpha, k in ((0.0, K), (1.0, 0)):
        dA = torch.full((M * max(K, 1),), float("nan"), device="cuda")  # never read
        dB = torch.full((max(K, 1) * N,), float("nan"), device="cuda")
        dC = torch.from_numpy(C).cuda()
        st = lib.sgemm_run_skinny_noalloc(M, N, k, alpha, dA.data_ptr(), max(k, 1),
                                          dB.data_ptr(), N, -1.5, dC.data_ptr(), N, stream())
        assert st == 0, sg.status_string(st)
        assert lib.sgemm_skinny_noalloc_status(stream()) == 0
        got = dC.cpu().numpy().reshape(M, N)
        ref, absprod = oracle.sgemm_ref_flat(M, N, k, alpha, np.zeros(1, np.float32), max(k, 1),
                                             np.zeros(1, np.float32), N, -1.5, C, N)
        bound = oracle.error_bound(absprod, C.reshape(M, N), alpha, -1.5, k)
        assert_within(got, ref, bound, f"noalloc alpha={alpha} K={k}")


def test_noalloc_rejects_requests_beyond_its_buffer():
    lib = sg.library()
    buf = torch.zeros(1 << 16, device="cuda")
    p = buf.data_ptr()
    s = stream()
    # M above 16
    assert lib.sgemm_run_skinny_noalloc(17, 64, 64, 1.0, p, 64, p, 64, 0.0, p, 64, s) == SCRATCH_LIMIT
    # N above 4096 slabs of 256 columns (rejected before any pointer is used)
    n = 4096 * 256 + 1
    assert lib.sgemm_run_skinny_noalloc(1, n, 4, 1.0, p, 4, p, n, 0.0, p, n, s) == SCRATCH_LIMIT
    # lda not a multiple of 4
    assert lib.sgemm_run_skinny_noalloc(4, 64, 63, 1.0, p, 63, p, 64, 0.0, p, 64, s) == SCRATCH_LIMIT
    assert lib.sgemm_run_skinny_noalloc(4, 64, 64, 1.0, p, 65, p, 64, 0.0, p, 64, s) == SCRATCH_LIMIT
    # ldb not a multiple of 4
    assert lib.sgemm_run_skinny_noalloc(4, 63, 64, 1.0, p, 64, p, 63, 0.0, p, 64, s) == SCRATCH_LIMIT
    # A or B 4-byte but not 16-byte aligned
    assert lib.sgemm_run_skinny_noalloc(4, 64, 64, 1.0, p + 4, 64, p, 64, 0.0, p, 64, s) == SCRATCH_LIMIT
    assert lib.sgemm_run_skinny_noalloc(4, 64, 64, 1.0, p, 64, p + 8, 64, 0.0, p, 64, s) == SCRATCH_LIMIT
    # invalid arguments stay invalid
    assert lib.sgemm_run_skinny_noalloc(4, 64, 64, 1.0, p + 2, 64, p, 64, 0.0, p, 64, s) == INVALID_ARG
    assert lib.sgemm_run_skinny_noalloc(4, 64, 64, 1.0, p, 63, p, 64, 0.0, p, 64, s) == INVALID_ARG
    assert sg.status_string(SCRATCH_LIMIT) == "SGEMM_ERR_SCRATCH_LIMIT"
    torch.cuda.synchronize()
    assert (buf == 0).all(), "a rejected call wrote device memory"


def test_noalloc_timeout_is_reported_then_the_next_call_is_correct():
    # The copy producer stops issuing loads at its fourth position, so the
    # bounded waits for the following copies run out (no fault, no hang): the
    # kernel records it in the fixed buffer's error word.
    lib = sg.library()
    M, N, K = 16, 8192, 4096
    A = datagen.matrix("uniform", 2020, "A", M, K)
    B = datagen.matrix("uniform", 2020, "B", K, N)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros(M * N, device="cuda")
    sg.set_wait_timeout_ns(2_000_000, 3)
    try:
        st = lib.sgemm_run_skinny_noalloc(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0,
                                          dC.data_ptr(), N, stream())
        assert st == 0, sg.status_string(st)
        assert lib.sgemm_skinny_noalloc_status(stream()) == TIMEOUT
        assert lib.sgemm_skinny_noalloc_status(stream()) == 0, "the status read did not clear it"
    finally:
        sg.set_wait_timeout_ns(0, -1)
    noalloc_case(M, N, K, 1.0, 0.0, 2020)
    noalloc_case(5, 1000, 777 * 4, 1.0, 0.0, 2021)
