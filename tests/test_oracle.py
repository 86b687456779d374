"""Pins for the CPU oracle, checked against values fixed by the pages and the
mathematics rather than against the oracle itself.

- All-ones operands: every output is K ("Optimizing Matrix Multiply on CUDA,
  Part 1", section "Counting the Work": an output is a K-term dot product).
- Identity / permutation operands: the product reproduces (rows of) the other
  operand, which pins indexing and leading-dimension handling.
- alpha/beta closed forms ("GEMM from Scratch", Module 02 epilogue
  alpha*tmp + beta*C) with power-of-two scalars, so the expected values are
  exact.
- Exact integer brute force: small-integer operands, where Python integer
  arithmetic gives the exact product.
- Dot products (M = N = 1) against math.fsum, the correctly rounded sum.
- |A||B| against numpy's float64 matmul of the absolute values.
- An FP32 library GEMM (numpy / BLAS) stays within the elementwise bound of
  the oracle: the bound and the oracle cannot both be off in a compensating
  way and still agree with an independent implementation.
"""
import math

import numpy as np
import pytest

import datagen
import oracle
from tests.checks import assert_within


def ref(A, B, C=None, alpha=1.0, beta=0.0, **kw):
    return oracle.sgemm_ref(A, B, C, alpha=alpha, beta=beta, **kw)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 9, 33), (64, 48, 130)])
def test_all_ones_gives_k(M, N, K):
    A = np.ones((M, K), np.float32)
    B = np.ones((K, N), np.float32)
    out, absprod = ref(A, B)
    assert (out == K).all()
    assert (absprod == K).all()


def test_all_ones_alpha_beta_closed_form():
    M, N, K = 9, 11, 40
    A = np.ones((M, K), np.float32)
    B = np.ones((K, N), np.float32)
    C = np.full((M, N), 3.0, np.float32)
    out, _ = ref(A, B, C, alpha=0.5, beta=2.0)
    assert (out == 0.5 * K + 2.0 * 3.0).all()


def test_identity_left_and_right():
    rng_b = datagen.uniform_pm1(7, "B", 12 * 9).reshape(12, 9)
    C = datagen.uniform_pm1(7, "C", 12 * 9).reshape(12, 9)
    eye = np.eye(12, dtype=np.float32)
    out, _ = ref(eye, rng_b, C, alpha=0.5, beta=2.0)
    assert (out == 0.5 * rng_b.astype(np.float64) + 2.0 * C.astype(np.float64)).all()
    A = datagen.uniform_pm1(8, "A", 6 * 9).reshape(6, 9)
    out, _ = ref(A, np.eye(9, dtype=np.float32))
    assert (out == A.astype(np.float64)).all()


def test_permutation_rows():
    K, N = 10, 7
    perm = np.array([3, 0, 9, 1, 1, 5, 8, 2])
    P = np.zeros((perm.size, K), np.float32)
    P[np.arange(perm.size), perm] = 1.0
    B = datagen.normal01(9, "B", K * N).reshape(K, N)
    out, _ = ref(P, B)
    assert (out == B[perm].astype(np.float64)).all()


def test_exact_integer_brute_force():
    M, N, K = 13, 11, 29
    A = datagen.small_ints(10, "A", M * K).reshape(M, K)
    B = datagen.small_ints(10, "B", K * N).reshape(K, N)
    C = datagen.small_ints(10, "C", M * N).reshape(M, N)
    out, absprod = ref(A, B, C, alpha=2.0, beta=-1.0)
    Ai = [[int(v) for v in row] for row in A]
    Bi = [[int(v) for v in row] for row in B]
    for i in range(M):
        for j in range(N):
            s = sum(Ai[i][k] * Bi[k][j] for k in range(K))
            sa = sum(abs(Ai[i][k] * Bi[k][j]) for k in range(K))
            assert out[i, j] == 2 * s - int(C[i, j]), (i, j)
            assert absprod[i, j] == sa, (i, j)


def test_leading_dimensions_and_gap_never_read():
    M, N, K = 9, 6, 14
    lda, ldb, ldc = K + 5, N + 3, N + 7
    A = datagen.matrix("ints", 11, "A", M, K, ld=lda)
    B = datagen.matrix("ints", 11, "B", K, N, ld=ldb)
    C = datagen.matrix("ints", 11, "C", M, N, ld=ldc)
    out, _ = oracle.sgemm_ref_flat(M, N, K, 1.0, A, lda, B, ldb, 1.0, C, ldc)
    A2 = A.reshape(M, lda)[:, :K].astype(np.int64)
    B2 = B.reshape(K, ldb)[:, :N].astype(np.int64)
    C2 = C.reshape(M, ldc)[:, :N].astype(np.int64)
    want = A2 @ B2 + C2
    assert np.isfinite(out).all()
    assert (out == want).all()


def test_dot_product_against_fsum():
    K = 3001
    a = datagen.normal01(12, "A", K).reshape(1, K)
    b = datagen.normal01(12, "B", K).reshape(K, 1)
    out, absprod = ref(a, b)
    prods = [float(x) * float(y) for x, y in zip(a[0], b[:, 0])]
    exact = math.fsum(prods)
    assert abs(out[0, 0] - exact) <= K * 2.0 ** -52 * absprod[0, 0]
    assert abs(absprod[0, 0] - math.fsum(abs(p) for p in prods)) <= K * 2.0 ** -52 * absprod[0, 0]


def test_gemv_columns_against_fsum():
    M, K = 5, 200
    A = datagen.uniform_pm1(13, "A", M * K).reshape(M, K)
    x = datagen.uniform_pm1(13, "B", K).reshape(K, 1)
    out, absprod = ref(A, x)
    for i in range(M):
        exact = math.fsum(float(A[i, k]) * float(x[k, 0]) for k in range(K))
        assert abs(out[i, 0] - exact) <= K * 2.0 ** -52 * absprod[i, 0]


def test_absprod_matches_library_matmul():
    M, N, K = 33, 21, 70
    A = datagen.normal01(14, "A", M * K).reshape(M, K)
    B = datagen.normal01(14, "B", K * N).reshape(K, N)
    _, absprod = ref(A, B)
    lib = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    assert np.allclose(absprod, lib, rtol=1e-12, atol=0)


def test_beta_zero_does_not_read_c():
    A = datagen.uniform_pm1(15, "A", 4 * 5).reshape(4, 5)
    B = datagen.uniform_pm1(15, "B", 5 * 3).reshape(5, 3)
    C = np.full((4, 3), np.nan, np.float32)
    out, _ = ref(A, B, C, alpha=1.0, beta=0.0)
    assert np.isfinite(out).all()


def test_alpha_zero_and_k_zero_scale_c():
    C = datagen.uniform_pm1(16, "C", 4 * 3).reshape(4, 3)
    A = np.full((4, 5), np.inf, np.float32)
    B = np.ones((5, 3), np.float32)
    out, _ = ref(A, B, C, alpha=0.0, beta=2.0)
    assert (out == 2.0 * C.astype(np.float64)).all()
    out0, _ = ref(np.zeros((4, 0), np.float32), np.zeros((0, 3), np.float32), C,
                  alpha=1.0, beta=-0.5)
    assert (out0 == -0.5 * C.astype(np.float64)).all()


def test_row_subset_equals_full_rows():
    M, N, K = 20, 9, 31
    A = datagen.normal01(17, "A", M * K).reshape(M, K)
    B = datagen.normal01(17, "B", K * N).reshape(K, N)
    full, fabs_ = ref(A, B)
    rows = [19, 0, 7, 7]
    part, pabs = ref(A, B, rows=rows)
    assert (part == full[rows]).all()
    assert (pabs == fabs_[rows]).all()


def test_thread_count_does_not_change_result():
    M, N, K = 37, 13, 50
    A = datagen.normal01(18, "A", M * K).reshape(M, K)
    B = datagen.normal01(18, "B", K * N).reshape(K, N)
    one, _ = ref(A, B, threads=1)
    many, _ = ref(A, B, threads=7)
    assert (one == many).all()


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.5, 2.0), (-1.5, 0.25)])
def test_fp32_library_gemm_within_bound(alpha, beta):
    M, N, K = 70, 50, 300
    A = datagen.uniform_pm1(19, "A", M * K).reshape(M, K)
    B = datagen.uniform_pm1(19, "B", K * N).reshape(K, N)
    C = datagen.uniform_pm1(19, "C", M * N).reshape(M, N)
    out, absprod = ref(A, B, C, alpha=alpha, beta=beta)
    lib32 = (np.float32(alpha) * (A @ B) + np.float32(beta) * C).astype(np.float32)
    bound = oracle.error_bound(absprod, C, alpha, beta, K)
    assert_within(lib32, out, bound, "numpy fp32 gemm vs oracle")
    # The bound is not vacuous: a result perturbed by more than it fails.
    worst = np.unravel_index(np.argmax(bound), bound.shape)
    bumped = lib32.astype(np.float64).copy()
    bumped[worst] += 3 * bound[worst]
    with pytest.raises(AssertionError):
        assert_within(bumped, out, bound, "perturbed")


def test_error_bound_k_floor():
    ab = np.ones((1, 1))
    assert oracle.error_bound(ab, None, 1.0, 0.0, 1)[0, 0] == 2 * 3 * 2.0 ** -24
    assert oracle.error_bound(ab, None, 1.0, 0.0, 100)[0, 0] == 2 * 100 * 2.0 ** -24


def check_bound_pins(error_bound):
    """Values of the stated bound 2*K*2^-24*(|alpha|(|A||B|)_ij + |beta||C_ij|)
    worked out by hand (K at least 3, at least 4 with a bias, whose magnitude
    joins the sum), so that a dropped or mis-scaled term, a signed scalar, a
    transposed C or a wrong constant in ``error_bound`` fails here."""
    u = 2.0 ** -24
    one = lambda v: np.array([[float(v)]])
    # alpha 0.5, beta 2, |C| 3, (|A||B|) 10, K 10: 2*10*u*(0.5*10 + 2*3) = 220 u
    assert error_bound(one(10), one(-3), 0.5, 2.0, 10)[0, 0] == 220 * u
    # the scalars enter by magnitude
    assert error_bound(one(10), one(3), -0.5, -2.0, 10)[0, 0] == 220 * u
    # K = 1 takes the K = 3 constant: 2*3*u*(1*4 + 0.25*8) = 36 u
    assert error_bound(one(4), one(8), 1.0, 0.25, 1)[0, 0] == 36 * u
    # K = 7 with only the beta term: 2*7*u*(0 + 3*5) = 210 u
    assert error_bound(one(0), one(5), 1.0, 3.0, 7)[0, 0] == 210 * u
    # beta = 0: C takes no part, even when it holds a NaN: 2*5*u*4 = 40 u
    assert error_bound(one(4), one(np.nan), 1.0, 0.0, 5)[0, 0] == 40 * u
    # a bias: K = 2 takes the K = 4 constant: 2*4*u*(2*1 + 1*1 + 5) = 64 u
    assert error_bound(one(1), one(1), 2.0, -1.0, 2, bias=np.array([-5.0]))[0, 0] == 64 * u
    # elementwise, row-major: element (i, j) uses C[i][j] and bias[j]
    C = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0]])
    ab = np.array([[0.0, 1.0, 2.0], [3.0, 4.0, 5.0]])
    got = error_bound(ab, C, 1.0, 0.5, 8)
    assert np.array_equal(got, 2 * 8 * u * (ab + 0.5 * C))
    bias = np.array([10.0, -20.0, 30.0])
    got = error_bound(ab, C, 1.0, 0.5, 8, bias=bias)
    assert np.array_equal(got, 2 * 8 * u * (ab + 0.5 * C + np.abs(bias)[None, :]))


def test_error_bound_hand_computed_values():
    check_bound_pins(oracle.error_bound)


# ----- the fused epilogue: bias per column, then ReLU -------------------------------

def test_epilogue_all_ones_closed_form():
    # All-ones operands give K everywhere; a bias b_j makes K + b_j, and ReLU
    # clears exactly the columns whose bias is below -K.
    M, N, K = 5, 8, 12
    A = np.ones((M, K), np.float32)
    B = np.ones((K, N), np.float32)
    bias = np.array([-20, -13, -12, -11, 0, 1, 7, -100], np.float32)
    out, _ = ref(A, B)
    plain = oracle.apply_epilogue(out, bias, oracle.ACT_NONE)
    relu = oracle.apply_epilogue(out, bias, oracle.ACT_RELU)
    for j, b in enumerate(bias):
        assert (plain[:, j] == K + b).all()
        assert (relu[:, j] == max(K + b, 0.0)).all()


def test_epilogue_integer_brute_force():
    # Python integers give the exact act(A B + C + bias); the bias is indexed
    # by column and the activation comes after it.
    M, N, K = 7, 9, 16
    A = datagen.small_ints(21, "A", M * K).reshape(M, K)
    B = datagen.small_ints(21, "B", K * N).reshape(K, N)
    C = datagen.small_ints(21, "C", M * N).reshape(M, N)
    bias = (np.arange(N, dtype=np.float32) * 7 - 30).astype(np.float32)
    out, _ = ref(A, B, C, alpha=1.0, beta=1.0)
    got = oracle.apply_epilogue(out, bias, oracle.ACT_RELU)
    for i in range(M):
        for j in range(N):
            s = sum(int(A[i, k]) * int(B[k, j]) for k in range(K)) + int(C[i, j]) + int(bias[j])
            assert got[i, j] == (s if s > 0 else 0), (i, j)


def test_relu_passes_nan_and_keeps_sign_of_zero():
    x = np.array([[np.nan, -0.0, 0.0, -1.0, 2.5]])
    y = oracle.apply_epilogue(x, None, oracle.ACT_RELU)
    assert np.isnan(y[0, 0])
    assert y[0, 1] == 0.0 and np.signbit(y[0, 1])
    assert list(y[0, 2:]) == [0.0, 0.0, 2.5]
    with pytest.raises(ValueError):
        oracle.apply_epilogue(x, None, 7)


def test_error_bound_with_bias_adds_its_magnitude():
    ab = np.ones((2, 3))
    bias = np.array([1.0, -2.0, 0.0])
    b = oracle.error_bound(ab, None, 1.0, 0.0, 2, bias=bias)
    u = 2.0 ** -24
    assert np.array_equal(b, np.broadcast_to(2 * 4 * u * (1.0 + np.abs(bias)), (2, 3)))
