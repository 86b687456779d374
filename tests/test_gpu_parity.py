"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Floating point is judged elementwise by
|C_gpu - C_ref| <= 2*K*2^-24*(|alpha|(|A||B|)_ij + |beta||C_ij|) (K >= 3);
integer-valued inputs whose partial sums stay below 2^24 must match exactly.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen
import dense_fp32_sgemm_gb300 as sg
import oracle
from tests.checks import assert_within
from tests.gpu_harness import run_gemm
from tests.oracle_cache import workload_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.build()
    sg.set_plan_override(-1, 0)
    sg.set_wait_timeout_ns(0, -1)
    yield
    sg.set_plan_override(-1, 0)
    sg.set_wait_timeout_ns(0, -1)


def inputs(dist, seed, M, N, K, lda=None, ldb=None, ldc=None, with_c=True):
    lda, ldb, ldc = lda or max(K, 1), ldb or max(N, 1), ldc or max(N, 1)
    A = datagen.matrix(dist, seed, "A", M, K, ld=lda) if M * K else np.zeros(max(M * lda, 1), np.float32)
    B = datagen.matrix(dist, seed, "B", K, N, ld=ldb) if K * N else np.zeros(max(K * ldb, 1), np.float32)
    C = datagen.matrix(dist, seed, "C", M, N, ld=ldc) if with_c else None
    return A, lda, B, ldb, C, ldc


def reference(M, N, K, alpha, beta, A, lda, B, ldb, C, ldc, rows=None):
    ref, absprod = oracle.sgemm_ref_flat(M, N, K, alpha, A, lda, B, ldb, beta,
                                         C if beta != 0 else None, ldc, rows=rows)
    rows_idx = np.arange(M) if rows is None else np.asarray(rows)
    Cm = C.reshape(M, ldc)[rows_idx, :N] if (C is not None and beta != 0) else None
    return ref, oracle.error_bound(absprod, Cm, alpha, beta, K)


def check(M, N, K, alpha, beta, dist="uniform", seed=1, lda=None, ldb=None, ldc=None,
          variant=-1, splits=0, offsets=(0, 0, 0), rows=None, label=""):
    A, lda, B, ldb, C, ldc = inputs(dist, seed, M, N, K, lda, ldb, ldc, with_c=True)
    out, _ = run_gemm(M, N, K, alpha, beta, A, lda, B, ldb, C if beta != 0 else None, ldc,
                      offsets=offsets, variant=variant, splits=splits,
                      c_fill=None if beta != 0 else float("nan"))
    ref, bound = reference(M, N, K, alpha, beta, A, lda, B, ldb, C, ldc, rows=rows)
    got = out if rows is None else out[np.asarray(rows)]
    assert_within(got, ref, bound, label or f"{M}x{N}x{K} variant={variant} splits={splits}")
    return out


# ----- every workload at full size, launched as the benchmark launches them ------

@pytest.mark.parametrize("name", [
    "s1_128", "s2_2048", "s3_4092", "s4_rect", "s5_odd", "s6_skinny", "s7_gemv", "s8_2049",
    "s9_ax",
])
def test_workload_full_size(name):
    # Every element of every workload, launched as the benchmark launches it.
    cfg, A, B, C, ref, bound = workload_reference(name)
    M, N, K, alpha, beta = cfg["M"], cfg["N"], cfg["K"], cfg["alpha"], cfg["beta"]
    out, _ = run_gemm(M, N, K, alpha, beta, A, K, B, N, C, N,
                      c_fill=None if beta != 0 else float("nan"))
    assert np.isfinite(out).all()
    assert_within(out, ref, bound, name)


def test_cublas_fp32_meets_the_same_bound():
    # cuBLAS FP32 with TF32 off, on the 2048^3 workload: a second GPU product,
    # independent of this library, must also sit within the bound against the
    # oracle at every element, which checks the oracle and the bound at a
    # size the exact tests do not reach.
    cfg, A, B, C, ref, bound = workload_reference("s2_2048")
    M, N, K = cfg["M"], cfg["N"], cfg["K"]
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        out = torch.mm(torch.from_numpy(A).cuda().view(M, K),
                       torch.from_numpy(B).cuda().view(K, N)).cpu().numpy()
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    assert_within(out, ref, bound, "cuBLAS FP32")


# ----- exact integer inputs: every variant must be bit-exact ---------------------

@pytest.mark.parametrize("variant,splits", [(0, 0), (1, 0), (2, 2), (2, 3), (2, 4), (-1, 0),
                                            (4, 0), (4, 2), (4, 3), (5, 0), (5, 4), (6, 0), (8, 0),
                                            (9, 0)])
@pytest.mark.parametrize("M,N,K", [(64, 64, 64), (300, 520, 64), (129, 257, 40)])
def test_small_integers_bit_exact(variant, splits, M, N, K):
    Kp = (K + 3) // 4 * 4
    Np = (N + 3) // 4 * 4
    A, lda, B, ldb, C, ldc = inputs("ints", 3, M, N, K, lda=Kp, ldb=Np, ldc=Np)
    out, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, variant=variant, splits=splits)
    Ai = A.reshape(M, lda)[:, :K].astype(np.int64)
    Bi = B.reshape(K, ldb)[:, :N].astype(np.int64)
    Ci = C.reshape(M, ldc)[:, :N].astype(np.int64)
    want = Ai @ Bi + Ci
    assert np.array_equal(out.astype(np.int64), want)


# ----- ragged shapes, leading dimensions, alignment -----------------------------

SIZES = [1, 3, 8, 31, 33, 127, 129, 255, 257]


# Automatic plan, the tiled kernel whole (1) and split (2), the mid-size
# kernel with 128-row (4) and 64-row (5) tiles and the split-K kernel (6) on
# the same edges (8: the split-K kernel with 64-column tiles; 9: the small-
# product kernel).
@pytest.mark.parametrize("variant", [-1, 1, 2, 4, 5, 6, 8, 9])
@pytest.mark.parametrize("M", [1, 33, 129, 257])
@pytest.mark.parametrize("N", [1, 31, 255, 257])
@pytest.mark.parametrize("K", [1, 8, 127])
def test_ragged_shapes_aligned_ld(M, N, K, variant):
    Kp, Np = (K + 3) // 4 * 4 + 4, (N + 3) // 4 * 4 + 8
    check(M, N, K, 0.5, 2.0, dist="normal", seed=M * 7 + N * 3 + K, lda=Kp, ldb=Np, ldc=Np,
          variant=variant)


@pytest.mark.parametrize("variant", [-1, 0, 4, 5, 6, 8, 9])
@pytest.mark.parametrize("M,N,K", [(3, 5, 7), (33, 255, 31), (257, 129, 127), (130, 300, 65)])
def test_ragged_shapes_odd_ld(M, N, K, variant):
    check(M, N, K, 1.0, 0.0, dist="uniform", seed=5, lda=K + 1, ldb=N + 3, ldc=N + 5,
          variant=variant)


@pytest.mark.parametrize("variant", [-1, 0, 4, 5, 6, 8, 9])
@pytest.mark.parametrize("offsets", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1)])
def test_misaligned_pointers(offsets, variant):
    check(200, 300, 100, 1.0, 1.0, seed=6, offsets=offsets, lda=104, ldb=300, ldc=300,
          variant=variant)


# ----- the mid-size kernel: any alignment, copies of 4 or 16 bytes -------------

@pytest.mark.parametrize("variant,splits", [(4, 0), (4, 2), (4, 5), (5, 0), (5, 3), (6, 0),
                                            (8, 0), (9, 0)])
@pytest.mark.parametrize("offsets,lds", [
    ((0, 0, 0), (516, 1028, 1028)),      # aligned: 16-byte copies of B
    ((1, 0, 0), (513, 1028, 1025)),      # A and C unaligned, B aligned
    ((0, 3, 0), (516, 1025, 1028)),      # B unaligned: 4-byte copies of B
    ((2, 1, 3), (515, 1027, 1031)),      # everything off 16 bytes
])
def test_mid_kernel_any_alignment_integers_bit_exact(variant, splits, offsets, lds):
    # The 1023 x 1025 x 513 shape (all tails ragged) on small integers: every
    # copy path, zero fill and split must give the exact sum.
    M, N, K = 1023, 1025, 513
    A, lda, B, ldb, C, ldc = inputs("ints", 60, M, N, K, lda=lds[0], ldb=lds[1], ldc=lds[2])
    out, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, offsets=offsets,
                      variant=variant, splits=splits)
    want = (A.reshape(M, lda)[:, :K].astype(np.int64) @ B.reshape(K, ldb)[:, :N].astype(np.int64)
            + C.reshape(M, ldc)[:, :N].astype(np.int64))
    assert np.array_equal(out.astype(np.int64), want)


@pytest.mark.parametrize("variant", [4, 5, 6, 8, 9])
@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 4097, 3), (65, 129, 17), (128, 128, 16),
                                   (200, 2000, 1500), (17, 8192, 4096), (3000, 300, 5000)])
def test_mid_kernel_floats_within_bound(variant, M, N, K):
    check(M, N, K, -0.75, 1.5, dist="normal", seed=61 + M + N, lda=K + 1, ldb=N + 2, ldc=N + 3,
          offsets=(1, 2, 3), variant=variant)


def test_mid_kernel_stream_k_is_bitwise_deterministic():
    M, N, K = 700, 900, 3000
    A, lda, B, ldb, _, _ = inputs("uniform", 62, M, N, K, lda=K + 1, ldb=N + 1)
    first, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N, variant=4, splits=5)
    for _ in range(3):
        again, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N, variant=4, splits=5)
        assert np.array_equal(first, again)


@pytest.mark.parametrize("variant", [6, 8, 9])
def test_split_k_kernel_is_bitwise_deterministic(variant):
    # The groups' sums are added in group order, whatever the timing.
    M, N, K = 1000, 1100, 2500
    A, lda, B, ldb, _, _ = inputs("uniform", 63, M, N, K, lda=K + 1, ldb=N + 1)
    first, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N, variant=variant)
    for _ in range(3):
        again, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N, variant=variant)
        assert np.array_equal(first, again)


@pytest.mark.parametrize("M,N,K,variant", [(3000, 4, 20000, 7), (2050, 2052, 700, -1)])
def test_narrow_and_thin_edge_plans_are_bitwise_deterministic(M, N, K, variant):
    # The narrow kernel's lanes add their k in a fixed order and the warp adds
    # the lanes by a fixed butterfly; a thin-edge plan runs three kernels on
    # two streams, each deterministic, with no shared output element.
    A, lda, B, ldb, _, _ = inputs("uniform", 64, M, N, K, lda=K, ldb=N)
    first, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N, variant=variant)
    for _ in range(3):
        again, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N, variant=variant)
        assert np.array_equal(first, again)


@pytest.mark.parametrize("variant", [6, 8, 9])
@pytest.mark.parametrize("K", [1, 7, 8, 9, 15, 16, 17, 31, 32, 33, 63, 64, 65, 100, 129])
def test_split_k_kernel_every_k_remainder(K, variant):
    # Each k-group takes 16 (eight groups: 8) of every 64-k slice; in the last
    # slice a group multiplies only the k that exist: every remainder of K
    # modulo 64 that changes a group's count, on exact integers.
    M, N = 70, 200
    A, lda, B, ldb, C, ldc = inputs("ints", 64 + K, M, N, K, lda=K + 3, ldb=N + 1, ldc=N)
    out, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, variant=variant)
    want = (A.reshape(M, lda)[:, :K].astype(np.int64) @ B.reshape(K, ldb)[:, :N].astype(np.int64)
            + C.reshape(M, ldc)[:, :N].astype(np.int64))
    assert np.array_equal(out.astype(np.int64), want)


@pytest.mark.parametrize("offsets,lds,variant", [
    ((1, 0, 0), (512, 1300, 1300), -1), ((0, 3, 0), (512, 1300, 1303), -1),
    ((1, 2, 3), (513, 1301, 1302), -1), ((0, 0, 0), (513, 1300, 1300), 1),
    ((2, 1, 0), (515, 1305, 1300), 2)])
def test_unaligned_operands_copied_for_the_tiled_kernel(offsets, lds, variant):
    # Large enough for the tiled kernel: the unaligned operand(s) are first
    # copied to aligned rows; guard bands and leading-dimension gaps of the
    # caller's buffers stay untouched.
    M, N, K = 1400, 1300, 512
    p = sg.plan_describe(M, N, K, lda=lds[0], ldb=lds[1], ldc=lds[2], a_addr=256 + 4 * offsets[0],
                         b_addr=512 + 4 * offsets[1], c_addr=768 + 4 * offsets[2])
    if variant < 0:
        assert p["variant"] in ("mid", "ksplit") or (
            p["variant"] in ("tile", "streamk") and (p["pack_a"], p["pack_b"]) != ("0", "0"))
    check(M, N, K, 0.5, 2.0, dist="normal", seed=40 + sum(offsets), offsets=offsets,
          lda=lds[0], ldb=lds[1], ldc=lds[2], variant=variant)


# ----- narrow N (a warp per row of A) and thin edges beside the tiles ----------

@pytest.mark.parametrize("N", [1, 2, 3, 4])
@pytest.mark.parametrize("M,K,lda_pad,off", [(1, 1, 0, 0), (9, 3, 1, 1), (40, 1024, 0, 0),
                                             (300, 1025, 3, 0), (1000, 3000, 0, 2),
                                             (5000, 129, 1, 3)])
def test_narrow_kernel_integers_bit_exact(N, M, K, lda_pad, off):
    # Every row of A against N columns of B: chunk edges of K (1024), rows
    # that do not fill the last pass of eight, 16-byte and 4-byte loads of A.
    A, lda, B, ldb, C, ldc = inputs("ints", 80 + N + K, M, N, K, lda=K + lda_pad, ldb=N + 1,
                                    ldc=N + 2)
    out, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, offsets=(off, 1, 0), variant=7)
    want = (A.reshape(M, lda)[:, :K].astype(np.int64) @ B.reshape(K, ldb)[:, :N].astype(np.int64)
            + C.reshape(M, ldc)[:, :N].astype(np.int64))
    assert np.array_equal(out.astype(np.int64), want)


@pytest.mark.parametrize("M,N,K", [(8192, 1, 4096), (3000, 4, 2049), (64, 3, 20000), (7, 2, 5),
                                   (40, 2, 30000), (33, 1, 50000)])
def test_narrow_kernel_floats_within_bound(M, N, K):
    # K of 20000-50000 takes several chunks of B for every column count.
    check(M, N, K, 0.5, -2.0, dist="normal", seed=90 + M, lda=K, ldb=N, ldc=N, variant=7)
    check(M, N, K, 1.0, 0.0, dist="uniform", seed=91 + M, lda=K + 1, ldb=N + 3, ldc=N + 1,
          offsets=(1, 0, 2))


@pytest.mark.parametrize("M,N,K,lds,offsets,em,en", [
    (2049, 2049, 1000, (1000, 2049, 2049), (0, 0, 0), 1, 1),  # both copied to aligned rows
    (2050, 2052, 700, (700, 2052, 2052), (0, 0, 0), 2, 4),    # aligned: no copy
    (2080, 2051, 1024, (1024, 2051, 2051), (0, 1, 0), 32, 3),  # B copied
    (4128, 2051, 512, (512, 2051, 2053), (0, 1, 3), 32, 3),
])
def test_thin_edges_integers_bit_exact(M, N, K, lds, offsets, em, en):
    # The automatic plan leaves the last rows to the skinny kernel and the last
    # columns to the narrow kernel; the three kernels together give the exact
    # sum over every element.
    p = sg.plan_describe(M, N, K, lda=lds[0], ldb=lds[1], ldc=lds[2], a_addr=256 + 4 * offsets[0],
                         b_addr=512 + 4 * offsets[1], c_addr=768 + 4 * offsets[2])
    assert p["variant"] in ("tile", "streamk") and (int(p["edge_m"]), int(p["edge_n"])) == (em, en)
    A, lda, B, ldb, C, ldc = inputs("ints", 95 + K, M, N, K, lda=lds[0], ldb=lds[1], ldc=lds[2])
    out, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, offsets=offsets)
    # small integers: every partial sum is an integer below 2^24, so the FP64
    # product (a library matmul) is the exact one
    want = (A.reshape(M, lda)[:, :K].astype(np.float64) @ B.reshape(K, ldb)[:, :N].astype(np.float64)
            + C.reshape(M, ldc)[:, :N].astype(np.float64))
    assert np.array_equal(out.astype(np.float64), want)


def test_thin_edges_floats_and_epilogue():
    # Floats within the bound, and the bias of the last columns taken from
    # their own columns.
    M, N, K = 2049, 2049, 512
    check(M, N, K, 0.75, 1.5, dist="normal", seed=97, lda=K, ldb=N, ldc=N)
    A, lda, B, ldb, C, ldc = inputs("ints", 98, M, N, K, lda=K, ldb=N, ldc=N)
    bias = (np.arange(N) % 37 - 18).astype(np.float32)
    out, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, bias=bias, activation=1)
    want = (A.reshape(M, lda)[:, :K].astype(np.float64) @ B.reshape(K, ldb)[:, :N].astype(np.float64)
            + C.reshape(M, ldc)[:, :N].astype(np.float64) + bias.astype(np.float64)[None, :])
    assert np.array_equal(out.astype(np.float64), np.maximum(want, 0))


@pytest.mark.parametrize("M,N,K", [(300, 40, 50), (70, 1000, 9), (33, 3, 130), (5, 700, 300),
                                   (129, 257, 1000)])
def test_copy_pass_row_widths(M, N, K):
    # The copy to aligned rows runs 32 to 256 threads over a row depending on
    # its width (a block copies several short rows at once); every width, with
    # both operands unaligned, through the tiled kernel on small integers.
    lda, ldb, ldc = K + 1, N + 3, N + 1
    A, lda, B, ldb, C, ldc = inputs("ints", 70 + K, M, N, K, lda=lda, ldb=ldb, ldc=ldc)
    out, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, offsets=(1, 3, 0), variant=1)
    want = (A.reshape(M, lda)[:, :K].astype(np.int64) @ B.reshape(K, ldb)[:, :N].astype(np.int64)
            + C.reshape(M, ldc)[:, :N].astype(np.int64))
    assert np.array_equal(out.astype(np.int64), want)


@pytest.mark.parametrize("variant", [-1, 1, 2, 4, 6])
def test_odd_workload_bit_exact(variant):
    # 1023 x 1025 x 513 with small integers, as planned and through the tiled
    # kernel (operands copied to aligned rows first) and the mid-size kernel.
    M, N, K = 1023, 1025, 513
    A, lda, B, ldb, C, ldc = inputs("ints", 41, M, N, K)
    out, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, variant=variant)
    want = (A.reshape(M, K).astype(np.int64) @ B.reshape(K, N).astype(np.int64)
            + C.reshape(M, N).astype(np.int64))
    assert np.array_equal(out.astype(np.int64), want)


@pytest.mark.parametrize("splits", [2, 3, 4, 5])
def test_stream_k_forced_splits(splits):
    check(640, 1024, 1000, 1.0, 0.5, seed=8, variant=2, splits=splits)


@pytest.mark.parametrize("stages", [3, 4])
@pytest.mark.parametrize("splits", [0, 3])
def test_ring_depths(stages, splits):
    try:
        sg.set_tile_config(3, stages, 16)
        check(700, 900, 1100, 0.5, 2.0, seed=20 + stages, variant=2 if splits else -1,
              splits=splits, lda=1100, ldb=900, ldc=904)
    finally:
        sg.set_tile_config(3, 3, 16)


def test_generic_forced_matches_bound():
    check(300, 400, 500, -1.5, 0.25, seed=9, variant=0)


# ----- conventions ---------------------------------------------------------------

def test_beta_zero_ignores_nan_in_c():
    M, N, K = 150, 260, 70
    A, lda, B, ldb, _, _ = inputs("uniform", 10, M, N, K, ldb=260, lda=72)
    out, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N, c_fill=float("nan"))
    assert np.isfinite(out).all()


@pytest.mark.parametrize("alpha,K", [(0.0, 64), (1.0, 0)])
def test_alpha_zero_or_k_zero_scales_c(alpha, K):
    M, N = 70, 90
    A, lda, B, ldb, C, ldc = inputs("uniform", 11, M, N, K, lda=max(K, 4), ldb=92, ldc=92)
    out, _ = run_gemm(M, N, K, alpha, -2.0, A, lda, B, ldb, C, ldc)
    want = (np.float32(-2.0) * C.reshape(M, ldc)[:, :N]).astype(np.float32)
    assert np.array_equal(out, want)
    out0, _ = run_gemm(M, N, K, alpha, 0.0, A, lda, B, ldb, None, ldc, c_fill=float("nan"))
    assert np.array_equal(out0, np.zeros((M, N), np.float32))


def test_stream_k_is_bitwise_deterministic():
    M, N, K = 512, 2048, 2048
    A, lda, B, ldb, _, _ = inputs("uniform", 12, M, N, K)
    first, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N, variant=2, splits=3)
    for _ in range(4):
        again, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N, variant=2, splits=3)
        assert np.array_equal(first, again)


def test_fma_forms_are_bitwise_identical():
    # Every form issues the same fma sequence per output; only the packing differs.
    M, N, K = 256, 512, 300
    A, lda, B, ldb, _, _ = inputs("normal", 13, M, N, K, lda=300, ldb=512)
    results = []
    try:
        for fm, st, tm in [(0, 3, 16), (1, 3, 16), (2, 3, 16), (3, 3, 16), (3, 4, 16)]:
            sg.set_tile_config(fm, st, tm)
            out, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N, variant=1)
            results.append(out)
    finally:
        sg.set_tile_config(3, 3, 16)
    for r in results[1:]:
        assert np.array_equal(results[0], r)


def test_host_entry_point():
    M, N, K = 333, 444, 555
    A, lda, B, ldb, C, ldc = inputs("uniform", 14, M, N, K)
    Ah = A.reshape(M, K)
    Bh = B.reshape(K, N)
    Ch = C.reshape(M, N).copy()
    sg.run_host(Ah, Bh, Ch, alpha=0.5, beta=2.0)
    ref, bound = reference(M, N, K, 0.5, 2.0, A, lda, B, ldb, C, ldc)
    assert_within(Ch, ref, bound, "sgemm_run_host")


@pytest.mark.parametrize("M,N,K,alpha,beta,blocks", [(3000, 1030, 4100, 0.5, 2.0, 4),
                                                    (2048, 2056, 2048, 1.0, 0.0, 2),
                                                    (2049, 2049, 2049, 1.0, 0.5, 2)])
def test_host_entry_point_in_row_blocks(M, N, K, alpha, beta, blocks):
    # Large enough that the host entry point copies and computes row blocks in
    # a pipeline (4 blocks with a ragged last one; 2 blocks); pinned host
    # buffers; every element checked.
    A, lda, B, ldb, C, ldc = inputs("normal", 15, M, N, K)
    Ah = torch.from_numpy(A.reshape(M, K)).pin_memory()
    Bh = torch.from_numpy(B.reshape(K, N)).pin_memory()
    Ch = torch.from_numpy(C.reshape(M, N).copy()).pin_memory()
    sg.run_host(Ah, Bh, Ch, alpha=alpha, beta=beta)
    ref, bound = reference(M, N, K, alpha, beta, A, lda, B, ldb, C if beta else None, ldc)
    assert_within(Ch.numpy(), ref, bound, "sgemm_run_host in row blocks")


def test_thin_edges_on_two_streams_at_once():
    # Two streams, each with a product whose last row and column go to the
    # edge kernels on the library's second stream: each result is its own.
    M, N, K = 2049, 2049, 1000
    outs = []
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    data = []
    for i, st in enumerate(streams):
        A, lda, B, ldb, _, _ = inputs("ints", 120 + i, M, N, K, lda=K, ldb=N)
        dA = torch.from_numpy(A).cuda()
        dB = torch.from_numpy(B).cuda()
        dC = torch.full((M * N,), float("nan"), device="cuda")
        data.append((A, B, dA, dB, dC))
    torch.cuda.synchronize()
    for _ in range(3):
        for (A, B, dA, dB, dC), st in zip(data, streams):
            assert sg.sgemm_run(M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0,
                                dC.data_ptr(), N, st.cuda_stream) == 0
    torch.cuda.synchronize()
    for A, B, dA, dB, dC in data:
        want = A.reshape(M, K).astype(np.float64) @ B.reshape(K, N).astype(np.float64)
        assert np.array_equal(dC.cpu().numpy().reshape(M, N).astype(np.float64), want)


def test_torch_binding_with_strided_rows():
    M, N, K = 200, 300, 96
    A, _, B, _, _, _ = inputs("uniform", 15, M, N, K)
    At = torch.zeros(M, K + 8, device="cuda")[:, :K]
    At.copy_(torch.from_numpy(A.reshape(M, K)))
    Bt = torch.from_numpy(B.reshape(K, N)).cuda()
    Ct = torch.empty(M, N, device="cuda")
    sg.run(At, Bt, Ct)
    ref, bound = reference(M, N, K, 1.0, 0.0, A, K, B, N, None, N)
    assert_within(Ct.cpu().numpy(), ref, bound, "torch binding")


# ----- bounded waits --------------------------------------------------------------

def test_wait_timeout_reports_and_recovers():
    M, N, K = 512, 1024, 1024
    A, lda, B, ldb, _, _ = inputs("uniform", 16, M, N, K)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.zeros(M * N, device="cuda")
    stream = torch.cuda.current_stream()
    # The producer of the tiled kernel stops issuing copies at k-iteration 5,
    # so the consumers' wait for iteration 5 runs out after 2 ms; the kernel
    # records the timeout and returns.
    sg.set_wait_timeout_ns(2_000_000, 5)
    sg.set_plan_override(sg.VARIANT_TILE, 0)
    try:
        st = sg.sgemm_run(M, N, K, 1.0, dA.data_ptr(), lda, dB.data_ptr(), ldb, 0.0,
                          dC.data_ptr(), N, stream.cuda_stream)
        assert st == 0
        assert sg.device_status(stream) == 5  # SGEMM_ERR_DEVICE_TIMEOUT
    finally:
        sg.set_wait_timeout_ns(0, -1)
        sg.set_plan_override(-1, 0)
    assert sg.device_status(stream) == 0
    # The context and the library still work.
    out, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N)
    ref, bound = reference(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N)
    assert_within(out, ref, bound, "after timeout")


# ----- probes ----------------------------------------------------------------------

def test_probes_run():
    sink = torch.zeros(4096, device="cuda")
    buf = torch.ones(1 << 20, device="cuda")
    stream = torch.cuda.current_stream()
    for paired in (False, True):
        flops = sg.probe_ffma(paired, 100, 152, sink.data_ptr(), stream)
        assert flops == 152 * 512 * 100 * 128 * 2
    nbytes = sg.probe_read(buf.data_ptr(), buf.numel(), sink.data_ptr(), 152, stream)
    assert nbytes == 4 * buf.numel()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    flops = sg.probe_tf32(1000, sms, stream)
    assert flops == sms * 1000 * 4 * 2 * 128 * 256 * 8
    assert sg.device_status(stream) == 0
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    sg.probe_hold(2_000_000, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    assert 1.9 <= e0.elapsed_time(e1) < 50.0


# ----- fused epilogue: bias per column, then ReLU --------------------------------------

EPI_CASES = [  # (M, N, K, variant, splits): every kernel and the alpha == 0 path
    (130, 300, 96, 0, 0), (300, 520, 64, 1, 0), (300, 520, 256, 2, 3),
    (257, 1030, 2048, -1, 0), (9, 1030, 1000, 3, 0), (16, 1024, 96, 3, 2),
    (300, 520, 256, 4, 0), (301, 1030, 700, 4, 3), (40, 1030, 500, 5, 2),
    (300, 520, 256, 6, 0), (1023, 1030, 513, 6, 0), (300, 520, 256, 8, 0), (129, 70, 70, 8, 0),
    (130, 300, 96, 9, 0), (33, 65, 200, 9, 0), (500, 3, 300, 7, 0), (64, 4, 3000, 7, 0),
]


@pytest.mark.parametrize("activation", [0, 1])
@pytest.mark.parametrize("M,N,K,variant,splits", EPI_CASES)
def test_epilogue_integers_bit_exact(M, N, K, variant, splits, activation):
    Kp, Np = (K + 3) // 4 * 4, (N + 3) // 4 * 4
    A, lda, B, ldb, C, ldc = inputs("ints", 31, M, N, K, lda=Kp, ldb=Np, ldc=Np)
    bias = (np.arange(N) % 41 - 20).astype(np.float32)
    out, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, variant=variant, splits=splits,
                      bias=bias, activation=activation)
    want = (A.reshape(M, lda)[:, :K].astype(np.int64) @ B.reshape(K, ldb)[:, :N].astype(np.int64)
            + C.reshape(M, ldc)[:, :N].astype(np.int64) + bias.astype(np.int64)[None, :])
    if activation == 1:
        want = np.maximum(want, 0)
    assert np.array_equal(out.astype(np.int64), want)


@pytest.mark.parametrize("M,N,K,variant,splits", EPI_CASES)
def test_epilogue_floats_within_bound(M, N, K, variant, splits):
    Kp, Np = (K + 3) // 4 * 4, (N + 3) // 4 * 4
    A, lda, B, ldb, C, ldc = inputs("normal", 32, M, N, K, lda=Kp, ldb=Np, ldc=Np + 4)
    bias = datagen.normal01(33, "C", N)
    out, _ = run_gemm(M, N, K, 0.75, -0.5, A, lda, B, ldb, C, ldc, variant=variant, splits=splits,
                      bias=bias, activation=1)
    ref, absprod = oracle.sgemm_ref_flat(M, N, K, 0.75, A, lda, B, ldb, -0.5, C, ldc)
    want = oracle.apply_epilogue(ref, bias, oracle.ACT_RELU)
    bound = oracle.error_bound(absprod, C.reshape(M, ldc)[:, :N], 0.75, -0.5, K, bias=bias)
    assert_within(out, want, bound, f"epilogue {M}x{N}x{K} variant={variant}")
    assert (out >= 0).all()


@pytest.mark.parametrize("K,alpha", [(0, 1.0), (64, 0.0)])
def test_epilogue_on_the_scale_path(K, alpha):
    # No product: C = relu(beta * C + bias), and a NaN in C stays NaN.
    M, N = 33, 70
    A, lda, B, ldb, C, ldc = inputs("normal", 34, M, N, max(K, 1), ldc=N)
    C = C.copy()
    C.reshape(M, ldc)[5, :] = np.nan
    bias = datagen.normal01(35, "C", N)
    out, _ = run_gemm(M, N, K, alpha, 2.0, A, lda, B, ldb, C, ldc, bias=bias, activation=1)
    want = oracle.apply_epilogue(2.0 * C.reshape(M, ldc)[:, :N].astype(np.float64), bias,
                                 oracle.ACT_RELU)
    bound = oracle.error_bound(np.zeros((M, N)), C.reshape(M, ldc)[:, :N], 0.0, 2.0, 1, bias=bias)
    assert np.isnan(out[5]).all() and np.isnan(want[5]).all()
    keep = np.ones(M, bool)
    keep[5] = False
    assert_within(out[keep], want[keep], bound[keep], "scale path epilogue")


def test_epilogue_torch_binding():
    M, N, K = 70, 260, 130
    A = torch.randn(M, K, device="cuda")
    B = torch.randn(K, N, device="cuda")
    C = torch.empty(M, N, device="cuda")
    bias = torch.randn(N, device="cuda")
    sg.run(A, B, C, 1.0, 0.0, bias=bias, activation=sg.ACT_RELU)
    ref, absprod = oracle.sgemm_ref(A.cpu().numpy(), B.cpu().numpy())
    want = oracle.apply_epilogue(ref, bias.cpu().numpy(), oracle.ACT_RELU)
    bound = oracle.error_bound(absprod, None, 1.0, 0.0, K, bias=bias.cpu().numpy())
    assert_within(C.cpu().numpy(), want, bound, "torch binding epilogue")


# ----- skinny-M streaming kernel ---------------------------------------------------

def ceil4(x):
    return (x + 3) // 4 * 4


@pytest.mark.parametrize("M", [1, 5, 8, 9, 16, 17, 24, 31, 32])
@pytest.mark.parametrize("N,K", [(256, 32), (300, 70), (1030, 1000), (4096, 513),
                                 (10240, 320), (40000, 64)])
def test_skinny_shapes(M, N, K):
    check(M, N, K, 0.5, 2.0, dist="normal", seed=M + N + K, lda=ceil4(K), ldb=ceil4(N),
          ldc=N + 1, label=f"skinny {M}x{N}x{K}")


@pytest.mark.parametrize("M", [16, 32, 27])
@pytest.mark.parametrize("splits", [0, 2, 3, 7])
def test_skinny_integers_bit_exact(splits, M):
    N, K = 1024, 96
    A, lda, B, ldb, C, ldc = inputs("ints", 17, M, N, K)
    out, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, variant=3, splits=splits)
    want = (A.reshape(M, K).astype(np.int64) @ B.reshape(K, N).astype(np.int64)
            + C.reshape(M, N).astype(np.int64))
    assert np.array_equal(out.astype(np.int64), want)


@pytest.mark.parametrize("M", [16, 32])
def test_skinny_is_bitwise_deterministic(M):
    N, K = 2048, 4096
    A, lda, B, ldb, _, _ = inputs("uniform", 18, M, N, K)
    first, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N)
    for _ in range(3):
        again, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N)
        assert np.array_equal(first, again)


@pytest.mark.parametrize("M", [16, 32])
def test_skinny_wait_timeout_reports_and_recovers(M):
    N, K = 1024, 4096
    A, lda, B, ldb, _, _ = inputs("uniform", 19, M, N, K)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.zeros(M * N, device="cuda")
    stream = torch.cuda.current_stream()
    # Every CTA has at least two k-steps here; the second one's copy is never issued.
    assert int(sg.plan_describe(M, N, K)["sk_share"]) >= 2
    sg.set_wait_timeout_ns(2_000_000, 1)
    try:
        st = sg.sgemm_run(M, N, K, 1.0, dA.data_ptr(), lda, dB.data_ptr(), ldb, 0.0,
                          dC.data_ptr(), N, stream.cuda_stream)
        assert st == 0
        assert sg.device_status(stream) == 5
    finally:
        sg.set_wait_timeout_ns(0, -1)
    out, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N)
    ref, bound = reference(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N)
    assert_within(out, ref, bound, "skinny after timeout")


# ----- CUDA graphs -------------------------------------------------------------------

@pytest.mark.parametrize("M,N,K,variant", [(16, 4096, 2048, -1), (1100, 1300, 512, 2),
                                           (300, 520, 200, 0), (1023, 1025, 513, 4),
                                           (700, 900, 3000, 5), (1023, 1025, 513, 6),
                                           (2049, 2049, 1000, -1), (3000, 3, 1000, 7),
                                           (513, 515, 500, 8), (200, 300, 150, 9)])
def test_capture_in_a_cuda_graph_and_replay(M, N, K, variant):
    # After a first call has set up the stream's workspace, sgemm_run queues
    # kernels only (no allocation, no host synchronisation), so it can be
    # captured in a CUDA graph and replayed: the skinny, stream-K, 64 x 64 and
    # mid-size paths each give the eager result, bit for bit, on every replay.
    sg.set_plan_override(variant, 0)
    try:
        capture_and_replay(M, N, K)
    finally:
        sg.set_plan_override(-1, 0)


def capture_and_replay(M, N, K):
    A, lda, B, ldb, C, ldc = inputs("uniform", 50 + M, M, N, K)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.zeros(M * N, device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        st = sg.sgemm_run(M, N, K, 1.0, dA.data_ptr(), lda, dB.data_ptr(), ldb, 0.0,
                          dC.data_ptr(), N, side.cuda_stream)
        assert st == 0
    torch.cuda.synchronize()
    eager = dC.clone()
    dC.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        st = sg.sgemm_run(M, N, K, 1.0, dA.data_ptr(), lda, dB.data_ptr(), ldb, 0.0,
                          dC.data_ptr(), N, side.cuda_stream)
    assert st == 0
    for _ in range(3):
        dC.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(dC, eager)
    assert sg.device_status() == 0


def _random_ffma_cases(seed, count):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        M = int(rng.integers(1, 1400))
        N = int(rng.integers(1, 1400))
        K = int(rng.integers(1, 2500))
        pad = [int(rng.choice([0, 0, 1, 3])) for _ in range(3)]
        out.append((M, N, K, float(rng.choice([1.0, -0.5])), float(rng.choice([0.0, 2.0])), pad))
    return out


@pytest.mark.parametrize("M,N,K,alpha,beta,pad", _random_ffma_cases(7, 24))
def test_random_shapes_planned(M, N, K, alpha, beta, pad):
    # Seeded random shapes and leading-dimension padding through whatever
    # plan the planner picks (skinny, 64 x 64, tiled, stream-K, copies).
    check(M, N, K, alpha, beta, lda=K + pad[0], ldb=N + pad[1], ldc=N + pad[2], seed=M ^ N ^ K,
          label=f"random {M}x{N}x{K} pad={pad}")
