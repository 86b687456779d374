"""GPU parity of the 3xTF32 tensor-core entry point (sgemm_run_3xtf32) against
the CPU oracle, through the C ABI.

The variant must meet the bound of the FFMA path,
|C_gpu - C_ref| <= 2*K*2^-24*(|alpha|(|A||B|)_ij + |beta||C_ij|), and be
bit-exact on small-integer inputs (every TF32 split of an integer below 2^11
has lo = 0, and the products and partial sums are exact).
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

X3 = "sgemm_run_3xtf32"


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.build()
    sg.set_plan_override(-1, 0)
    sg.set_wait_timeout_ns(0, -1)
    sg.set_3xtf32_config(16, None)
    yield
    sg.set_plan_override(-1, 0)
    sg.set_wait_timeout_ns(0, -1)
    sg.set_3xtf32_config(16, None)


def inputs(dist, seed, M, N, K, lda=None, ldb=None, ldc=None):
    lda, ldb, ldc = lda or K, ldb or N, ldc or N
    A = datagen.matrix(dist, seed, "A", M, K, ld=lda)
    B = datagen.matrix(dist, seed, "B", K, N, ld=ldb)
    C = datagen.matrix(dist, seed, "C", M, N, ld=ldc)
    return A, lda, B, ldb, C, ldc


def reference(M, N, K, alpha, beta, A, lda, B, ldb, C, ldc, rows=None):
    ref, absprod = oracle.sgemm_ref_flat(M, N, K, alpha, A, lda, B, ldb, beta,
                                         C if beta != 0 else None, ldc, rows=rows)
    rows_idx = np.arange(M) if rows is None else np.asarray(rows)
    Cm = C.reshape(M, ldc)[rows_idx, :N] if (C is not None and beta != 0) else None
    return ref, oracle.error_bound(absprod, Cm, alpha, beta, K)


def check(M, N, K, alpha=1.0, beta=0.0, dist="uniform", seed=3, lda=None, ldb=None, ldc=None,
          offsets=(0, 0, 0), rows=None, exact=False):
    A, lda, B, ldb, C, ldc = inputs(dist, seed, M, N, K, lda, ldb, ldc)
    out, _ = run_gemm(M, N, K, alpha, beta, A, lda, B, ldb, C if beta != 0 else None, ldc,
                      offsets=offsets, c_fill=None if beta != 0 else float("nan"), entry=X3)
    ref, bound = reference(M, N, K, alpha, beta, A, lda, B, ldb, C, ldc, rows=rows)
    got = out if rows is None else out[np.asarray(rows)]
    label = f"3xTF32 {M}x{N}x{K} {dist} alpha={alpha} beta={beta}"
    if exact:
        np.testing.assert_array_equal(got, ref.astype(np.float32), err_msg=label)
    else:
        assert_within(got, ref, bound, label)
    return out, got, ref, bound


# Shapes above the FFMA hand-over (M > 16, K >= 64) spanning several 128 x 256
# tiles, with ragged edges in M, N and K (K not a multiple of the 32-deep slice).
SHAPES = [(128, 256, 64), (257, 513, 100), (1000, 1030, 333), (17, 300, 64), (640, 2304, 1000),
          (300, 520, 200)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_small_integers_bit_exact(M, N, K):
    check(M, N, K, 1.0, 0.0, dist="ints", exact=True)


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.5, 2.0)])
def test_floats_within_bound(M, N, K, alpha, beta):
    check(M, N, K, alpha, beta, dist="uniform")


def test_normal_inputs_within_bound():
    check(700, 900, 1500, 1.0, 0.0, dist="normal")


@pytest.mark.parametrize("bk,a_in_kernel,cps", [(16, False, 0), (32, True, 0), (32, False, 0),
                                                (16, None, 0), (16, True, 2), (16, False, 2),
                                                (16, None, 1)])
def test_kernel_forms_bitwise_identical(bk, a_in_kernel, cps):
    # Same split, same products, same order: the K depth of a stage and where
    # A is split do not change a bit of the result.
    M, N, K = 520, 770, 700
    A, lda, B, ldb, C, ldc = inputs("uniform", 5, M, N, K)
    sg.set_3xtf32_config(16, True)
    ref_out, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, ldc, entry=X3)
    sg.set_3xtf32_config(bk, a_in_kernel, 0, cps)
    try:
        out, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, ldc, entry=X3)
    finally:
        sg.set_3xtf32_config(16, None)
    assert np.array_equal(out.view(np.uint32), ref_out.view(np.uint32))
    ref, bound = reference(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, ldc)
    assert_within(out, ref, bound, f"3xTF32 bk={bk} a_in_kernel={a_in_kernel} cps={cps}")


@pytest.mark.parametrize("bk,a_in_kernel,cps", [(16, False, 0), (16, True, 0), (32, True, 0),
                                                (16, True, 2), (16, False, 2)])
def test_timeout_in_other_forms(bk, a_in_kernel, cps):
    sg.set_3xtf32_config(bk, a_in_kernel, 0, cps)
    try:
        test_wait_timeout_reports_and_recovers()
    finally:
        sg.set_3xtf32_config(16, None)


@pytest.mark.parametrize("a_in_kernel", [True, False])
@pytest.mark.parametrize("offsets,pad", [((1, 2, 3), (1, 3, 5)), ((0, 0, 0), (7, 1, 2)),
                                         ((4, 0, 0), (3, 0, 0))])
def test_unaligned_pointers_and_leading_dimensions(offsets, pad, a_in_kernel):
    # A that the TMA cannot map is copied to aligned rows when the kernel
    # splits it; the split pass reads any alignment.
    M, N, K = 300, 333, 257
    sg.set_3xtf32_config(16, a_in_kernel)
    try:
        check(M, N, K, 1.5, -0.5, lda=K + pad[0], ldb=N + pad[1], ldc=N + pad[2], offsets=offsets)
    finally:
        sg.set_3xtf32_config(16, None)


@pytest.mark.parametrize("M,N,K", [(16, 4096, 512), (300, 500, 63), (5, 7, 3)])
def test_short_products_take_the_ffma_kernels(M, N, K):
    # K < 64 or M <= 16: the same kernels and results as sgemm_run.
    A, lda, B, ldb, C, ldc = inputs("uniform", 9, M, N, K)
    out3, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, entry=X3)
    out1, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc)
    assert np.array_equal(out3.view(np.uint32), out1.view(np.uint32))


def test_bitwise_deterministic():
    M, N, K = 600, 700, 800
    A, lda, B, ldb, C, ldc = inputs("uniform", 4, M, N, K)
    o1, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, ldc, entry=X3)
    o2, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, ldc, entry=X3)
    assert np.array_equal(o1.view(np.uint32), o2.view(np.uint32))


@pytest.mark.parametrize("name", ["s2_2048", "s3_4092", "s4_rect"])
def test_workload_full_size(name):
    # Every element of the workloads the tensor-core entry point is timed on.
    cfg, A, B, C, ref, bound = workload_reference(name)
    M, N, K, alpha, beta = cfg["M"], cfg["N"], cfg["K"], cfg["alpha"], cfg["beta"]
    out, _ = run_gemm(M, N, K, alpha, beta, A, K, B, N, C, N,
                      c_fill=None if beta != 0 else float("nan"), entry=X3)
    assert np.isfinite(out).all()
    assert_within(out, ref, bound, f"3xTF32 {name}")
    ratio = float(np.max(np.abs(out - ref) / bound))
    print(f"3xTF32 {name}: max |err|/bound = {ratio:.3g}")


def test_torch_binding():
    M, N, K = 384, 512, 320
    A = torch.from_numpy(datagen.matrix("uniform", 8, "A", M, K)).cuda().view(M, K)
    B = torch.from_numpy(datagen.matrix("uniform", 8, "B", K, N)).cuda().view(K, N)
    C = torch.full((M, N), float("nan"), device="cuda")
    sg.run_3xtf32(A, B, C)
    torch.cuda.synchronize()
    ref, absprod = oracle.sgemm_ref_flat(M, N, K, 1.0, A.cpu().numpy().ravel(), K,
                                         B.cpu().numpy().ravel(), N, 0.0, None, N)
    assert_within(C.cpu().numpy(), ref, oracle.error_bound(absprod, None, 1.0, 0.0, K), "binding")


def test_wait_timeout_reports_and_recovers():
    M, N, K = 512, 1024, 1024
    A, lda, B, ldb, _, _ = inputs("uniform", 16, M, N, K)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.zeros(M * N, device="cuda")
    stream = torch.cuda.current_stream()
    # The load issuer stops at K slice 3, so the MMA issuer's wait for slice 3
    # runs out after 2 ms; the kernel records the timeout, lets its MMAs
    # finish, frees its tensor memory and returns.
    sg.set_wait_timeout_ns(2_000_000, 3)
    try:
        st = sg.sgemm_run_3xtf32(M, N, K, 1.0, dA.data_ptr(), lda, dB.data_ptr(), ldb, 0.0,
                                 dC.data_ptr(), N, stream.cuda_stream)
        assert st == 0
        assert sg.device_status(stream) == 5  # SGEMM_ERR_DEVICE_TIMEOUT
    finally:
        sg.set_wait_timeout_ns(0, -1)
    assert sg.device_status(stream) == 0
    out, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N, entry=X3)
    ref, bound = reference(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, N)
    assert_within(out, ref, bound, "3xTF32 after timeout")


@pytest.mark.parametrize("M,N,K", [(17, 100, 64), (200, 7, 64), (129, 129, 65), (300, 1000, 8192)])
def test_edges_of_the_tensor_core_path(M, N, K):
    # K at the hand-over (64), N far below the narrowest tile (128), odd
    # sizes one past a tile, and a long K (error growth of the FP32
    # accumulation in the tensor core): all within the bound.
    check(M, N, K, 1.0, 0.0, dist="uniform", seed=21)
    check(M, N, K, -0.75, 0.5, dist="normal", seed=22)


def test_nan_in_a_reaches_only_its_row():
    # IEEE semantics the FFMA path also has: a NaN in row i of A makes row i
    # of C NaN and leaves every other row finite and within the bound.
    M, N, K = 384, 512, 256
    A, lda, B, ldb, C, ldc = inputs("uniform", 23, M, N, K)
    A = A.copy()
    A[5 * lda + 17] = np.nan
    out, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, ldc, entry=X3)
    assert np.isnan(out[5]).all()
    rows = [r for r in range(M) if r != 5]
    assert np.isfinite(out[rows]).all()
    ref, bound = reference(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, ldc, rows=rows)
    assert_within(out[rows], ref, bound, "3xTF32 NaN row")


@pytest.mark.parametrize("a_in_kernel", [True, False])
def test_capture_in_a_cuda_graph_and_replay(a_in_kernel):
    # After a first call has sized the stream's workspace, the split pass and
    # the MMA kernel are queued without allocation or host synchronisation:
    # the call can be captured in a CUDA graph and replayed bit for bit.
    M, N, K = 640, 700, 512
    A, lda, B, ldb, C, ldc = inputs("uniform", 24, M, N, K)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC0 = torch.from_numpy(C).cuda()
    dC = dC0.clone()
    sg.set_3xtf32_config(16, a_in_kernel)
    try:
        side = torch.cuda.Stream()
        with torch.cuda.stream(side):
            assert sg.sgemm_run_3xtf32(M, N, K, 0.5, dA.data_ptr(), lda, dB.data_ptr(), ldb, 2.0,
                                       dC.data_ptr(), ldc, side.cuda_stream) == 0
        torch.cuda.synchronize()
        eager = dC.clone()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            st = sg.sgemm_run_3xtf32(M, N, K, 0.5, dA.data_ptr(), lda, dB.data_ptr(), ldb, 2.0,
                                     dC.data_ptr(), ldc, side.cuda_stream)
        assert st == 0
        for _ in range(3):
            dC.copy_(dC0)
            graph.replay()
            torch.cuda.synchronize()
            assert torch.equal(dC, eager)
        assert sg.device_status() == 0
    finally:
        sg.set_3xtf32_config(16, None)


@pytest.mark.parametrize("splits", [2, 3, 5])
def test_forced_k_split(splits):
    # Each K range writes its raw tile; the reduction adds the ranges in
    # order and applies alpha and beta.  Integers stay bit-exact (every
    # partial sum is exact), floats stay within the bound.
    M, N, K = 300, 520, 2000
    sg.set_3xtf32_config(16, None, splits)
    try:
        check(M, N, K, 1.0, 0.0, dist="ints", seed=31, exact=True)
        check(M, N, K, 0.5, 2.0, dist="uniform", seed=32)
        A, lda, B, ldb, C, ldc = inputs("uniform", 33, M, N, K)
        o1, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, ldc, entry=X3)
        o2, _ = run_gemm(M, N, K, 1.0, 0.0, A, lda, B, ldb, None, ldc, entry=X3)
        assert np.array_equal(o1.view(np.uint32), o2.view(np.uint32))
    finally:
        sg.set_3xtf32_config(16, None, 0)


@pytest.mark.parametrize("M,N,K", [(256, 512, 8192), (768, 768, 4096), (130, 1000, 3000)])
def test_deep_products_with_few_tiles(M, N, K):
    # The planner cuts these into K ranges (few tiles, long K).
    check(M, N, K, 1.0, 0.0, dist="uniform", seed=34)
    check(M, N, K, -1.5, 0.25, dist="normal", seed=35)


def test_timeout_with_a_k_split():
    sg.set_3xtf32_config(16, None, 2)
    try:
        test_wait_timeout_reports_and_recovers()
    finally:
        sg.set_3xtf32_config(16, None, 0)


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.5, 2.0)])
def test_two_ctas_per_sm_with_beta(alpha, beta):
    # The two-CTA form reads C directly (no room for the TMA C tile).
    sg.set_3xtf32_config(16, None, 0, 2)
    try:
        check(1000, 1030, 333, alpha, beta, dist="uniform", seed=41)
        check(257, 513, 100, alpha, beta, dist="ints", seed=42, exact=(beta == 0.0))
    finally:
        sg.set_3xtf32_config(16, None)


def _random_cases(seed, count):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(count):
        M = int(rng.integers(17, 1500))
        N = int(rng.integers(1, 1500))
        K = int(rng.integers(64, 3000))
        alpha = float(rng.choice([1.0, 0.5, -2.0]))
        beta = float(rng.choice([0.0, 1.0, -0.5]))
        bk = int(rng.choice([16, 32]))
        a_mode = [None, True, False][int(rng.integers(0, 3))]
        splits = int(rng.choice([0, 0, 2, 3, 8]))
        cps = 0 if bk == 32 else int(rng.choice([0, 1, 2]))
        cases.append((M, N, K, alpha, beta, bk, a_mode, splits, cps))
    return cases


@pytest.mark.parametrize("M,N,K,alpha,beta,bk,a_mode,splits,cps", _random_cases(2026, 24))
def test_random_shapes_and_forms(M, N, K, alpha, beta, bk, a_mode, splits, cps):
    # Seeded random shapes (ragged in every dimension) crossed with random
    # kernel forms, K splits and CTAs per SM: all within the bound.
    sg.set_3xtf32_config(bk, a_mode, splits, cps)
    try:
        check(M, N, K, alpha, beta, dist="uniform", seed=M + N + K)
    finally:
        sg.set_3xtf32_config(16, None)


# (M, N, K, splits, ctas per SM): the MMA kernel's store in both forms, the
# reduction of a K split, and the FFMA hand-over (M <= 16).
X3_EPI_CASES = [(300, 520, 256, 0, 0), (640, 1030, 1024, 0, 2), (300, 520, 2000, 3, 0),
                (16, 1024, 300, 0, 0)]


@pytest.mark.parametrize("activation", [0, 1])
@pytest.mark.parametrize("M,N,K,splits,cps", X3_EPI_CASES)
def test_epilogue_integers_bit_exact(M, N, K, splits, cps, activation):
    A, lda, B, ldb, C, ldc = inputs("ints", 51, M, N, K)
    bias = (np.arange(N) % 41 - 20).astype(np.float32)
    sg.set_3xtf32_config(16, None, splits, cps)
    try:
        out, _ = run_gemm(M, N, K, 1.0, 1.0, A, lda, B, ldb, C, ldc, bias=bias,
                          activation=activation, entry=X3)
    finally:
        sg.set_3xtf32_config(16, None)
    want = (A.reshape(M, lda)[:, :K].astype(np.int64) @ B.reshape(K, ldb)[:, :N].astype(np.int64)
            + C.reshape(M, ldc)[:, :N].astype(np.int64) + bias.astype(np.int64)[None, :])
    if activation == 1:
        want = np.maximum(want, 0)
    assert np.array_equal(out.astype(np.int64), want)


@pytest.mark.parametrize("M,N,K,splits,cps", X3_EPI_CASES)
def test_epilogue_floats_within_bound(M, N, K, splits, cps):
    A, lda, B, ldb, C, ldc = inputs("normal", 52, M, N, K, ldc=N + 4)
    bias = datagen.normal01(53, "C", N)
    sg.set_3xtf32_config(16, None, splits, cps)
    try:
        out, _ = run_gemm(M, N, K, 0.75, -0.5, A, lda, B, ldb, C, ldc, bias=bias, activation=1,
                          entry=X3)
    finally:
        sg.set_3xtf32_config(16, None)
    ref, absprod = oracle.sgemm_ref_flat(M, N, K, 0.75, A, lda, B, ldb, -0.5, C, ldc)
    want = oracle.apply_epilogue(ref, bias, oracle.ACT_RELU)
    bound = oracle.error_bound(absprod, C.reshape(M, ldc)[:, :N], 0.75, -0.5, K, bias=bias)
    assert_within(out, want, bound, f"3xTF32 epilogue {M}x{N}x{K} splits={splits} cps={cps}")
    assert (out >= 0).all()


def test_epilogue_torch_binding():
    M, N, K = 384, 512, 320
    A = torch.from_numpy(datagen.matrix("ints", 54, "A", M, K)).cuda().view(M, K)
    B = torch.from_numpy(datagen.matrix("ints", 54, "B", K, N)).cuda().view(K, N)
    C = torch.zeros(M, N, device="cuda")
    bias = torch.arange(N, dtype=torch.float32, device="cuda") - 256.0
    sg.run_3xtf32(A, B, C, bias=bias, activation=sg.ACT_RELU)
    torch.cuda.synchronize()
    want = torch.clamp(A.cpu().double() @ B.cpu().double() + bias.cpu().double(), min=0)
    assert torch.equal(C.cpu().double(), want)
