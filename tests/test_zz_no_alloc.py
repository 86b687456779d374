"""sgemm_run_skinny_noalloc: the skinny-M product for callers that cannot call
cudaMalloc (code running under a framework allocator that owns the device
memory, loops that must not allocate after start-up).  Its partial sums and
tickets live in a fixed buffer compiled into the library instead of a
workspace allocated on first use.

Checked through the C ABI against sgemm_run, the entry point that allocates
its workspace, on two calls in a row (the second one sees the buffer exactly
as the first left it), within the elementwise FP32 bound the other tests use.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import datagen
import dense_fp32_sgemm_gb300 as sg
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sg.build()
    sg.set_plan_override(-1, 0)


def one_case(M, N, K, alpha, beta, seed):
    lib = sg.library()
    A = datagen.matrix("uniform", seed, "A", M, K)
    B = datagen.matrix("uniform", seed, "B", K, N)
    C = datagen.matrix("uniform", seed, "C", M, N)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    c_alloc = torch.from_numpy(C).cuda()
    c_fixed = torch.from_numpy(C).cuda()
    s = torch.cuda.current_stream().cuda_stream
    st = lib.sgemm_run(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                       c_alloc.data_ptr(), N, s)
    assert st == 0, sg.status_string(st)
    st = lib.sgemm_run_skinny_noalloc(M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta,
                                      c_fixed.data_ptr(), N, s)
    assert st == 0, sg.status_string(st)
    torch.cuda.synchronize()
    got = c_fixed.cpu().numpy().reshape(M, N).astype(np.float64)
    want = c_alloc.cpu().numpy().reshape(M, N).astype(np.float64)
    _, absprod = oracle.sgemm_ref_flat(M, N, K, alpha, A, K, B, N, beta, C, N)
    bound = oracle.error_bound(absprod, C.reshape(M, N), alpha, beta, K)
    err = np.abs(got - want)
    assert (err <= bound).all(), f"max |noalloc - sgemm_run| / bound = {(err / bound).max()}"


def test_noalloc_matches_sgemm_run_on_two_calls_in_a_row():
    one_case(16, 8192, 4096, 1.0, 0.0, 2001)
    one_case(7, 3000, 1000, 0.5, 2.0, 2002)


def test_noalloc_rejects_requests_beyond_its_buffer():
    lib = sg.library()
    buf = torch.zeros(1 << 16, device="cuda")
    p = buf.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    assert lib.sgemm_run_skinny_noalloc(17, 64, 64, 1.0, p, 64, p, 64, 0.0, p, 64, s) == 8
    assert lib.sgemm_run_skinny_noalloc(4, 64, 63, 1.0, p, 63, p, 64, 0.0, p, 64, s) == 8
    assert sg.status_string(8) == "SGEMM_ERR_SCRATCH_LIMIT"
