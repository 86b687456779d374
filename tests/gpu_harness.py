"""Device-side harness for the GPU tests: places seeded host matrices in
device buffers with guard bands, calls the library through its C ABI and
checks that nothing outside C's M x N elements was written."""
from __future__ import annotations

import numpy as np
import torch

import dense_fp32_sgemm_gb300 as sg

GUARD = 1024          # floats of canary before and after every buffer
CANARY = 12345.678    # float32-exact enough to compare bitwise after a round trip


def same_bits(a, b) -> bool:
    """Bitwise equality (NaN canaries compare equal to themselves)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    return a.shape == b.shape and bool(np.array_equal(a.view(np.uint32), b.view(np.uint32)))


class DeviceMatrix:
    """rows x ld float32 buffer on the GPU at a chosen float offset from a
    256-byte aligned allocation, surrounded by canaries."""

    def __init__(self, flat: np.ndarray | None, rows: int, ld: int, offset: int = 0,
                 fill: float | None = None):
        self.rows, self.ld, self.offset = rows, ld, offset
        n = max(rows * ld, 1)
        self.n = n
        host = np.full(GUARD + offset + n + GUARD, CANARY, dtype=np.float32)
        if flat is not None:
            host[GUARD + offset:GUARD + offset + flat.size] = flat
        elif fill is not None:
            host[GUARD + offset:GUARD + offset + n] = fill
        self.host_init = host
        self.buf = torch.from_numpy(host).to("cuda")

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr() + 4 * (GUARD + self.offset)

    def to_host(self) -> np.ndarray:
        return self.buf.cpu().numpy()

    def region(self, host=None) -> np.ndarray:
        host = self.to_host() if host is None else host
        return host[GUARD + self.offset:GUARD + self.offset + self.n]

    def guards_intact(self, host=None) -> bool:
        host = self.to_host() if host is None else host
        lo = host[:GUARD + self.offset]
        hi = host[GUARD + self.offset + self.n:]
        return bool(same_bits(lo, self.host_init[:GUARD + self.offset])
                    and same_bits(hi, self.host_init[GUARD + self.offset + self.n:]))


def run_gemm(M, N, K, alpha, beta, A, lda, B, ldb, C, ldc, offsets=(0, 0, 0),
             variant=-1, splits=0, c_fill=None, bias=None, activation=0, entry="sgemm_run"):
    """Run sgemm_run (sgemm_run_epilogue when a bias or an activation is
    given; sgemm_run_3xtf32 with entry="sgemm_run_3xtf32") on device copies;
    returns (C result as M x N float32, the DeviceMatrix for C)."""
    dA = DeviceMatrix(A, M, lda, offsets[0])
    dB = DeviceMatrix(B, K, ldb, offsets[1])
    dC = DeviceMatrix(C, M, ldc, offsets[2], fill=c_fill)
    dbias = DeviceMatrix(bias, 1, N) if bias is not None else None
    sg.set_plan_override(variant, splits)
    try:
        stream = torch.cuda.current_stream().cuda_stream
        if entry == "sgemm_run_3xtf32" and (bias is not None or activation != 0):
            st = sg.sgemm_run_3xtf32_epilogue(M, N, K, alpha, dA.ptr, lda, dB.ptr, ldb, beta,
                                              dC.ptr, ldc,
                                              dbias.ptr if dbias is not None else None,
                                              activation, stream)
        elif entry == "sgemm_run_3xtf32":
            st = sg.sgemm_run_3xtf32(M, N, K, alpha, dA.ptr, lda, dB.ptr, ldb, beta, dC.ptr, ldc,
                                     stream)
        elif bias is None and activation == 0:
            st = sg.sgemm_run(M, N, K, alpha, dA.ptr, lda, dB.ptr, ldb, beta, dC.ptr, ldc, stream)
        else:
            st = sg.sgemm_run_epilogue(M, N, K, alpha, dA.ptr, lda, dB.ptr, ldb, beta, dC.ptr, ldc,
                                       dbias.ptr if dbias is not None else None, activation,
                                       stream)
    finally:
        sg.set_plan_override(-1, 0)
    assert st == 0, sg.status_string(st)
    dev = sg.device_status(torch.cuda.current_stream())
    assert dev == 0, sg.status_string(dev)
    host = dC.to_host()
    assert dA.guards_intact() and dB.guards_intact(), "an operand buffer was written"
    if dbias is not None:
        assert dbias.guards_intact() and same_bits(dbias.region(), dbias.region(dbias.host_init)), \
            "the bias buffer was written"
    assert dC.guards_intact(host), "C's guard band was written"
    region = dC.region(host)
    out = region[:M * ldc].reshape(M, ldc) if M * ldc else np.zeros((M, ldc), np.float32)
    if ldc > N and M > 0:
        gap = out[:, N:]
        init = dC.region(dC.host_init)[:M * ldc].reshape(M, ldc)[:, N:]
        assert same_bits(gap, init), "C's leading-dimension gap was written"
    return out[:, :N].copy(), dC
