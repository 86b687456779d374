"""Python binding of the GB300 FP32 SGEMM library (libsgemm_gb300.so).

Argument marshalling only: every step of C = alpha*A*B + beta*C runs in the
library's CUDA kernels.  The functions mirror the C ABI in include/sgemm.h
and include/sgemm_probe.h; ``run`` and ``run_host`` add the conversion from
torch tensors / numpy arrays to pointers and leading dimensions.

There is no fallback: if the library has not been built, or no sm_103 GPU is
present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

__all__ = [
    "SgemmError", "build", "library", "library_path", "sgemm_run", "sgemm_run_epilogue",
    "sgemm_run_host", "ACT_NONE", "ACT_RELU",
    "run", "run_host", "status_string", "device_status", "plan_describe",
    "set_plan_override", "set_wait_timeout_ns", "set_tile_config",
    "release_workspace", "probe_ffma", "probe_read", "probe_hold", "probe_tf32", "EXPORTED_SYMBOLS",
    "VARIANT_AUTO", "VARIANT_GENERIC", "VARIANT_TILE", "VARIANT_STREAMK",
    "VARIANT_SKINNY", "VARIANT_MID", "VARIANT_MID64", "VARIANT_KSPLIT", "VARIANT_NARROW", "VARIANT_KSPLIT64", "VARIANT_SMALL",
    "STATUS",
]

STATUS = {
    0: "SGEMM_OK", 1: "SGEMM_ERR_INVALID_ARG", 2: "SGEMM_ERR_ALLOC",
    3: "SGEMM_ERR_TMA", 4: "SGEMM_ERR_LAUNCH", 5: "SGEMM_ERR_DEVICE_TIMEOUT",
    6: "SGEMM_ERR_NO_DEVICE", 7: "SGEMM_ERR_UNSUPPORTED", 8: "SGEMM_ERR_SCRATCH_LIMIT",
}
VARIANT_AUTO, VARIANT_GENERIC, VARIANT_TILE, VARIANT_STREAMK, VARIANT_SKINNY = -1, 0, 1, 2, 3
VARIANT_MID, VARIANT_MID64, VARIANT_KSPLIT, VARIANT_NARROW, VARIANT_KSPLIT64 = 4, 5, 6, 7, 8
VARIANT_SMALL = 9
ACT_NONE, ACT_RELU = 0, 1

_i64, _f32, _vp, _int = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int

# name -> (restype, argtypes); one entry per function declared in include/*.h
_SIGNATURES = {
    "sgemm_run": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]),
    "sgemm_run_epilogue": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64,
                                  _vp, _int, _vp]),
    "sgemm_run_host": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]),
    "sgemm_run_skinny_noalloc": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp,
                                        _i64, _vp]),
    "sgemm_run_3xtf32": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]),
    "sgemm_run_3xtf32_epilogue": (_int, [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp,
                                         _i64, _vp, _int, _vp]),
    "sgemm_set_3xtf32_config": (_int, [_int, _int, _int, _int]),
    "sgemm_status_string": (ctypes.c_char_p, [_int]),
    "sgemm_device_status": (_int, [_vp]),
    "sgemm_skinny_noalloc_status": (_int, [_vp]),
    "sgemm_plan_describe": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, ctypes.c_uint64,
                                   ctypes.c_uint64, ctypes.c_uint64, _f32, _int,
                                   ctypes.c_char_p, ctypes.c_size_t]),
    "sgemm_plan_describe_3xtf32": (_int, [_i64, _i64, _i64, _i64, ctypes.c_uint64, _int,
                                          ctypes.c_char_p, ctypes.c_size_t]),
    "sgemm_set_plan_override": (_int, [_int, _int]),
    "sgemm_set_wait_timeout_ns": (_int, [ctypes.c_uint64, _int]),
    "sgemm_set_tile_config": (_int, [_int, _int, _int]),
    "sgemm_release_workspace": (_int, []),
    "sgemm_probe_ffma": (_int, [_int, _i64, _int, _vp, _vp]),
    "sgemm_probe_read": (_int, [_vp, _i64, _vp, _int, _vp]),
    "sgemm_probe_hold": (_int, [_i64, _vp]),
    "sgemm_probe_tf32": (_int, [_i64, _int, _vp]),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lib = None
_lock = threading.Lock()


class SgemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = STATUS.get(status, f"status {status}")
        super().__init__(f"{what}: {name}" if what else name)


def library_path() -> str:
    return _build.LIB_PATH


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    return _build.build(force=force)


def library() -> ctypes.CDLL:
    """Load the built library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing: build it first "
                    "(dense_fp32_sgemm_gb300.build() or __graft_entry__.build())")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def _check(status: int, what: str) -> None:
    if status != 0:
        raise SgemmError(status, what)


def status_string(status: int) -> str:
    return library().sgemm_status_string(int(status)).decode()


def sgemm_run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """Raw C-ABI call with integer device addresses; returns the status."""
    return library().sgemm_run(int(M), int(N), int(K), float(alpha), A, int(lda), B, int(ldb),
                               float(beta), C, int(ldc), stream)


def sgemm_run_epilogue(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias=None,
                       activation=ACT_NONE, stream=None) -> int:
    """Raw C-ABI call of C = act(alpha*A*B + beta*C + bias); returns the status."""
    return library().sgemm_run_epilogue(int(M), int(N), int(K), float(alpha), A, int(lda), B,
                                        int(ldb), float(beta), C, int(ldc), bias,
                                        int(activation), stream)


def sgemm_run_3xtf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """Raw C-ABI call of the 3xTF32 tensor-core variant; returns the status."""
    return library().sgemm_run_3xtf32(int(M), int(N), int(K), float(alpha), A, int(lda), B,
                                      int(ldb), float(beta), C, int(ldc), stream)


def sgemm_run_3xtf32_epilogue(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias=None,
                              activation=ACT_NONE, stream=None) -> int:
    """Raw C-ABI call of the 3xTF32 variant with bias / activation."""
    return library().sgemm_run_3xtf32_epilogue(int(M), int(N), int(K), float(alpha), A, int(lda),
                                               B, int(ldb), float(beta), C, int(ldc), bias,
                                               int(activation), stream)


def sgemm_run_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None) -> int:
    """Raw C-ABI call with integer host addresses; returns the status."""
    return library().sgemm_run_host(int(M), int(N), int(K), float(alpha), A, int(lda), B,
                                    int(ldb), float(beta), C, int(ldc), stream)


def _matrix_args(t, name):
    if str(t.dtype) != "torch.float32":
        raise TypeError(f"{name} must be float32")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D")
    rows, cols = t.shape
    if cols > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit column stride (row-major)")
    ld = t.stride(0) if rows > 1 else max(1, cols)
    return t.data_ptr(), max(ld, cols, 1)


def run(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None, bias=None,
        activation: int = ACT_NONE):
    """C = act(alpha * A @ B + beta * C + bias) in place on CUDA float32 tensors.

    Tensors are row-major with unit column stride; a row stride larger than
    the row length is passed on as the leading dimension.  ``bias`` is None or
    a contiguous CUDA float32 tensor of N elements, added to every row;
    ``activation`` is ACT_NONE or ACT_RELU.  ``stream`` is a torch.cuda.Stream
    (default: the current stream).  Returns C.
    """
    import torch

    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)} B {tuple(B.shape)} C {tuple(C.shape)}")
    for t, name in ((A, "A"), (B, "B"), (C, "C")):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    a, lda = _matrix_args(A, "A")
    b, ldb = _matrix_args(B, "B")
    c, ldc = _matrix_args(C, "C")
    bias_ptr = None
    if bias is not None:
        if not bias.is_cuda or str(bias.dtype) != "torch.float32" or bias.numel() != N or (
                bias.dim() != 1 and not bias.is_contiguous()) or (bias.dim() == 1 and bias.stride(0) != 1):
            raise ValueError("bias must be a contiguous CUDA float32 tensor of N elements")
        bias_ptr = bias.data_ptr()
    s = (stream or torch.cuda.current_stream(C.device)).cuda_stream
    with torch.cuda.device(C.device):
        if bias_ptr is None and activation == ACT_NONE:
            _check(sgemm_run(M, N, K, alpha, a, lda, b, ldb, beta, c, ldc, s), "sgemm_run")
        else:
            _check(sgemm_run_epilogue(M, N, K, alpha, a, lda, b, ldb, beta, c, ldc, bias_ptr,
                                      activation, s), "sgemm_run_epilogue")
    return C


def run_3xtf32(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None, bias=None,
               activation: int = ACT_NONE):
    """C = act(alpha * A @ B + beta * C + bias) in place, on the tensor cores
    by the 3xTF32 split (hi*hi + hi*lo + lo*hi of TF32 parts, FP32
    accumulation).  Same tensors and conventions as run()."""
    import torch

    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch: A {tuple(A.shape)} B {tuple(B.shape)} C {tuple(C.shape)}")
    for t, name in ((A, "A"), (B, "B"), (C, "C")):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    a, lda = _matrix_args(A, "A")
    b, ldb = _matrix_args(B, "B")
    c, ldc = _matrix_args(C, "C")
    s = (stream or torch.cuda.current_stream(C.device)).cuda_stream
    bias_ptr = None
    if bias is not None:
        if not bias.is_cuda or str(bias.dtype) != "torch.float32" or bias.numel() != N or (
                bias.dim() != 1 and not bias.is_contiguous()) or (bias.dim() == 1 and bias.stride(0) != 1):
            raise ValueError("bias must be a contiguous CUDA float32 tensor of N elements")
        bias_ptr = bias.data_ptr()
    with torch.cuda.device(C.device):
        if bias_ptr is None and activation == ACT_NONE:
            _check(sgemm_run_3xtf32(M, N, K, alpha, a, lda, b, ldb, beta, c, ldc, s),
                   "sgemm_run_3xtf32")
        else:
            _check(sgemm_run_3xtf32_epilogue(M, N, K, alpha, a, lda, b, ldb, beta, c, ldc, bias_ptr,
                                             activation, s), "sgemm_run_3xtf32_epilogue")
    return C


def set_3xtf32_config(bk: int = 16, a_in_kernel=None, splits: int = 0,
                      ctas_per_sm: int = 0) -> None:
    """3xTF32 kernel form: K depth of one pipeline stage (16, default, or 32);
    whether A is split inside the kernel (True), by a split pass (False) or as
    the library chooses per call (None, default); K ranges per output tile
    (1 to 8, or 0 = chosen per call); CTAs per SM (1, 2, or 0 = chosen per
    call)."""
    mode = -1 if a_in_kernel is None else int(bool(a_in_kernel))
    _check(library().sgemm_set_3xtf32_config(int(bk), mode, int(splits), int(ctas_per_sm)),
           "sgemm_set_3xtf32_config")


def run_host(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """The same on host matrices (numpy arrays or CPU tensors, ideally pinned).

    Copies in, computes, copies C back and synchronises before returning.
    """
    import numpy as np

    def host_args(x, name):
        if hasattr(x, "data_ptr"):
            return _matrix_args(x, name) + (tuple(x.shape),)
        arr = x
        if arr.dtype != np.float32 or arr.ndim != 2:
            raise TypeError(f"{name} must be a 2-D float32 array")
        if arr.shape[1] > 1 and arr.strides[1] != 4:
            raise ValueError(f"{name} must have unit column stride")
        ld = arr.strides[0] // 4 if arr.shape[0] > 1 else max(1, arr.shape[1])
        return arr.ctypes.data, max(ld, arr.shape[1], 1), arr.shape

    a, lda, (M, K) = host_args(A, "A")
    b, ldb, (K2, N) = host_args(B, "B")
    c, ldc, cshape = host_args(C, "C")
    if K2 != K or tuple(cshape) != (M, N):
        raise ValueError("shape mismatch")
    s = None
    if stream is not None:
        s = stream.cuda_stream
    _check(sgemm_run_host(M, N, K, alpha, a, lda, b, ldb, beta, c, ldc, s), "sgemm_run_host")
    return C


def device_status(stream=None) -> int:
    s = stream.cuda_stream if stream is not None else None
    return int(library().sgemm_device_status(s))


def plan_describe(M, N, K, lda=None, ldb=None, ldc=None, a_addr=0, b_addr=0, c_addr=0,
                  beta=0.0, num_sms=0) -> dict:
    """The plan sgemm_run would take, as a dict of strings (host only)."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    ldc = N if ldc is None else ldc
    buf = ctypes.create_string_buffer(512)
    _check(library().sgemm_plan_describe(int(M), int(N), int(K), int(max(lda, 1)),
                                         int(max(ldb, 1)), int(max(ldc, 1)), int(a_addr),
                                         int(b_addr), int(c_addr), float(beta), int(num_sms),
                                         buf, len(buf)), "sgemm_plan_describe")
    # key=value pairs; the last one, reason, is free text.
    head, sep, reason = buf.value.decode().partition(" reason=")
    out = {}
    for kv in head.split():
        k, _, v = kv.partition("=")
        out[k] = v
    if sep:
        out["reason"] = reason
    return out


def plan_describe_3xtf32(M, N, K, lda=None, a_addr=0, num_sms=0) -> dict:
    """What sgemm_run_3xtf32 would do for these sizes (host only), as a dict of
    strings: path (ffma or tensor) and, for the tensor path, bk, stages,
    ctas_per_sm, a_in_kernel, tile_n, splits, kt and ctas."""
    lda = K if lda is None else lda
    buf = ctypes.create_string_buffer(256)
    _check(library().sgemm_plan_describe_3xtf32(int(M), int(N), int(K), int(max(lda, 1)),
                                                int(a_addr), int(num_sms), buf, len(buf)),
           "sgemm_plan_describe_3xtf32")
    return dict(kv.partition("=")[::2] for kv in buf.value.decode().split())


def set_plan_override(variant: int = VARIANT_AUTO, splits: int = 0) -> None:
    _check(library().sgemm_set_plan_override(int(variant), int(splits)), "sgemm_set_plan_override")


def set_wait_timeout_ns(timeout_ns: int = 0, skip_loads_from: int = -1) -> None:
    _check(library().sgemm_set_wait_timeout_ns(int(timeout_ns), int(skip_loads_from)),
           "sgemm_set_wait_timeout_ns")


def set_tile_config(fma_mode: int = 3, stages: int = 3, micro_m: int = 16) -> None:
    _check(library().sgemm_set_tile_config(int(fma_mode), int(stages), int(micro_m)),
           "sgemm_set_tile_config")


def release_workspace() -> None:
    _check(library().sgemm_release_workspace(), "sgemm_release_workspace")


def probe_ffma(paired: bool, iters: int, blocks: int, sink_ptr: int, stream=None) -> float:
    """Queue the FFMA probe; returns the FLOPs it performs."""
    s = stream.cuda_stream if stream is not None else None
    _check(library().sgemm_probe_ffma(1 if paired else 0, int(iters), int(blocks), sink_ptr, s),
           "sgemm_probe_ffma")
    return float(blocks) * 512 * iters * 128 * 2


def probe_tf32(iters: int, blocks: int, stream=None) -> float:
    """Queue the tcgen05 TF32 rate probe; returns the FLOPs it performs."""
    s = stream.cuda_stream if stream is not None else None
    _check(library().sgemm_probe_tf32(int(iters), int(blocks), s), "sgemm_probe_tf32")
    return float(blocks) * iters * 4 * 2 * 128 * 256 * 8


def probe_read(buf_ptr: int, n_floats: int, sink_ptr: int, blocks: int, stream=None) -> float:
    """Queue the streaming-read probe; returns the bytes it reads."""
    s = stream.cuda_stream if stream is not None else None
    _check(library().sgemm_probe_read(buf_ptr, int(n_floats), sink_ptr, int(blocks), s),
           "sgemm_probe_read")
    return 4.0 * n_floats


def probe_hold(ns: int, stream=None) -> None:
    """Queue a kernel that keeps `stream` busy for `ns` nanoseconds."""
    s = stream.cuda_stream if stream is not None else None
    _check(library().sgemm_probe_hold(int(ns), s), "sgemm_probe_hold")
