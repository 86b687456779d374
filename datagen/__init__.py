"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no GEMM arithmetic: it only turns (seed, tensor id, shape)
into float32 matrices.  Both the CUDA path and the oracle are fed from here;
neither is imported by it.

Generator: SplitMix64 in counter form.  For the stream with initial state s0,
output i (i >= 0) is mix(s0 + (i + 1) * GAMMA), where mix is the SplitMix64
finaliser (xor-shift 30, multiply, xor-shift 27, multiply, xor-shift 31) and
GAMMA = 0x9E3779B97F4A7C15.  The stream of a matrix is s0 = (seed << 8) | tid,
tid being 0 for A, 1 for B and 2 for C, so the three operands never share a
stream.

Distributions (the configurations ask for uniform[-1, 1] or normal(0, 1)
entries "from seed" and name no generator):
- uniform: the top 24 bits n of each output give (n - 2^23) / 2^23, a value in
  [-1, 1) that float32 holds exactly;
- normal: Box-Muller in double on outputs (2i, 2i+1), u1 in (0, 1] and
  u2 in [0, 1) from their top 53 bits, z = sqrt(-2 ln u1) cos(2 pi u2),
  rounded to float32;
- ints: small integers in [-lim, lim] (x mod (2 lim + 1) - lim), for cases
  that must come out bit-exact;
- ones: all ones.
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TENSOR_ID = {"A": 0, "B": 1, "C": 2}

_CHUNK = 1 << 20


def splitmix64_scalar(state: int):
    """Reference scalar SplitMix64 step: returns (new_state, output)."""
    mask = (1 << 64) - 1
    state = (state + 0x9E3779B97F4A7C15) & mask
    z = state
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & mask
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & mask
    return state, z ^ (z >> 31)


def _splitmix64_chunk(out, tmp, base, first):
    """Fill out[:] with outputs first, first+1, ... (first counted from 0)."""
    n = out.shape[0]
    with np.errstate(over="ignore"):
        out[:] = np.arange(first + 1, first + 1 + n, dtype=np.uint64)
        np.multiply(out, GAMMA, out=out)
        np.add(out, base, out=out)
        np.right_shift(out, np.uint64(30), out=tmp)
        np.bitwise_xor(out, tmp, out=out)
        np.multiply(out, _M1, out=out)
        np.right_shift(out, np.uint64(27), out=tmp)
        np.bitwise_xor(out, tmp, out=out)
        np.multiply(out, _M2, out=out)
        np.right_shift(out, np.uint64(31), out=tmp)
        np.bitwise_xor(out, tmp, out=out)


def _parallel_chunks(count: int, dtype, fill):
    """out[off:off+n] = fill(off, n) over chunks, on a thread pool.

    numpy releases the GIL in its ufuncs; every value depends only on its own
    index, so the result does not depend on how the range is split.
    """
    out = np.empty(count, dtype=dtype)
    offsets = list(range(0, count, _CHUNK))

    def work(off):
        n = min(_CHUNK, count - off)
        out[off:off + n] = fill(off, n)

    if len(offsets) <= 1:
        for off in offsets:
            work(off)
    else:
        import concurrent.futures as cf
        import os
        workers = min(len(offsets), os.cpu_count() or 1, 16)
        with cf.ThreadPoolExecutor(max_workers=workers) as pool:
            list(pool.map(work, offsets))
    return out


def _stream_chunk(s0: int, first: int, n: int) -> np.ndarray:
    z = np.empty(n, dtype=np.uint64)
    _splitmix64_chunk(z, np.empty(n, dtype=np.uint64),
                      np.uint64(s0 & ((1 << 64) - 1)), first)
    return z


def splitmix64(s0: int, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of the stream with initial state s0."""
    return _parallel_chunks(count, np.uint64,
                            lambda off, n: _stream_chunk(s0, start + off, n))


def stream_state(seed: int, tensor: str | int) -> int:
    tid = TENSOR_ID[tensor] if isinstance(tensor, str) else int(tensor)
    if not 0 <= tid < 256:
        raise ValueError("tensor id must fit in 8 bits")
    if not 0 <= seed < (1 << 56):
        raise ValueError("seed must be in [0, 2^56)")
    return (int(seed) << 8) | tid


def uniform_pm1(seed: int, tensor, count: int) -> np.ndarray:
    s0 = stream_state(seed, tensor)

    def fill(off, n):
        x = _stream_chunk(s0, off, n)
        v = (x >> np.uint64(40)).astype(np.int32) - (1 << 23)
        return v.astype(np.float32) * np.float32(2.0 ** -23)

    return _parallel_chunks(count, np.float32, fill)


def normal01(seed: int, tensor, count: int) -> np.ndarray:
    s0 = stream_state(seed, tensor)

    def fill(off, n):
        x = _stream_chunk(s0, 2 * off, 2 * n)
        u1 = ((x[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (x[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)

    return _parallel_chunks(count, np.float32, fill)


def small_ints(seed: int, tensor, count: int, lim: int = 8) -> np.ndarray:
    s0 = stream_state(seed, tensor)

    def fill(off, n):
        x = _stream_chunk(s0, off, n)
        return (x % np.uint64(2 * lim + 1)).astype(np.int64) - lim

    return _parallel_chunks(count, np.float32, fill)


def values(dist: str, seed: int, tensor, count: int) -> np.ndarray:
    if dist == "uniform":
        return uniform_pm1(seed, tensor, count)
    if dist == "normal":
        return normal01(seed, tensor, count)
    if dist == "ints":
        return small_ints(seed, tensor, count)
    if dist == "ones":
        return np.ones(count, dtype=np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def matrix(dist: str, seed: int, tensor, rows: int, cols: int,
           ld: int | None = None, gap_fill: float = float("nan")) -> np.ndarray:
    """A rows x cols matrix in a flat float32 buffer with leading dimension ld.

    Returns the flat buffer of rows*ld elements (the last row is padded to ld
    too).  Elements in the gap between cols and ld hold ``gap_fill`` (NaN by
    default, so a kernel that reads the gap poisons its result).
    """
    ld = cols if ld is None else int(ld)
    if ld < cols:
        raise ValueError("ld must be >= cols")
    vals = values(dist, seed, tensor, rows * cols).reshape(rows, cols)
    if ld == cols:
        return vals.reshape(-1)
    buf = np.full((rows, ld), gap_fill, dtype=np.float32)
    buf[:, :cols] = vals
    return buf.reshape(-1)


# The configurations the workloads are drawn from: shape, alpha, beta,
# distribution.  Seeds are 1000 + index.
CONFIGS = {
    "s1_128": dict(M=128, N=128, K=128, alpha=1.0, beta=0.0, dist="uniform"),
    "s2_2048": dict(M=2048, N=2048, K=2048, alpha=1.0, beta=0.0, dist="uniform"),
    "s3_4092": dict(M=4092, N=4092, K=4092, alpha=0.5, beta=2.0, dist="uniform"),
    "s4_rect": dict(M=8192, N=6144, K=2048, alpha=1.0, beta=0.0, dist="normal"),
    "s5_odd": dict(M=1023, N=1025, K=513, alpha=1.0, beta=0.0, dist="normal"),
    "s6_skinny": dict(M=16, N=8192, K=8192, alpha=1.0, beta=0.0, dist="uniform"),
    # one row of A: the decode-step GEMV (matrix-vector) case of the skinny regime
    "s7_gemv": dict(M=1, N=8192, K=8192, alpha=1.0, beta=0.0, dist="uniform"),
    # one past the tile size in every dimension (the last tile row and column
    # hold one useful row or column)
    "s8_2049": dict(M=2049, N=2049, K=2049, alpha=1.0, beta=0.0, dist="uniform"),
    # one column of B: the matrix-vector product A x
    "s9_ax": dict(M=8192, N=1, K=8192, alpha=1.0, beta=0.0, dist="uniform"),
}
CONFIG_SEEDS = {name: 1000 + i for i, name in enumerate(CONFIGS)}


def config_inputs(name: str):
    """(cfg, A, B, C) flat float32 buffers (row-major, ld = row length).

    C is generated only when beta != 0; otherwise it is None.
    """
    cfg = CONFIGS[name]
    seed = CONFIG_SEEDS[name]
    M, N, K, dist = cfg["M"], cfg["N"], cfg["K"], cfg["dist"]
    A = matrix(dist, seed, "A", M, K)
    B = matrix(dist, seed, "B", K, N)
    C = matrix(dist, seed, "C", M, N) if cfg["beta"] != 0.0 else None
    return cfg, A, B, C
