// Narrow SIMT FP32 GEMM for sm_103a: C = alpha * A * B + beta * C, row-major,
// for N <= kNarrowMaxN columns (a matrix-vector product A x when N = 1), and
// for the last few columns of C when the tiled kernel takes the rest.
//
// Every element of A feeds only N multiply-adds, so the product is bound by
// streaming A ("GEMM from Scratch", Module 01: small and skinny shapes are not
// compute-bound; the mirror of the small-M case of Module 08).  A tile of 128
// or more columns would spend at least 128 / N times the multiply-adds, most
// of them on zeros.  Here each warp takes one row of A at a time and its lanes
// walk K four consecutive k at a time (16-byte loads when A's rows are 16-byte
// aligned, else 4-byte loads), so a warp instruction reads 512 (or 128)
// consecutive bytes; B's N columns are staged transposed in shared memory
// (b[j][k]), all of K at once when it fits (else in chunks), and read back
// with 128-bit loads.
//
// A CTA of 8 warps owns a contiguous range of rows, taken in groups of up to
// four passes of eight; for each staged chunk of B every pass of a group
// walks the chunk in steps of 1024 k, each lane's loads of the next step in flight
// while the current one is multiplied (32 values of A a lane; loads issued
// one 128-k group at a time and waited for before the next read 2.7 TB/s at
// 8192 x 1 x 8192).  Barriers come only where a new chunk of B is staged: once
// per CTA when K fits one chunk, else once per chunk and group (staging per
// pass read 110 us at 8192 x 4 x 8192); a lane's k are the same, and taken in
// the same order, however K is chunked.  A lane keeps N sums over its k (in increasing k), and the
// warp adds its lanes' sums with a fixed butterfly of shuffles, so the result
// does not depend on timing.  No CTA depends on another.

#include "device_common.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

constexpr int NW = 8;            // warps per CTA
constexpr int NTH = NW * 32;
constexpr int KI = 8;            // 4-k groups a lane loads per step
constexpr int STEP = 128 * KI;   // k per step of a warp: 1024

// The full steps' 16-byte loads of A, which is read once: through the
// non-coherent path without allocating in L1 (8192 x 1 x 8192: 47.1-48.1 us
// against 48.8-49.1 with L1 allocation; 8192 x 4 x 8192 57.3-57.6 against
// 58.9).  Volatile, so that no load is moved ahead
// of the check that the whole step lies inside the row.  The bounds-checked
// loads of a row's last step keep __ldg: as volatile predicated loads they made
// 100000 x 1 x 1000 (every row a single short step) 88 us against 73.
__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// A lane's A values of one step: a[i] holds k = 4 lane + 128 i + (0..3) of
// the step (zeros past kn).  Full steps load without bounds checks, so all KI
// loads of a lane are in flight together.
template <int AVEC>
__device__ __forceinline__ void narrow_load_a(const float *a_step, int kn, int lane,
                                              float4 (&a)[KI]) {
    if (kn >= STEP) {
#pragma unroll
        for (int i = 0; i < KI; ++i) {
            const float *q = a_step + 4 * lane + 128 * i;
            if (AVEC == 4) {
                a[i] = ld_stream_f4(q);
            } else {
                a[i] = make_float4(__ldg(q), __ldg(q + 1), __ldg(q + 2), __ldg(q + 3));
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < KI; ++i) {
            const int kk = 4 * lane + 128 * i;
            const float *q = a_step + kk;
            a[i].x = kk + 0 < kn ? __ldg(q + 0) : 0.0f;
            a[i].y = kk + 1 < kn ? __ldg(q + 1) : 0.0f;
            a[i].z = kk + 2 < kn ? __ldg(q + 2) : 0.0f;
            a[i].w = kk + 3 < kn ? __ldg(q + 3) : 0.0f;
        }
    }
}

// B[k0 .. k0 + kch) transposed into bs (row stride kch + 4), zeros past K
// and past N, with 4-byte asynchronous copies (a source size of 0 writes the
// zero): they take no registers, so all of a thread's copies are in flight
// at once, and the chunk costs about one L2 round trip.  Thread t copies
// column t % NN of rows t / NN, t / NN + NTH / NN, ...; consecutive threads
// read consecutive columns of one row of B.  Returns once this thread's
// copies have landed; the caller's barrier publishes them.
template <int NN>
__device__ __forceinline__ void narrow_stage_b(const NarrowParams &p, float *bs, int k0, int kch) {
    static_assert(NTH % NN == 0, "a thread keeps its column");
    constexpr int KSTEP = NTH / NN;  // rows of B between a thread's copies
    const int kn = min(kch, p.K - k0);
    const int j = threadIdx.x % NN;
    const bool col_ok = j < p.N;
    float *dst = bs + j * (kch + 4);
    const float *src = p.B + (long long)k0 * p.ldb + j;
    for (int kk = threadIdx.x / NN; kk < kch; kk += KSTEP) {
        const bool ok = col_ok && kk < kn;
        cp_async4(dst + kk, ok ? src + (long long)kk * p.ldb : p.B, ok ? 4u : 0u);
    }
    cp_async_commit();
    cp_async_wait<0>();
}

constexpr int PMAX = 4;  // passes of eight rows that share one staging of B

template <int NN, int AVEC>
__global__ void __launch_bounds__(NTH) sgemm_narrow_kernel(const __grid_constant__ NarrowParams p) {
    extern __shared__ __align__(16) float bs[];  // bs[j * (kch + 4) + kk] = B[k0 + kk][j]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long r0 = (long long)blockIdx.x * p.rows_per_cta;
    const long long r1 = min((long long)p.M, r0 + p.rows_per_cta);
    const int kch = p.kch;
    const int chunks = (p.K + kch - 1) / kch;
    const int brow = kch + 4;
    // One chunk (K <= kch): B is staged once for every row of the CTA.
    if (chunks == 1) {
        narrow_stage_b<NN>(p, bs, 0, kch);
        __syncthreads();
    }

    // Groups of up to PMAX passes of eight rows (uniform over the CTA).
#pragma unroll 1
    for (long long g0 = r0; g0 < r1; g0 += PMAX * NW) {
        const int npass = (int)min((long long)PMAX, (r1 - g0 + NW - 1) / NW);
        // Pass ps takes row g0 + 8 ps + warp of this warp.
        const float *arow[PMAX];
        bool act[PMAX];
#pragma unroll
        for (int ps = 0; ps < PMAX; ++ps) {
            const long long row = g0 + ps * NW + warp;
            act[ps] = ps < npass && row < r1;
            arow[ps] = p.A + (act[ps] ? row : r0) * p.lda;
        }
        float acc[PMAX][NN];
#pragma unroll
        for (int ps = 0; ps < PMAX; ++ps)
#pragma unroll
            for (int j = 0; j < NN; ++j) acc[ps][j] = 0.0f;

        // Steps of STEP k: for every chunk of B, every pass walks the chunk;
        // the next step's loads are issued before this step's multiply-adds
        // (and before a chunk's barriers and staging), so B is staged once
        // per chunk for the group's rows.
        float4 a_next[KI];
        if (act[0]) narrow_load_a<AVEC>(arow[0], min(STEP, min(kch, p.K)), lane, a_next);

#pragma unroll 1
        for (int c = 0; c < chunks; ++c) {
            const int k0 = c * kch;
            const int kn = min(kch, p.K - k0);
            if (chunks > 1) {
                __syncthreads();  // the previous chunk of B is consumed
                narrow_stage_b<NN>(p, bs, k0, kch);
                __syncthreads();
            }
#pragma unroll
            for (int ps = 0; ps < PMAX; ++ps) {
                if (ps >= npass) break;  // uniform over the CTA
#pragma unroll 1
                for (int s0 = 0; s0 < kn; s0 += STEP) {
                    float4 a[KI];
#pragma unroll
                    for (int i = 0; i < KI; ++i) a[i] = a_next[i];
                    if (s0 + STEP < kn) {
                        if (act[ps])
                            narrow_load_a<AVEC>(arow[ps] + k0 + s0 + STEP,
                                                min(STEP, kn - s0 - STEP), lane, a_next);
                    } else if (ps + 1 < npass) {
                        if (ps + 1 < PMAX && act[ps + 1])
                            narrow_load_a<AVEC>(arow[ps + 1] + k0, min(STEP, kn), lane, a_next);
                    } else if (c + 1 < chunks) {
                        if (act[0])
                            narrow_load_a<AVEC>(arow[0] + k0 + kch,
                                                min(STEP, min(kch, p.K - k0 - kch)), lane, a_next);
                    }
                    if (act[ps]) {
#pragma unroll
                        for (int i = 0; i < KI; ++i) {
                            // Groups past the chunk's end hold zeros of A;
                            // they are skipped (uniform over the warp), so
                            // that every read of bs stays inside row j.
                            if (s0 + 128 * i >= kn) break;
                            const int kk = s0 + 4 * lane + 128 * i;
#pragma unroll
                            for (int j = 0; j < NN; ++j) {
                                const float4 b = ld_shared_f4(bs + j * brow + kk);
                                acc[ps][j] = __fmaf_rn(a[i].x, b.x, acc[ps][j]);
                                acc[ps][j] = __fmaf_rn(a[i].y, b.y, acc[ps][j]);
                                acc[ps][j] = __fmaf_rn(a[i].z, b.z, acc[ps][j]);
                                acc[ps][j] = __fmaf_rn(a[i].w, b.w, acc[ps][j]);
                            }
                        }
                    }
                }
            }
        }
        // Per row: the lanes' sums added by a fixed butterfly (every lane
        // ends with the same total); lane j stores column j.
#pragma unroll
        for (int ps = 0; ps < PMAX; ++ps) {
            if (ps >= npass) break;
#pragma unroll
            for (int j = 0; j < NN; ++j)
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    acc[ps][j] += __shfl_xor_sync(0xffffffffu, acc[ps][j], off);
            float mine = acc[ps][0];
#pragma unroll
            for (int j = 1; j < NN; ++j) mine = lane == j ? acc[ps][j] : mine;
            if (act[ps] && lane < NN && lane < p.N) {
                float *c = p.C + (g0 + ps * NW + warp) * p.ldc + lane;
                float v = p.alpha * mine;
                if (p.beta != 0.0f) v = __fmaf_rn(p.beta, *c, v);
                *c = apply_epilogue(v, p.epi, lane);
            }
        }
    }
}

template <int NN, int AVEC>
cudaError_t launch_impl(const NarrowParams &p, int grid, cudaStream_t stream) {
    const size_t smem = (size_t)NN * (p.kch + 4) * sizeof(float);
    if (p.kch <= 0 || p.kch % 128 != 0 || smem > kNarrowSmemBytes) return cudaErrorInvalidValue;
    sgemm_narrow_kernel<NN, AVEC><<<grid, NTH, smem, stream>>>(p);
    return cudaGetLastError();
}

// No carveout preference: A's 16-byte loads go through L1, and with the
// largest shared-memory carveout (L1 shrunk to its minimum) 8192 x 1 x 8192
// took 53.2 us against 49.2, 8192 x 4 x 8192 67.6 against 58.9.
template <int NN, int AVEC>
cudaError_t configure_impl() {
    return cudaFuncSetAttribute(sgemm_narrow_kernel<NN, AVEC>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kNarrowSmemBytes);
}

}  // namespace

cudaError_t narrow_configure(int nn, int a_vec) {
#define SGEMM_NARROW_CONF(NN_, AV_) \
    if (nn == NN_ && a_vec == AV_) return configure_impl<NN_, AV_>();
    SGEMM_NARROW_CONF(1, 4) SGEMM_NARROW_CONF(1, 1)
    SGEMM_NARROW_CONF(2, 4) SGEMM_NARROW_CONF(2, 1)
    SGEMM_NARROW_CONF(4, 4) SGEMM_NARROW_CONF(4, 1)
#undef SGEMM_NARROW_CONF
    return cudaErrorInvalidValue;
}

cudaError_t launch_narrow(int nn, int a_vec, const NarrowParams &p, int grid, cudaStream_t stream) {
#define SGEMM_NARROW_LAUNCH(NN_, AV_) \
    if (nn == NN_ && a_vec == AV_) return launch_impl<NN_, AV_>(p, grid, stream);
    SGEMM_NARROW_LAUNCH(1, 4) SGEMM_NARROW_LAUNCH(1, 1)
    SGEMM_NARROW_LAUNCH(2, 4) SGEMM_NARROW_LAUNCH(2, 1)
    SGEMM_NARROW_LAUNCH(4, 4) SGEMM_NARROW_LAUNCH(4, 1)
#undef SGEMM_NARROW_LAUNCH
    return cudaErrorInvalidValue;
}

}  // namespace sgemm
