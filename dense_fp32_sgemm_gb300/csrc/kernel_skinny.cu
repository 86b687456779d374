// Skinny-M FP32 GEMM (M <= 16): the decode-like regime where B is streamed
// from HBM once and every B element feeds only M multiply-adds, so the
// kernel is bound by memory bandwidth, not by the FP32 pipe ("GEMM from
// Scratch", Module 08, "The Regime That Runs LLM Inference": a tall-skinny
// product re-reads all the weights and is memory-bound; Module 01: small or
// skinny matrices are not compute-bound).
//
// Work: N is cut into slabs of 256 columns; the (slab, k) plane is shared
// out in equal contiguous ranges of 32-row k-iterations to a persistent grid
// (stream-K over the slabs).  For each k-iteration a TMA copy brings the
// 32 x 256 block of B and the M x 32 block of A into a ring of shared-memory
// stages completed on mbarriers, several stages ahead, so enough bytes are in
// flight to keep HBM busy.  The threads rewrite A's block k-major with each
// value duplicated, (a, a), so a 128-bit shared load gives two packed
// operands for __ffma2_rn; a lane owns 8 columns (two groups of four, 128
// apart) and the eight warps take the 32 rows of a block round-robin.
//
// After a unit the eight warps' partial sums are added in warp order through
// shared memory; a unit covering part of a slab writes them to a fixed slot
// and the last CTA to arrive adds the pieces in CTA order (no CTA waits for
// another), then applies alpha and beta.

#include "device_common.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

constexpr int SBN = kSkinnyBN;      // 256 columns per slab
constexpr int SBK = kSkinnyBK;      // 32 rows of B per stage
constexpr int SNT = kSkinnyThreads;  // 256 threads
constexpr int SSTAGES = kSkinnyStages;
constexpr int WARPS = SNT / 32;
constexpr int CPL = 8;  // columns per lane
static_assert(32 * CPL == SBN, "one warp covers a slab row");

template <int MT>
struct SkinnyLayout {
    static constexpr int a_floats = MT * SBK;
    static constexpr int b_floats = SBK * SBN;
    static constexpr int stage_floats = a_floats + b_floats;
    static constexpr size_t stage_bytes = size_t(stage_floats) * 4;
    static constexpr int at_floats = SBK * 2 * MT;  // duplicated, k-major
    static constexpr int red_floats = WARPS * 4 * SBN;  // 4 rows of M per round
    static constexpr size_t at_off = SSTAGES * stage_bytes;
    static constexpr size_t red_off = at_off + 2 * size_t(at_floats) * 4;
    static constexpr size_t bar_off = red_off + size_t(red_floats) * 4;
    static constexpr size_t flag_off = bar_off + SSTAGES * 8;
    static constexpr size_t total = flag_off + 16;
    static constexpr uint32_t tx_bytes = stage_floats * 4;
    static_assert(total <= 232448, "exceeds the 227 KB of shared memory a CTA may use");
};

// One unit of work: k-iterations [k0, k1) of slab `slab`.
struct SkinnyIter {
    int u, end;
    __device__ __forceinline__ void init(const SkinnyParams &p, int cta) {
        const int total = p.slabs * p.kt_total;
        u = min(cta * p.share, total);
        end = min(u + p.share, total);
    }
    __device__ __forceinline__ bool next(const SkinnyParams &p, int &slab, int &k0, int &k1) {
        if (u >= end) return false;
        slab = u / p.kt_total;
        k0 = u - slab * p.kt_total;
        k1 = min(p.kt_total, k0 + (end - u));
        u += k1 - k0;
        return true;
    }
};

__device__ __forceinline__ int skinny_slot(const SkinnyParams &p, int cta, int slab) {
    const int start = slab * p.kt_total;
    const int k0 = max(cta * p.share, start) - start;
    return 2 * cta + (k0 == 0 ? 1 : 0);
}

// A block (MT rows x 32 k, k fastest) -> k-major duplicated pairs.
template <int MT>
__device__ __forceinline__ void skinny_transpose(const float *raw, float *at, int tid) {
    if (tid < MT * (SBK / 4)) {
        const int m = tid / (SBK / 4), kc = tid % (SBK / 4);
        const float4 v = ld_shared_f4(raw + m * SBK + kc * 4);
        const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<float2 *>(at + (kc * 4 + i) * 2 * MT + 2 * m) = make_float2(e[i], e[i]);
    }
}

template <int MT>
__global__ void __launch_bounds__(SNT, 1)
    sgemm_skinny_kernel(const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapB, const SkinnyParams p) {
    using L = SkinnyLayout<MT>;
    extern __shared__ __align__(1024) uint8_t smem[];
    float *stages = reinterpret_cast<float *>(smem);
    float *at_buf = reinterpret_cast<float *>(smem + L::at_off);
    float *red = reinterpret_cast<float *>(smem + L::red_off);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + L::flag_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;

    SkinnyIter it0;
    it0.init(p, cta);
    const int q_total = it0.end - it0.u;
    if (q_total <= 0) return;

    if (tid == 0) {
        for (int s = 0; s < SSTAGES; ++s) mbar_init(&full[s], 1);
        flags[0] = 0;
        flags[1] = 0;
        fence_barrier_init();
        prefetch_tensormap(&mapA);
        prefetch_tensormap(&mapB);
    }
    __syncthreads();

    // ---- copy producer (thread 0) ----
    SkinnyIter prod = it0;
    int pq = 0, p_slab = 0, p_k = 0, p_k1 = 0;
    auto issue_next = [&]() {
        if (pq >= q_total) return;
        if (p.skip_loads_from >= 0 && pq >= p.skip_loads_from) return;
        if (p_k >= p_k1) prod.next(p, p_slab, p_k, p_k1);
        const int s = pq % SSTAGES;
        float *sa = stages + s * L::stage_floats;
        float *sb = sa + L::a_floats;
        mbar_arrive_expect_tx(&full[s], L::tx_bytes);
        tma_load_2d(sa, &mapA, &full[s], p_k * SBK, 0);
        tma_load_2d(sb, &mapB, &full[s], p_slab * SBN, p_k * SBK);
        ++p_k;
        ++pq;
    };
    if (tid == 0)
        for (int s = 0; s < SSTAGES; ++s) issue_next();

    SkinnyIter cons = it0;
    int q = 0;
    bool aborted = false;
    if (!mbar_wait_bounded(&full[0], 0, p.timeout_ns)) {
        flags[0] = 1;
        atomicOr(p.err, kErrWaitTimeout);
    }
    skinny_transpose<MT>(stages, at_buf, tid);
    __syncthreads();
    if (flags[0]) aborted = true;

    int slab, k0, k1;
    while (!aborted && cons.next(p, slab, k0, k1)) {
        float2 acc[MT][CPL / 2];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int j = 0; j < CPL / 2; ++j) acc[m][j] = make_float2(0.f, 0.f);

        for (int kt = k0; kt < k1; ++kt, ++q) {
            const int s = q % SSTAGES;
            if (q + 1 < q_total) {
                const int s1 = (q + 1) % SSTAGES;
                if (!mbar_wait_bounded(&full[s1], ((q + 1) / SSTAGES) & 1, p.timeout_ns)) {
                    flags[0] = 1;
                    atomicOr(p.err, kErrWaitTimeout);
                }
                skinny_transpose<MT>(stages + s1 * L::stage_floats,
                                     at_buf + ((q + 1) & 1) * L::at_floats, tid);
            }
            const float *at = at_buf + (q & 1) * L::at_floats;
            const float *bs = stages + s * L::stage_floats + L::a_floats;
#pragma unroll
            for (int r = 0; r < SBK / WARPS; ++r) {
                const int k = warp + r * WARPS;
                const float4 b0 = ld_shared_f4(bs + k * SBN + lane * 4);
                const float4 b1 = ld_shared_f4(bs + k * SBN + 128 + lane * 4);
                const float2 bp[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                                      make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
                for (int m2 = 0; m2 < MT / 2; ++m2) {
                    const float4 a = ld_shared_f4(at + k * 2 * MT + m2 * 4);
                    const float2 a0 = make_float2(a.x, a.y), a1 = make_float2(a.z, a.w);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[2 * m2][j] = __ffma2_rn(a0, bp[j], acc[2 * m2][j]);
                        acc[2 * m2 + 1][j] = __ffma2_rn(a1, bp[j], acc[2 * m2 + 1][j]);
                    }
                }
            }
            __syncthreads();
            if (flags[0]) {
                aborted = true;
                ++q;
                break;
            }
            if (tid == 0) issue_next();
        }
        if (aborted) break;

        // ---- add the eight warps' sums in warp order; thread t owns column t ----
        float fin[MT];
#pragma unroll
        for (int mr = 0; mr < MT / 4; ++mr) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = mr * 4 + i;
                float *dst = red + (warp * 4 + i) * SBN;
                *reinterpret_cast<float4 *>(dst + lane * 4) =
                    make_float4(acc[m][0].x, acc[m][0].y, acc[m][1].x, acc[m][1].y);
                *reinterpret_cast<float4 *>(dst + 128 + lane * 4) =
                    make_float4(acc[m][2].x, acc[m][2].y, acc[m][3].x, acc[m][3].y);
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float sum = red[(0 * 4 + i) * SBN + tid];
#pragma unroll
                for (int w = 1; w < WARPS; ++w) sum += red[(w * 4 + i) * SBN + tid];
                fin[mr * 4 + i] = sum;
            }
            __syncthreads();
        }

        const int n = slab * SBN + tid;
        bool write_c = true;
        if (!(k0 == 0 && k1 == p.kt_total)) {
            float *slot = p.partials + (size_t)skinny_slot(p, cta, slab) * (kSkinnyMaxM * SBN);
#pragma unroll
            for (int m = 0; m < MT; ++m) __stcg(slot + m * SBN + tid, fin[m]);
            __threadfence();
            __syncthreads();
            const int c_first = (slab * p.kt_total) / p.share;
            const int c_last = (slab * p.kt_total + p.kt_total - 1) / p.share;
            if (tid == 0) {
                const int old = atomicAdd(&p.counters[slab], 1);
                flags[1] = (old == c_last - c_first) ? 1 : 0;
            }
            __syncthreads();
            write_c = flags[1] != 0;
            if (write_c) {
                __threadfence();
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float s = 0.f;
                    for (int cc = c_first; cc <= c_last; ++cc) {
                        const float v =
                            (cc == cta) ? fin[m]
                                        : __ldcg(p.partials +
                                                 (size_t)skinny_slot(p, cc, slab) * (kSkinnyMaxM * SBN) +
                                                 m * SBN + tid);
                        s = (cc == c_first) ? v : s + v;
                    }
                    fin[m] = s;
                }
                if (tid == 0) p.counters[slab] = 0;
            }
        }
        if (write_c && n < p.N) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                if (m < p.M) {
                    float *c = p.C + (long long)m * p.ldc + n;
                    float o = p.alpha * fin[m];
                    if (p.beta != 0.0f) o = __fmaf_rn(p.beta, *c, o);
                    *c = o;
                }
            }
        }
    }

    if (aborted && tid == 0) {
        for (int j = q; j < pq; ++j) {
            if (!mbar_wait_bounded(&full[j % SSTAGES], (j / SSTAGES) & 1, 1000000000ull)) {
                atomicOr(p.err, kErrDrainTimeout);
                break;
            }
        }
    }
}

}  // namespace

size_t skinny_smem_bytes(int m_tile, int /*share*/) {
    if (m_tile == 8) return SkinnyLayout<8>::total;
    if (m_tile == 16) return SkinnyLayout<16>::total;
    return 0;
}

cudaError_t skinny_configure(int m_tile) {
    if (m_tile == 8)
        return cudaFuncSetAttribute(sgemm_skinny_kernel<8>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)SkinnyLayout<8>::total);
    if (m_tile == 16)
        return cudaFuncSetAttribute(sgemm_skinny_kernel<16>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)SkinnyLayout<16>::total);
    return cudaErrorInvalidValue;
}

cudaError_t launch_skinny(int m_tile, const CUtensorMap &mapA, const CUtensorMap &mapB,
                          const SkinnyParams &p, int grid, cudaStream_t stream) {
    if (m_tile == 8) {
        sgemm_skinny_kernel<8><<<grid, SNT, SkinnyLayout<8>::total, stream>>>(mapA, mapB, p);
    } else if (m_tile == 16) {
        sgemm_skinny_kernel<16><<<grid, SNT, SkinnyLayout<16>::total, stream>>>(mapA, mapB, p);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace sgemm
