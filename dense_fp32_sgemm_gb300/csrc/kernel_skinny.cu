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
// 32 x 256 block of B and the M x 32 block of A (128-byte swizzled rows) into
// a ring of shared-memory stages completed on mbarriers, several stages
// ahead, so enough bytes are in flight to keep HBM busy.
//
// Lanes own groups of four columns (so a quarter-warp's 128-bit loads cover
// 32 consecutive banks): with 8 columns per lane, 8 warps each cover the
// whole 256-column row; with 4, 16 warps cover it in halves.  Row group g
// (one per 8 rows) takes rows g, g + 8, g + 16, g + 24 of each block.  A warp rewrites only
// the four A columns it needs k-major into its own corner of shared memory,
// so no CTA-wide barrier is needed inside a unit: warps run through the
// stages independently, and the last warp to finish with a stage (a counter
// in shared memory) refills it.  The update is the packed FP32 fma
// (__ffma2_rn) on pairs along m: (a_m, a_m+1) * (b_n, b_n).
//
// After a unit the eight row groups' sums are added in group order through
// shared memory; a unit covering part of a slab writes them to a fixed slot
// and the last CTA to arrive adds the pieces in CTA order (no CTA waits for
// another), then applies alpha and beta.

#include "device_common.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

constexpr int SBN = kSkinnyBN;       // 256 columns per slab
constexpr int SBK = kSkinnyBK;       // 32 rows of B per stage
constexpr int SNT = kSkinnyThreads;
constexpr int SSTAGES = kSkinnyStages;
constexpr int CPL = kSkinnyCPL;            // columns per lane: 8 (8 warps) or 4 (16 warps)
constexpr int HALVES = 8 / CPL;            // warps sharing one row of a block
constexpr int WARPS = SNT / 32;
constexpr int GROUPS = WARPS / HALVES;     // row groups
constexpr int RPW = SBK / GROUPS;          // rows of a block per warp
static_assert(RPW == 4 && GROUPS == 8 && 32 * CPL * HALVES == SBN, "warp layout");

template <int MT>
struct SkinnyLayout {
    static constexpr int a_floats = MT * SBK;  // M x 32, 128-byte rows, swizzled
    static constexpr int b_floats = SBK * SBN;
    static constexpr int stage_floats = a_floats + b_floats;
    static constexpr size_t stage_bytes = size_t(stage_floats) * 4;
    static_assert(stage_bytes % 1024 == 0, "stages must keep 1024-byte alignment");
    static constexpr int at_floats = RPW * MT;  // per warp: 4 k x MT m
    static constexpr int RED_ROWS = 2;  // rows of M per reduction round
    static constexpr int red_floats = GROUPS * RED_ROWS * SBN;
    static constexpr size_t at_off = SSTAGES * stage_bytes;
    static constexpr size_t red_off = at_off + size_t(WARPS) * at_floats * 4;
    static constexpr size_t bar_off = red_off + size_t(red_floats) * 4;
    static constexpr size_t cnt_off = bar_off + SSTAGES * 8;
    static constexpr size_t flag_off = cnt_off + SSTAGES * 4 * 2;
    static constexpr size_t total = flag_off + 16;
    static constexpr uint32_t tx_bytes = stage_floats * 4;
    static_assert(total <= 232448, "exceeds the 227 KB of shared memory a CTA may use");
};

__device__ __forceinline__ int skinny_slot(const SkinnyParams &p, int cta, int slab) {
    const int start = slab * p.kt_total;
    const int k0 = max(cta * p.share, start) - start;
    return 2 * cta + (k0 == 0 ? 1 : 0);
}

// Element (m, k) of the TMA-loaded A block: rows of 32 floats whose 16-byte
// chunks are XOR-swizzled with (row mod 8).
__device__ __forceinline__ float a_elem(const float *raw, int m, int k) {
    return raw[m * SBK + ((((k >> 2) ^ (m & 7)) << 2) | (k & 3))];
}

template <int MT>
__global__ void __launch_bounds__(SNT, 1)
    sgemm_skinny_kernel(const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapB, const SkinnyParams p) {
    using L = SkinnyLayout<MT>;
    extern __shared__ __align__(1024) uint8_t smem[];
    float *stages = reinterpret_cast<float *>(smem);
    float *red = reinterpret_cast<float *>(smem + L::red_off);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    int *release = reinterpret_cast<int *>(smem + L::cnt_off);
    volatile int *issued = reinterpret_cast<volatile int *>(smem + L::cnt_off + SSTAGES * 4);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + L::flag_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = warp / HALVES, h = warp % HALVES;
    const int cta = blockIdx.x;
    float *at_w = reinterpret_cast<float *>(smem + L::at_off) + warp * L::at_floats;

    const int total = p.slabs * p.kt_total;
    const int u0 = min(cta * p.share, total);
    const int q_total = min(u0 + p.share, total) - u0;
    if (q_total <= 0) return;

    // Copy of position q (the CTA's q-th k-iteration) into stage q % SSTAGES.
    auto issue = [&](int q) {
        if (p.skip_loads_from >= 0 && q >= p.skip_loads_from) return;
        const int s = q % SSTAGES;
        const int u = u0 + q;
        const int slab = u / p.kt_total, k = u - slab * p.kt_total;
        float *sa = stages + s * L::stage_floats;
        issued[s] = q;
        mbar_arrive_expect_tx(&full[s], L::tx_bytes);
        tma_load_2d(sa, &mapA, &full[s], k * SBK, 0);
        tma_load_2d(sa + L::a_floats, &mapB, &full[s], slab * SBN, k * SBK);
    };

    if (tid == 0) {
        for (int s = 0; s < SSTAGES; ++s) {
            mbar_init(&full[s], 1);
            release[s] = 0;
            issued[s] = -1;
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_barrier_init();
        prefetch_tensormap(&mapA);
        prefetch_tensormap(&mapB);
    }
    __syncthreads();
    if (tid == 0)
        for (int q = 0; q < SSTAGES && q < q_total; ++q) issue(q);

    int q = 0;
    bool aborted = false;
    int timed_out = 0;  // this thread saw a wait run out (made uniform at unit end)
    while (q < q_total && !aborted) {
        const int u = u0 + q;
        const int slab = u / p.kt_total;
        const int k0 = u - slab * p.kt_total;
        const int k1 = min(p.kt_total, k0 + (q_total - q));

        float2 acc[MT / 2][CPL];  // acc[ip][j] = (C[2ip][n_j], C[2ip+1][n_j])
#pragma unroll
        for (int i = 0; i < MT / 2; ++i)
#pragma unroll
            for (int j = 0; j < CPL; ++j) acc[i][j] = make_float2(0.f, 0.f);

        for (int kt = k0; kt < k1; ++kt, ++q) {
            const int s = q % SSTAGES;
            // After a timeout anywhere in the CTA (flags[0], a hint) the
            // remaining waits are skipped; the garbage computed is discarded.
            if (!timed_out && !flags[0] &&
                !mbar_wait_bounded(&full[s], (q / SSTAGES) & 1, p.timeout_ns)) {
                timed_out = 1;
                flags[0] = 1;
                atomicOr(p.err, kErrWaitTimeout);
            }
            const float *raw = stages + s * L::stage_floats;
            const float *bs = raw + L::a_floats;
            // This warp's A columns k = g + 8 * kk, k-major: at_w[kk * MT + m].
#pragma unroll
            for (int e = lane; e < RPW * MT; e += 32) {
                const int m = e % MT, kk = e / MT;
                at_w[kk * MT + m] = a_elem(raw, m, g + GROUPS * kk);
            }
            __syncwarp();

            const float *bcol = bs + h * 128 + lane * 4;
            float4 bf[2][CPL / 4];
#pragma unroll
            for (int c = 0; c < CPL / 4; ++c) bf[0][c] = ld_shared_f4(bcol + g * SBN + c * 128);
#pragma unroll
            for (int kk = 0; kk < RPW; ++kk) {
                const int cur = kk & 1, nxt = cur ^ 1;
                if (kk + 1 < RPW) {
                    const float *brow = bcol + (g + GROUPS * (kk + 1)) * SBN;
#pragma unroll
                    for (int c = 0; c < CPL / 4; ++c) bf[nxt][c] = ld_shared_f4(brow + c * 128);
                }
                float b[CPL];
#pragma unroll
                for (int c = 0; c < CPL / 4; ++c) {
                    b[4 * c + 0] = bf[cur][c].x;
                    b[4 * c + 1] = bf[cur][c].y;
                    b[4 * c + 2] = bf[cur][c].z;
                    b[4 * c + 3] = bf[cur][c].w;
                }
                // A values of this row: broadcast loads from the warp's own
                // k-major copy.
#pragma unroll
                for (int r = 0; r < MT / 4; ++r) {
                    const float4 a = ld_shared_f4(at_w + kk * MT + r * 4);
                    const float2 a01 = make_float2(a.x, a.y);
                    const float2 a23 = make_float2(a.z, a.w);
#pragma unroll
                    for (int j = 0; j < CPL; ++j) {
                        const float2 bb = make_float2(b[j], b[j]);
                        acc[2 * r][j] = __ffma2_rn(a01, bb, acc[2 * r][j]);
                        acc[2 * r + 1][j] = __ffma2_rn(a23, bb, acc[2 * r + 1][j]);
                    }
                }
            }
            __syncwarp();
            // Release the stage; the last of the 16 warps refills it.
            if (lane == 0) {
                __threadfence_block();
                const int old = atomicAdd(&release[s], 1);
                if (old == WARPS - 1) {
                    release[s] = 0;
                    if (q + SSTAGES < q_total && !flags[0]) {
                        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        issue(q + SSTAGES);
                    }
                }
            }
        }

        // Abort uniformly if any thread of the CTA gave up a wait in this unit.
        if (__syncthreads_or(timed_out)) {
            aborted = true;
            break;
        }

        // ---- add the eight row groups' sums in group order ----
        // Thread t owns column t and all MT rows.
        constexpr int RR = L::RED_ROWS;
        float fin[MT];
#pragma unroll
        for (int r = 0; r < MT / RR; ++r) {
#pragma unroll
            for (int i = 0; i < RR; ++i) {
                const int m = RR * r + i;
#pragma unroll
                for (int c = 0; c < CPL / 4; ++c) {
                    float4 v;
                    v.x = (m & 1) ? acc[m >> 1][4 * c + 0].y : acc[m >> 1][4 * c + 0].x;
                    v.y = (m & 1) ? acc[m >> 1][4 * c + 1].y : acc[m >> 1][4 * c + 1].x;
                    v.z = (m & 1) ? acc[m >> 1][4 * c + 2].y : acc[m >> 1][4 * c + 2].x;
                    v.w = (m & 1) ? acc[m >> 1][4 * c + 3].y : acc[m >> 1][4 * c + 3].x;
                    *reinterpret_cast<float4 *>(red + (g * RR + i) * SBN + h * 128 + c * 128 +
                                                lane * 4) = v;
                }
            }
            __syncthreads();
#pragma unroll
            for (int i = 0; i < RR; ++i) {
                const int col = tid & (SBN - 1);
                float sum = red[i * SBN + col];
#pragma unroll
                for (int gg = 1; gg < GROUPS; ++gg) sum += red[(gg * RR + i) * SBN + col];
                fin[RR * r + i] = sum;
            }
            __syncthreads();
        }

        // With 512 threads the upper half repeats the lower half's sums and
        // stores nothing.
        const int col = tid & (SBN - 1);
        const bool owner = tid < SBN;
        const int n = slab * SBN + col;
        bool write_c = true;
        if (!(k0 == 0 && k1 == p.kt_total)) {
            float *slot = p.partials + (size_t)skinny_slot(p, cta, slab) * (kSkinnyMaxM * SBN);
            if (owner) {
#pragma unroll
                for (int m = 0; m < MT; ++m) __stcg(slot + m * SBN + col, fin[m]);
            }
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
                // Pieces are added in CTA order.  The loads of every other
                // piece for a group of rows are issued together, so a group
                // costs one L2 round trip (up to kFastPieces pieces; more
                // take a plain loop).
                constexpr int kFastPieces = 6;
                const int npieces = c_last - c_first + 1;
                if (npieces <= kFastPieces) {
#pragma unroll
                    for (int m0 = 0; m0 < MT; m0 += 2) {
                        float v[kFastPieces][2];
#pragma unroll
                        for (int i = 0; i < kFastPieces; ++i) {
                            const int cc = c_first + i;
                            if (cc <= c_last && cc != cta) {
                                const float *slot = p.partials +
                                                    (size_t)skinny_slot(p, cc, slab) * (kSkinnyMaxM * SBN) +
                                                    col;
#pragma unroll
                                for (int r = 0; r < 2; ++r) v[i][r] = __ldcg(slot + (m0 + r) * SBN);
                            }
                        }
#pragma unroll
                        for (int r = 0; r < 2; ++r) {
                            const float own = fin[m0 + r];
                            float sum = own;
#pragma unroll
                            for (int i = 0; i < kFastPieces; ++i) {
                                const int cc = c_first + i;
                                if (cc > c_last) break;
                                const float x = (cc == cta) ? own : v[i][r];
                                sum = (i == 0) ? x : sum + x;
                            }
                            fin[m0 + r] = sum;
                        }
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        float sum = 0.f;
                        for (int cc = c_first; cc <= c_last; ++cc) {
                            const float v =
                                (cc == cta) ? fin[m]
                                            : __ldcg(p.partials +
                                                     (size_t)skinny_slot(p, cc, slab) * (kSkinnyMaxM * SBN) +
                                                     m * SBN + col);
                            sum = (cc == c_first) ? v : sum + v;
                        }
                        fin[m] = sum;
                    }
                }
                if (tid == 0) p.counters[slab] = 0;
            }
            __syncthreads();  // flags[1] is rewritten by the next unit
        }
        if (write_c && owner && n < p.N) {
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
        // Wait (bounded) for the last copy issued into every stage, so none
        // lands in shared memory after this CTA has exited.
        for (int s = 0; s < SSTAGES; ++s) {
            const int last = issued[s];
            if (last < 0) continue;
            if (!mbar_wait_bounded(&full[s], (last / SSTAGES) & 1, 1000000000ull)) {
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
