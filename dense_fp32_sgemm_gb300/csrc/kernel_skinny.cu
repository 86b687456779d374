// Skinny-M FP32 GEMM (M <= 32): the decode-like regime where B is streamed
// from HBM once and every B element feeds only M multiply-adds, so the
// kernel is bound by memory bandwidth, not by the FP32 pipe ("GEMM from
// Scratch", Module 08, "The Regime That Runs LLM Inference": a tall-skinny
// product re-reads all the weights and is memory-bound; Module 01: small or
// skinny matrices are not compute-bound).
//
// Work: N is cut into slabs of 256 columns; the (slab, k) plane of 32-row
// k-iterations ("positions") is shared out in contiguous ranges to a
// persistent grid (stream-K over the slabs), balanced in time by the planner:
// a range that crosses a slab boundary is shorter by the cost of its extra
// unit end.  For each k-iteration a TMA copy brings the
// 32 x 256 block of B and the M x 32 block of A (128-byte swizzled rows) into
// a ring of shared-memory stages completed on mbarriers, several stages
// ahead, so enough bytes are in flight to keep HBM busy.
//
// One CTA of 8 warps per SM holds a 6-stage ring (5 stages with a 32-row A
// tile; with the 4-warp build, two CTAs of 4 warps share an SM, 3 stages
// each).  Each lane owns 8 columns (two groups of four, so a quarter-warp's
// 128-bit loads cover 32 consecutive banks) and a warp the whole 256-column
// row.  With 16 rows of A the warps form two groups of four that take
// alternate positions, 8 rows of each block per warp; with 32 rows the two
// groups share every position, group g summing rows 16 g .. 16 g + 15 (so a
// thread still holds 16 x 8 sums); with 8 rows all 8 warps share every
// position, 4 rows each.  Either way warp w of a group takes rows w, w + W,
// w + 2W, ... of a block (W warps in the group).  A warp rewrites only the A columns it needs
// k-major into its own corner of shared memory, so no CTA-wide barrier is
// needed inside a unit: warps run through the stages independently, and the
// last warp of the group to finish with a stage (a counter in shared memory)
// refills it with the position SSTAGES further on, which belongs to the same
// group (with split rows, the last of all eight warps).  The update is the packed FP32 fma (__ffma2_rn) on pairs along m:
// (a_m, a_m+1) * (b_n, b_n).
//
// After a unit the warps' sums are added in warp order through shared
// memory; a unit covering part of a slab writes them to a fixed slot and the
// last CTA to arrive adds the pieces in CTA order (no CTA waits for another),
// then applies alpha and beta.  When that CTA has no copies outstanding (its
// last unit) it fetches the other pieces with bulk copies into its idle ring.

#include "device_common.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

constexpr int SBN = kSkinnyBN;       // 256 columns per slab
constexpr int SBK = kSkinnyBK;       // 32 rows of B per stage
constexpr int WARPS = kSkinnyWarps;  // 4 or 8
constexpr int SNT = kSkinnyThreads;
constexpr int CPL = 8;               // columns per lane: a warp covers the row
constexpr int OWN = SBN / SNT;       // adjacent columns a thread owns after the reduction
static_assert(32 * CPL == SBN && (OWN == 1 || OWN == 2), "warp layout");

// Warp groups: with 8 warps and 16 rows of A, two groups of four warps take
// alternate positions (8 rows of each block per warp); with 8 warps and 32
// rows, two groups of four share every position and split the rows of A
// (row_split); otherwise all warps share every position.
template <int MT>
struct WarpPlan {
    static constexpr bool row_split = (WARPS == 8 && MT == 32);
    static constexpr int groups = (WARPS == 8 && (MT == 16 || MT == 32)) ? 2 : 1;
    static constexpr int gwarps = WARPS / groups;  // warps per group
    static constexpr int rpw = SBK / gwarps;       // rows of a block per warp
    static constexpr int mr = row_split ? MT / groups : MT;  // rows of A a warp sums
    // warps that read a stage before it is refilled
    static constexpr int readers = row_split ? WARPS : gwarps;
    static_assert(rpw * gwarps == SBK, "rows per warp");
    static_assert(MT != 32 || WARPS == 8, "32-row tiles need the 8-warp build");
};

template <int MT>
struct SkinnyLayout {
    static constexpr int SSTAGES = skinny_stages(MT);
    static constexpr int RPW = WarpPlan<MT>::rpw;
    static constexpr int a_floats = MT * SBK;  // M x 32, 128-byte rows, swizzled
    static constexpr int b_floats = SBK * SBN;
    static constexpr int stage_floats = a_floats + b_floats;
    static constexpr size_t stage_bytes = size_t(stage_floats) * 4;
    static_assert(stage_bytes % 1024 == 0, "stages must keep 1024-byte alignment");
    static constexpr int at_floats = RPW * WarpPlan<MT>::mr;  // per warp: RPW k x mr m
    static constexpr int RED_ROWS = 2;          // rows of M per reduction round
    static constexpr int red_floats = WARPS * RED_ROWS * SBN;

    static constexpr size_t at_off = SSTAGES * stage_bytes;
    static constexpr size_t red_off = at_off + size_t(WARPS) * at_floats * 4;
    static constexpr size_t bar_off = red_off + size_t(red_floats) * 4;  // SSTAGES + 1 barriers
    static constexpr size_t cnt_off = bar_off + (SSTAGES + 1) * 8;
    static constexpr size_t flag_off = cnt_off + SSTAGES * 4 * 2;
    static constexpr size_t total = flag_off + 16;
    static constexpr uint32_t tx_bytes = stage_floats * 4;
    // Fix-up through the idle ring: one piece is MT rows of a slot.
    static constexpr uint32_t piece_bytes = uint32_t(MT) * SBN * 4;
    static constexpr int ring_pieces = int(SSTAGES * stage_bytes / piece_bytes);

    static_assert(total <= 232448, "exceeds the 227 KB of shared memory a CTA may use");
    // The CTAs of one SM must fit its 228 KB together with 1 KB reserved each.
    static_assert(kSkinnyCtasPerSm * (total + 1024) <= 233472, "CTAs per SM do not fit");
};

template <int MT>
__device__ __forceinline__ int skinny_slot(const SkinnyParams &p, int cta, int slab) {
    const int start = slab * p.kt_total;
    const int k0 = max(p.starts[cta], start) - start;
    return 2 * cta + (k0 == 0 ? 1 : 0);
}

// The CTA whose range holds position u (ranges are contiguous and ascending).
__device__ __forceinline__ int skinny_owner(const SkinnyParams &p, int u) {
    int lo = 0, hi = gridDim.x - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.starts[mid] <= u)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

// A slot holds MT rows of a slab.
template <int MT>
__device__ __forceinline__ const float *skinny_piece(const SkinnyParams &p, int cta, int slab) {
    return p.partials + (size_t)skinny_slot<MT>(p, cta, slab) * (MT * SBN);
}


__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, uint64_t *bar,
                                                 int c0, int c1, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(c0), "r"(c1), "l"(pol)
        : "memory");
}
// Element (m, k) of the TMA-loaded A block: rows of 32 floats whose 16-byte
// chunks are XOR-swizzled with (row mod 8).
__device__ __forceinline__ float a_elem(const float *raw, int m, int k) {
    return raw[m * SBK + ((((k >> 2) ^ (m & 7)) << 2) | (k & 3))];
}

// N adjacent floats: shared-memory load, L2 load and L2 store.
template <int N>
struct Vec;
template <>
struct Vec<1> {
    __device__ __forceinline__ static void load(const float *p, float *v) { v[0] = *p; }
    __device__ __forceinline__ static void load_cg(const float *p, float *v) { v[0] = __ldcg(p); }
    __device__ __forceinline__ static void store_cg(float *p, const float *v) { __stcg(p, v[0]); }
};
template <>
struct Vec<2> {
    __device__ __forceinline__ static void load(const float *p, float *v) {
        const float2 x = *reinterpret_cast<const float2 *>(p);
        v[0] = x.x;
        v[1] = x.y;
    }
    __device__ __forceinline__ static void load_cg(const float *p, float *v) {
        const float2 x = __ldcg(reinterpret_cast<const float2 *>(p));
        v[0] = x.x;
        v[1] = x.y;
    }
    __device__ __forceinline__ static void store_cg(float *p, const float *v) {
        __stcg(reinterpret_cast<float2 *>(p), make_float2(v[0], v[1]));
    }
};

// Adds the warps' sums in warp order through `buf`, RR of each warp's rows
// at a time.  Thread t ends with all MT rows of columns [OWN t, OWN t + OWN)
// in fin; row m sums the warps that hold it (all warps, or with split rows
// the warps of group m / MR).  Starts and ends with `buf` free to reuse.
template <int MT, int RR>
__device__ __forceinline__ void reduce_warps(const float2 (&acc)[WarpPlan<MT>::mr / 2][CPL],
                                             float *buf, float (&fin)[MT][OWN], int warp, int lane,
                                             int col0) {
    constexpr int MR = WarpPlan<MT>::mr;
    constexpr int SUMMED = WarpPlan<MT>::row_split ? WarpPlan<MT>::gwarps : WARPS;
#pragma unroll
    for (int r = 0; r < MR / RR; ++r) {
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
                *reinterpret_cast<float4 *>(buf + (warp * RR + i) * SBN + c * 128 + lane * 4) = v;
            }
        }
        __syncthreads();
#pragma unroll
        for (int g = 0; g < WARPS / SUMMED; ++g) {
#pragma unroll
            for (int i = 0; i < RR; ++i) {
                float sum[OWN], x[OWN];
                Vec<OWN>::load(buf + ((g * SUMMED) * RR + i) * SBN + col0, sum);
#pragma unroll
                for (int w = 1; w < SUMMED; ++w) {
                    Vec<OWN>::load(buf + ((g * SUMMED + w) * RR + i) * SBN + col0, x);
#pragma unroll
                    for (int o = 0; o < OWN; ++o) sum[o] += x[o];
                }
#pragma unroll
                for (int o = 0; o < OWN; ++o) fin[g * MR + RR * r + i][o] = sum[o];
            }
        }
        __syncthreads();
    }
}

template <int MT>
__global__ void __launch_bounds__(SNT, kSkinnyCtasPerSm)
    sgemm_skinny_kernel(const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapB,
                        const __grid_constant__ SkinnyParams p) {
    using L = SkinnyLayout<MT>;
    constexpr int SSTAGES = L::SSTAGES;
    extern __shared__ __align__(1024) uint8_t smem[];
    float *stages = reinterpret_cast<float *>(smem);
    float *red = reinterpret_cast<float *>(smem + L::red_off);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    uint64_t *fix_bar = full + SSTAGES;
    int *release = reinterpret_cast<int *>(smem + L::cnt_off);
    volatile int *issued = reinterpret_cast<volatile int *>(smem + L::cnt_off + SSTAGES * 4);
    volatile int *flags = reinterpret_cast<volatile int *>(smem + L::flag_off);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cta = blockIdx.x;
    float *at_w = reinterpret_cast<float *>(smem + L::at_off) + warp * L::at_floats;
    constexpr int GROUPS = WarpPlan<MT>::groups, GW = WarpPlan<MT>::gwarps;
    constexpr int RPW = WarpPlan<MT>::rpw;
    constexpr bool ROW_SPLIT = WarpPlan<MT>::row_split;
    constexpr int MR = WarpPlan<MT>::mr;  // rows of A this warp sums
    const int grp = warp / GW, wl = warp % GW;  // group, and warp within it
    const int row0 = ROW_SPLIT ? grp * MR : 0;  // first of those rows

    const int u0 = p.starts[cta];
    const int q_total = p.starts[cta + 1] - u0;
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
        tma_load_2d_hint(sa + L::a_floats, &mapB, &full[s], slab * SBN, k * SBK, policy_evict_first());
    };

    if (tid == 0) {
        for (int s = 0; s < SSTAGES; ++s) {
            mbar_init(&full[s], 1);
            release[s] = 0;
            issued[s] = -1;
        }
        mbar_init(fix_bar, 1);
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
    bool fix_pending = false;  // a fix-up copy may still be in flight (after a timeout)
    uint32_t fix_phase = 0;
    int timed_out = 0;  // this thread saw a wait run out (made uniform at unit end)
    const int col0 = tid * OWN;  // first column this thread owns after the reduction
    while (q < q_total && !aborted) {
        const int u = u0 + q;
        const int slab = u / p.kt_total;
        const int k0 = u - slab * p.kt_total;
        const int k1 = min(p.kt_total, k0 + (q_total - q));

        float2 acc[MR / 2][CPL];  // acc[ip][j] = (C[row0+2ip][n_j], C[row0+2ip+1][n_j])
#pragma unroll
        for (int i = 0; i < MR / 2; ++i)
#pragma unroll
            for (int j = 0; j < CPL; ++j) acc[i][j] = make_float2(0.f, 0.f);

        for (int kt = k0; kt < k1; ++kt, ++q) {
            if (GROUPS > 1 && !ROW_SPLIT && q % GROUPS != grp) continue;  // the other group's
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
            // This warp's A columns k = wl + GW * kk of its rows, k-major:
            // at_w[kk * MR + m] = A[row0 + m][k].
#pragma unroll
            for (int e = lane; e < RPW * MR; e += 32) {
                const int m = e % MR, kk = e / MR;
                at_w[kk * MR + m] = a_elem(raw, row0 + m, wl + GW * kk);
            }
            __syncwarp();

            const float *bcol = bs + lane * 4;
            float4 bf[2][CPL / 4];
#pragma unroll
            for (int c = 0; c < CPL / 4; ++c) bf[0][c] = ld_shared_f4(bcol + wl * SBN + c * 128);
#pragma unroll
            for (int kk = 0; kk < RPW; ++kk) {
                const int cur = kk & 1, nxt = cur ^ 1;
                if (kk + 1 < RPW) {
                    const float *brow = bcol + (wl + GW * (kk + 1)) * SBN;
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
                for (int r = 0; r < MR / 4; ++r) {
                    const float4 a = ld_shared_f4(at_w + kk * MR + r * 4);
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
            // Release the stage; the last of its readers refills it.
            if (lane == 0) {
                __threadfence_block();
                const int old = atomicAdd(&release[s], 1);
                if (old == WarpPlan<MT>::readers - 1) {
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

        // ---- add the warps' sums in warp order ----
        // The final unit has no copies outstanding, so the idle ring takes
        // all rows of every warp at once (one barrier instead of two per
        // pair of rows); other units use `red`, two rows per round.  (Same
        // order of sums either way.)
        static_assert(size_t(WARPS) * MR * SBN * 4 <= SSTAGES * L::stage_bytes,
                      "the warps' sums fit the ring");
        float fin[MT][OWN];
        if (q == q_total)
            reduce_warps<MT, MR>(acc, stages, fin, warp, lane, col0);
        else
            reduce_warps<MT, L::RED_ROWS>(acc, red, fin, warp, lane, col0);

        const bool partial = !(k0 == 0 && k1 == p.kt_total);
        const int c_first = partial ? skinny_owner(p, slab * p.kt_total) : cta;
        const int c_last = partial ? skinny_owner(p, slab * p.kt_total + p.kt_total - 1) : cta;
        bool write_c = true;
        if (partial) {
            float *slot = p.partials + (size_t)skinny_slot<MT>(p, cta, slab) * (MT * SBN);
#pragma unroll
            for (int m = 0; m < MT; ++m) Vec<OWN>::store_cg(slot + m * SBN + col0, fin[m]);
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                const int old = atomicAdd(&p.counters[slab], 1);
                flags[1] = (old == c_last - c_first) ? 1 : 0;
            }
            __syncthreads();
            write_c = flags[1] != 0;
            if (write_c) {
                __threadfence();
                float own[MT][OWN];
#pragma unroll
                for (int m = 0; m < MT; ++m)
#pragma unroll
                    for (int o = 0; o < OWN; ++o) own[m][o] = fin[m][o];
                if (q == q_total) {
                    // Last unit: no copies are outstanding, so the ring is
                    // idle.  The other pieces come in with bulk copies, up to
                    // ring_pieces at a time, and are added in CTA order.
                    bool ok = true;
                    int cc = c_first;
                    while (cc <= c_last) {
                        int cnt = 0, cc_end = cc;
                        while (cc_end <= c_last && (cc_end == cta || cnt < L::ring_pieces)) {
                            if (cc_end != cta) ++cnt;
                            ++cc_end;
                        }
                        if (cnt > 0) {
                            __syncthreads();  // the ring's previous contents are read
                            if (tid == 0) {
                                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                                fence_proxy_async_global();
                                mbar_arrive_expect_tx(fix_bar, cnt * L::piece_bytes);
                                int j = 0;
                                for (int c = cc; c < cc_end; ++c) {
                                    if (c == cta) continue;
                                    bulk_load(reinterpret_cast<char *>(stages) + j * L::piece_bytes,
                                              skinny_piece<MT>(p, c, slab), L::piece_bytes, fix_bar);
                                    ++j;
                                }
                            }
                            const bool got = mbar_wait_bounded(fix_bar, fix_phase, p.timeout_ns);
                            fix_phase ^= 1u;
                            if (__syncthreads_or(!got)) {
                                // Stop issuing; the copies of this round are
                                // waited for (bounded) before the CTA exits.
                                ok = false;
                                fix_pending = true;
                                if (tid == 0) atomicOr(p.err, kErrWaitTimeout);
                                break;
                            }
                        }
                        int j = 0;
                        for (int c = cc; c < cc_end; ++c) {
#pragma unroll
                            for (int m = 0; m < MT; ++m) {
                                float x[OWN];
                                if (c == cta) {
#pragma unroll
                                    for (int o = 0; o < OWN; ++o) x[o] = own[m][o];
                                } else {
                                    Vec<OWN>::load(stages + (size_t)j * (MT * SBN) + m * SBN + col0, x);
                                }
#pragma unroll
                                for (int o = 0; o < OWN; ++o)
                                    fin[m][o] = (c == c_first) ? x[o] : fin[m][o] + x[o];
                            }
                            if (c != cta) ++j;
                        }
                        cc = cc_end;
                    }
                    if (!ok) {  // uniform: set after a CTA-wide vote
                        write_c = false;
                        aborted = true;
                    }
                } else {
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        for (int c = c_first; c <= c_last; ++c) {
                            float x[OWN];
                            if (c == cta) {
#pragma unroll
                                for (int o = 0; o < OWN; ++o) x[o] = own[m][o];
                            } else {
                                Vec<OWN>::load_cg(skinny_piece<MT>(p, c, slab) + m * SBN + col0, x);
                            }
#pragma unroll
                            for (int o = 0; o < OWN; ++o)
                                fin[m][o] = (c == c_first) ? x[o] : fin[m][o] + x[o];
                        }
                    }
                }
                if (tid == 0) p.counters[slab] = 0;
            }
            __syncthreads();  // flags[1] is rewritten by the next unit
        }
        if (write_c) {
#pragma unroll
            for (int o = 0; o < OWN; ++o) {
                const int n = slab * SBN + col0 + o;
                if (n < p.N) {
#pragma unroll
                    for (int m = 0; m < MT; ++m) {
                        if (m < p.M) {
                            float *c = p.C + (long long)m * p.ldc + n;
                            float out = p.alpha * fin[m][o];
                            if (p.beta != 0.0f) out = __fmaf_rn(p.beta, *c, out);
                            *c = apply_epilogue(out, p.epi, n);
                        }
                    }
                }
            }
        }
    }

    if (aborted && tid == 0) {
        // Wait (bounded) for the last copy issued into every stage, and for a
        // fix-up copy that timed out, so none lands in shared memory after
        // this CTA has exited.
        for (int s = 0; s < SSTAGES; ++s) {
            const int last = issued[s];
            if (last < 0) continue;
            if (!mbar_wait_bounded(&full[s], (last / SSTAGES) & 1, 1000000000ull)) {
                atomicOr(p.err, kErrDrainTimeout);
                break;
            }
        }
        if (fix_pending && !mbar_wait_bounded(fix_bar, fix_phase ^ 1u, 1000000000ull))
            atomicOr(p.err, kErrDrainTimeout);
    }
}

template <int MT>
cudaError_t configure_impl() {
    cudaError_t e = cudaFuncSetAttribute(sgemm_skinny_kernel<MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SkinnyLayout<MT>::total);
    if (e != cudaSuccess) return e;
    // Two CTAs per SM need the whole unified L1 / shared array as shared memory.
    return cudaFuncSetAttribute(sgemm_skinny_kernel<MT>,
                                cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared);
}

}  // namespace

// 32-row tiles exist only in the 8-warp build (two row groups of four warps).
constexpr bool kHas32 = WARPS == 8;

size_t skinny_smem_bytes(int m_tile, int /*share*/) {
    if (m_tile == 8) return SkinnyLayout<8>::total;
    if (m_tile == 16) return SkinnyLayout<16>::total;
    if constexpr (kHas32)
        if (m_tile == 32) return SkinnyLayout<32>::total;
    return 0;
}

cudaError_t skinny_configure(int m_tile) {
    if (m_tile == 8) return configure_impl<8>();
    if (m_tile == 16) return configure_impl<16>();
    if constexpr (kHas32)
        if (m_tile == 32) return configure_impl<32>();
    return cudaErrorInvalidValue;
}

cudaError_t launch_skinny(int m_tile, const CUtensorMap &mapA, const CUtensorMap &mapB,
                          const SkinnyParams &p, int grid, cudaStream_t stream) {
    if (m_tile == 8) {
        sgemm_skinny_kernel<8><<<grid, SNT, SkinnyLayout<8>::total, stream>>>(mapA, mapB, p);
    } else if (m_tile == 16) {
        sgemm_skinny_kernel<16><<<grid, SNT, SkinnyLayout<16>::total, stream>>>(mapA, mapB, p);
    } else if (kHas32 && m_tile == 32) {
        if constexpr (kHas32)
            sgemm_skinny_kernel<32><<<grid, SNT, SkinnyLayout<32>::total, stream>>>(mapA, mapB, p);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace sgemm
