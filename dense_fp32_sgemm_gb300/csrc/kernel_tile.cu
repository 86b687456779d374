// Tiled SIMT FP32 GEMM for sm_103a: C = alpha * A * B + beta * C, row-major.
//
// One CTA of 256 threads owns a 128 x 256 tile of C and walks K in slices of
// 32.  Each thread keeps a 16 x 8 micro-tile of running sums in registers and
// updates it with an outer product per k: 16 values of A and 8 of B feed 128
// multiply-adds ("Optimizing Matrix Multiply on CUDA, Part 2", section
// "Increasing the Outputs per Thread": the 16 x 8 patch and 128 x 256 tile).
//
// Global -> shared staging uses TMA tiled copies into a ring of STAGES
// buffers completed on mbarriers.  A's slice arrives as stored (k fastest);
// the threads then rewrite it k-major ("transposed") into a second buffer so
// that a thread's A values for one k are adjacent and come in with 128-bit
// shared loads ("Optimizing CUDA matmul, steps 4 to 6", section "Two ladders,
// one kernel": the transposed tile and the fill's derived 2-way store
// conflict; "Part 2", section "Reducing the Slice Depth": 4-8 store passes).
// Here the fill reads four 16-byte rows and writes four 16-byte columns per
// thread, and the 16-byte chunk index of the transposed tile is XOR-ed with
// (k / 4) mod 8: the eight stores of a quarter-warp land in eight different
// bank groups, and the inner-loop reads are free of bank conflicts (ncu at
// 2048^3: 977 load conflicts against 34.8 M load wavefronts).  ncu still
// counts about 0.45 store conflicts per shared store instruction (125 K
// against 1.19 M store wavefronts per launch); the stores are 3 % of the
// shared-memory wavefronts, so they cost little either way.
//
// B is read in two groups of four columns 32 apart per thread ("Part 2",
// section "Changing the Shared-Memory Access Pattern"), so the eight threads
// of a quarter-warp cover 32 consecutive banks.
//
// Work distribution ("Part 2", sections "Choosing Tiles" and "Distributing
// the Partially Filled Wave"): a persistent grid computes the first dp_tiles
// tiles whole, round-robin, then shares the k-iterations of the remaining
// tiles evenly (stream-K).  A CTA whose range covers only part of a tile
// writes its partial sums to a fixed slot and takes a ticket; the CTA that
// arrives last adds the pieces in CTA order (so the result does not depend on
// arrival order) and applies the epilogue.  No CTA ever waits for another.
//
// The multiply-add is IEEE FP32 fma with round-to-nearest, either one product
// per instruction or two per instruction through the packed form (__ffma2_rn,
// identical per-component arithmetic); FmaMode picks how the pairs are formed.

#include "device_common.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

constexpr int BM = kTileBM;
constexpr int BN = kTileBN;
constexpr int BK = kTileBK;
constexpr int TN = 8;
constexpr int A_STAGE_FLOATS = BM * BK;
constexpr int B_STAGE_FLOATS = BK * BN;
constexpr int STAGE_FLOATS = A_STAGE_FLOATS + B_STAGE_FLOATS;
constexpr uint32_t STAGE_TX_BYTES = STAGE_FLOATS * 4;
constexpr int TILE_FLOATS = BM * BN;
constexpr int FILL_THREADS = BM * BK / 16;  // one 4 x 4 block of the A slice each
static_assert(BK == 32 && BM == 128, "the transposing fill assumes 32 x 128 A slices");

// Thread organisation for a micro-tile of TM rows x 8 columns.  A warp is 4
// (rows) x 8 (columns) threads; a thread's rows come in groups of four, 16
// apart, its columns in two groups of four, 32 apart.  TM = 16: 8 warps of
// 64 x 64 (two warps per scheduler, up to 255 registers); TM = 8: 16 warps of
// 32 x 64 (four per scheduler, at most 128 registers).
template <int TM_>
struct Cfg {
    static constexpr int TM = TM_;
    static constexpr int NT = TILE_FLOATS / (TM * TN);
    static constexpr int WARP_M = 4 * TM;
    static constexpr int WARP_N = 8 * TN;
    static constexpr int WARPS_N = BN / WARP_N;
    static constexpr int RG = TM / 4;  // row groups
    static_assert(NT % 32 == 0 && NT >= FILL_THREADS, "bad thread count");
};

template <int FM>
struct AtRow {
    static constexpr int value = (FM == kFmaPairDupA) ? 2 * BM : BM;
};

template <int FM, int STAGES>
struct SmemLayout {
    static constexpr size_t stage_bytes = size_t(STAGE_FLOATS) * 4;
    static constexpr size_t at_bytes = size_t(BK) * AtRow<FM>::value * 4;
    static constexpr size_t at_off = STAGES * stage_bytes;
    static constexpr size_t bar_off = at_off + 2 * at_bytes;
    static constexpr size_t redbar_off = bar_off + STAGES * 8;  // fixup bulk copies
    static constexpr size_t prebar_off = redbar_off + 8;        // partner prefetch, 2 parts
    static constexpr size_t flag_off = prebar_off + 16;
    static constexpr size_t prod_off = flag_off + 16;
    static constexpr size_t total = prod_off + 32;
    // The partner prefetch fills the two idle stages and then the last one.
    static_assert(STAGES != 3 || 3 * stage_bytes >= size_t(TILE_FLOATS) * 4, "prefetch layout");
    static_assert(STAGES * stage_bytes >= size_t(TILE_FLOATS) * 4,
                  "the final-unit fixup stages a whole partial tile in the ring");
    static_assert(total <= 232448, "exceeds the 227 KB of shared memory a CTA may use");
};

// ----- accumulators --------------------------------------------------------
template <int TM>
struct AccScalar {
    float v[TM][TN];
    __device__ __forceinline__ float &at(int i, int j) { return v[i][j]; }
};

template <int TM>
struct AccPairN {  // v[i][jp] = (C[i][2jp], C[i][2jp+1])
    float2 v[TM][TN / 2];
    __device__ __forceinline__ float &at(int i, int j) {
        return (j & 1) ? v[i][j >> 1].y : v[i][j >> 1].x;
    }
};

template <int TM>
struct AccPairM {  // v[ip][j] = (C[2ip][j], C[2ip+1][j])
    float2 v[TM / 2][TN];
    __device__ __forceinline__ float &at(int i, int j) {
        return (i & 1) ? v[i >> 1][j].y : v[i >> 1][j].x;
    }
};

template <int FM, int TM>
struct AccSel {
    using type = AccPairN<TM>;
};
template <int TM>
struct AccSel<kFmaScalar, TM> {
    using type = AccScalar<TM>;
};
template <int TM>
struct AccSel<kFmaPairMovB, TM> {
    using type = AccPairM<TM>;
};
template <int FM, int TM>
using Acc = typename AccSel<FM, TM>::type;

template <int FM, int TM>
__device__ __forceinline__ void acc_zero(Acc<FM, TM> &acc) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc.at(i, j) = 0.0f;
}

// ----- fragments -------------------------------------------------------------
// A fragment for one k: thread rows r*16 + ty*4 + (0..3), r < TM/4.
// B fragment for one k: thread columns c*32 + tx*4 + (0..3), c = 0..1.
template <int FM, int TM>
struct Frag {
    float4 a[FM == kFmaPairDupA ? TM / 2 : TM / 4];
    float4 b[2];
};

__device__ __forceinline__ float comp(const float4 &v, int i) {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Per-thread shared-memory offsets (in floats) for the rows of one block of
// four k values (the swizzle is constant over such a block).
struct FragPtrs {
    int a0, a1;  // A: two XOR-ed chunk bases (see load_frag)
    int b;       // B: first column group
};

template <int FM, int TM>
__device__ __forceinline__ FragPtrs frag_ptrs(int kblk, int wm, int wn, int ty, int tx) {
    constexpr int ROW = AtRow<FM>::value;
    const int swz = (kblk >> 2) & 7;
    FragPtrs f;
    if (FM == kFmaPairDupA) {
        // chunk(r, p) = wm*2*TM + r*8 + ty*2 + p; the XOR touches only the
        // low three bits, (2*ty + p).
        const int x0 = (2 * ty) ^ swz;
        f.a0 = kblk * ROW + (wm * 2 * TM + x0) * 4;
        f.a1 = kblk * ROW + (wm * 2 * TM + (x0 ^ 1)) * 4;
    } else {
        // chunk(r) = wm*TM + r*4 + ty; low three bits are (r&1)*4 + ty.
        const int x0 = ty ^ swz;
        f.a0 = kblk * ROW + (wm * TM + x0) * 4;
        f.a1 = kblk * ROW + (wm * TM + (x0 ^ 4)) * 4;
    }
    f.b = kblk * BN + wn * 64 + tx * 4;
    return f;
}

template <int FM, int TM>
__device__ __forceinline__ void load_frag(const float *at, const float *bs, const FragPtrs &fp,
                                          int j, Frag<FM, TM> &f) {
    constexpr int ROW = AtRow<FM>::value;
    const float *pa0 = at + fp.a0 + j * ROW;
    const float *pa1 = at + fp.a1 + j * ROW;
    if (FM == kFmaPairDupA) {
#pragma unroll
        for (int r = 0; r < TM / 4; ++r) {
            f.a[2 * r + 0] = ld_shared_f4(pa0 + r * 32);
            f.a[2 * r + 1] = ld_shared_f4(pa1 + r * 32);
        }
    } else {
#pragma unroll
        for (int r = 0; r < TM / 4; ++r)
            f.a[r] = ld_shared_f4(((r & 1) ? pa1 : pa0) + (r >> 1) * 32);
    }
    const float *pb = bs + fp.b + j * BN;
    f.b[0] = ld_shared_f4(pb);
    f.b[1] = ld_shared_f4(pb + 32);
}

template <int FM, int TM>
__device__ __forceinline__ void fma_frag(const Frag<FM, TM> &f, Acc<FM, TM> &acc) {
    if (FM == kFmaScalar) {
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const float a = comp(f.a[i >> 2], i & 3);
#pragma unroll
            for (int j = 0; j < TN; ++j)
                acc.at(i, j) = __fmaf_rn(a, comp(f.b[j >> 2], j & 3), acc.at(i, j));
        }
    } else if (FM == kFmaPairMovA || FM == kFmaPairDupA) {
        auto &v = reinterpret_cast<AccPairN<TM> &>(acc).v;
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            float2 a2;
            if (FM == kFmaPairDupA) {
                const float4 &d = f.a[i >> 1];
                a2 = (i & 1) ? make_float2(d.z, d.w) : make_float2(d.x, d.y);
            } else {
                const float a = comp(f.a[i >> 2], i & 3);
                a2 = make_float2(a, a);
            }
#pragma unroll
            for (int jp = 0; jp < TN / 2; ++jp) {
                const float4 &b = f.b[jp >> 1];
                const float2 b2 = (jp & 1) ? make_float2(b.z, b.w) : make_float2(b.x, b.y);
                v[i][jp] = __ffma2_rn(a2, b2, v[i][jp]);
            }
        }
    } else {  // kFmaPairMovB
        auto &v = reinterpret_cast<AccPairM<TM> &>(acc).v;
#pragma unroll
        for (int ip = 0; ip < TM / 2; ++ip) {
            const float4 &a = f.a[ip >> 1];
            const float2 a2 = (ip & 1) ? make_float2(a.z, a.w) : make_float2(a.x, a.y);
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const float b = comp(f.b[j >> 2], j & 3);
                v[ip][j] = __ffma2_rn(a2, make_float2(b, b), v[ip][j]);
            }
        }
    }
}

// One K slice (32 k) of outer products from the transposed A slice `at` and
// the B slice `bs`, fully unrolled: fragments are double-buffered in
// registers (the loads for k+1 are issued before the multiply-adds of k) and
// every shared-memory offset but the per-thread base is a constant, which
// gives the instruction scheduler the whole slice to interleave.  (Measured
// on GB300: 4-k blocks in a loop ran about 8% slower.)
template <int FM, int TM>
__device__ __forceinline__ void compute_slice(const float *at, const float *bs, Acc<FM, TM> &acc,
                                              int wm, int wn, int ty, int tx) {
    Frag<FM, TM> f[2];
    load_frag<FM, TM>(at, bs, frag_ptrs<FM, TM>(0, wm, wn, ty, tx), 0, f[0]);
#pragma unroll
    for (int k = 0; k < BK; ++k) {
        if (k + 1 < BK) {
            // Row k+1 sits in the 4-row block starting at (k+1) & ~3, whose
            // swizzle the pointers carry.
            const FragPtrs fp = frag_ptrs<FM, TM>((k + 1) & ~3, wm, wn, ty, tx);
            load_frag<FM, TM>(at, bs, fp, (k + 1) & 3, f[(k + 1) & 1]);
        }
        fma_frag<FM, TM>(f[k & 1], acc);
    }
}

// Rewrite the TMA-loaded A slice (BM rows x BK k, k fastest) k-major into
// `at`, XOR-swizzling the 16-byte chunk index with (k / 4) mod 8.  Thread t
// moves the 4 x 4 block rows 4*(t/8).., k 4*(t%8)..: the eight threads of a
// quarter-warp read eight different chunks of one 128-byte row and write
// eight different bank groups.
template <int FM>
__device__ __forceinline__ void transpose_slice(const float *raw, float *at, int tid) {
    constexpr int ROW = AtRow<FM>::value;
    if (tid >= FILL_THREADS) return;
    const int kc = tid & 7;
    const int mb = tid >> 3;
    float4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = ld_shared_f4(raw + (4 * mb + i) * BK + 4 * kc);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        float *row = at + (4 * kc + kk) * ROW;
        const float e0 = comp(v[0], kk), e1 = comp(v[1], kk);
        const float e2 = comp(v[2], kk), e3 = comp(v[3], kk);
        if (FM == kFmaPairDupA) {
            st_shared_f4(row + ((2 * mb) ^ kc) * 4, make_float4(e0, e0, e1, e1));
            st_shared_f4(row + ((2 * mb + 1) ^ kc) * 4, make_float4(e2, e2, e3, e3));
        } else {
            st_shared_f4(row + (mb ^ kc) * 4, make_float4(e0, e1, e2, e3));
        }
    }
}

__device__ __forceinline__ void tile_coords(const TileParams &p, int t, int &tm, int &tn) {
    // Grouped rasterisation: runs of group_m tile-rows are walked column by
    // column so CTAs that run together share A rows and B columns in L2.
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int rows = min(p.tiles_m - first_m, p.group_m);
    const int r = t - g * per_group;
    tm = first_m + r % rows;
    tn = r / rows;
}

// Iterates the units (tile, k-range) of one CTA: its round-robin share of
// the whole tiles, then its contiguous range of stream-K iterations.
struct UnitIter {
    int dp_next;
    int sk_u, sk_end;
    __device__ __forceinline__ void init(const TileParams &p, int cta) {
        dp_next = cta;
        const int sk_total = p.sk_tiles * p.kt_total;
        sk_u = min(cta * p.sk_share, sk_total);
        sk_end = min(sk_u + p.sk_share, sk_total);
    }
    __device__ __forceinline__ bool next(const TileParams &p, int G, int &tile, int &k0, int &k1) {
        if (dp_next < p.dp_tiles) {
            tile = dp_next;
            k0 = 0;
            k1 = p.kt_total;
            dp_next += G;
            return true;
        }
        if (sk_u < sk_end) {
            const int t = sk_u / p.kt_total;
            k0 = sk_u - t * p.kt_total;
            k1 = min(p.kt_total, k0 + (sk_end - sk_u));
            tile = p.dp_tiles + t;
            sk_u += k1 - k0;
            return true;
        }
        return false;
    }
};

struct ProducerState {
    UnitIter it;
    int pq, tm, tn, k, k1;  // next position to issue; its tile and k-range
};

// ---- the code after a unit's last slice ----
// It runs once per unit, and on GB300 the first run of straight-line code
// waits for its instructions: a fully unrolled 128 x 256 store measured about
// 20 us the first time through and 3 us when repeated.  The stream-K fix-up
// (whose unrolled form took 40 us at its first run) is therefore a few short
// rolled loops.

// One float4 of C: columns n .. n+3 of row m, from the raw sums a.
__device__ __forceinline__ void store_c4(const TileParams &p, int m, int n, float4 a) {
    if (m >= p.M) return;
    float *crow = p.C + (long long)m * p.ldc;
    float o[4] = {p.alpha * a.x, p.alpha * a.y, p.alpha * a.z, p.alpha * a.w};
    if (p.c_vec4 && n + 3 < p.N) {
        if (p.beta != 0.0f) {
            const float4 cv = *reinterpret_cast<const float4 *>(crow + n);
            o[0] = __fmaf_rn(p.beta, cv.x, o[0]);
            o[1] = __fmaf_rn(p.beta, cv.y, o[1]);
            o[2] = __fmaf_rn(p.beta, cv.z, o[2]);
            o[3] = __fmaf_rn(p.beta, cv.w, o[3]);
        }
        if (p.epi.bias || p.epi.act) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) o[jj] = apply_epilogue(o[jj], p.epi, n + jj);
        }
        *reinterpret_cast<float4 *>(crow + n) = make_float4(o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            if (n + jj < p.N) {
                float v = o[jj];
                if (p.beta != 0.0f) v = __fmaf_rn(p.beta, crow[n + jj], v);
                crow[n + jj] = apply_epilogue(v, p.epi, n + jj);
            }
        }
    }
}

// Tile coordinates of accumulator element (ti, j) of thread t (TM = 16:
// warps 2 x 4 of 64 x 64, lanes 4 x 8, rows in four groups of 4 at stride 16,
// columns in two groups of 4 at stride 32).
__device__ __forceinline__ int acc_row(int t, int ti) {
    const int warp = t >> 5, wm = warp / 4, ty = (t & 31) >> 3;
    return wm * 64 + (ti >> 2) * 16 + ty * 4 + (ti & 3);
}
__device__ __forceinline__ int acc_col(int t, int c) {
    const int warp = t >> 5, wn = warp % 4, tx = t & 7;
    return wn * 64 + c * 32 + tx * 4;
}

// Float4 number e4 of a thread's accumulators: row e4 / 2, columns
// (e4 % 2) * 4 .. + 3.  A switch, so the accumulators stay in registers
// while the caller's loop over e4 stays rolled.
template <class AccT>
__device__ __forceinline__ float4 acc_f4(AccT &acc, int e4) {
    switch (e4) {
#define SGEMM_E4(E)                                                                        \
    case E:                                                                                \
        return make_float4(acc.at((E) >> 1, ((E)&1) * 4 + 0), acc.at((E) >> 1, ((E)&1) * 4 + 1), \
                           acc.at((E) >> 1, ((E)&1) * 4 + 2), acc.at((E) >> 1, ((E)&1) * 4 + 3));
        SGEMM_E4(0) SGEMM_E4(1) SGEMM_E4(2) SGEMM_E4(3) SGEMM_E4(4) SGEMM_E4(5) SGEMM_E4(6)
        SGEMM_E4(7) SGEMM_E4(8) SGEMM_E4(9) SGEMM_E4(10) SGEMM_E4(11) SGEMM_E4(12)
        SGEMM_E4(13) SGEMM_E4(14) SGEMM_E4(15) SGEMM_E4(16) SGEMM_E4(17) SGEMM_E4(18)
        SGEMM_E4(19) SGEMM_E4(20) SGEMM_E4(21) SGEMM_E4(22) SGEMM_E4(23) SGEMM_E4(24)
        SGEMM_E4(25) SGEMM_E4(26) SGEMM_E4(27) SGEMM_E4(28) SGEMM_E4(29) SGEMM_E4(30)
        SGEMM_E4(31)
#undef SGEMM_E4
    }
    return make_float4(0.f, 0.f, 0.f, 0.f);
}

// C = alpha * acc (+ beta C, epilogue) for a whole tile, unrolled: a rolled
// version (one float4 per iteration through acc_f4) is compact but changes
// the register allocation of the whole kernel, and measured 2.6 % slower on
// the large products whose time is the main loop.
template <int FM, int TM>
__device__ __forceinline__ void store_tile(Acc<FM, TM> &acc, const TileParams &p, int tm, int tn,
                                           int wm, int wn, int ty, int tx) {
    const int m_base = tm * BM + wm * Cfg<TM>::WARP_M + ty * 4;
    const int n_base = tn * BN + wn * 64 + tx * 4;
    const float alpha = p.alpha, beta = p.beta;
#pragma unroll
    for (int r = 0; r < TM / 4; ++r) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = m_base + r * 16 + i;
            if (m >= p.M) continue;
            float *crow = p.C + (long long)m * p.ldc;
            const int ti = r * 4 + i;
            float4 cvr[2];
            if (beta != 0.0f && p.c_vec4) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int n = n_base + c * 32;
                    cvr[c] = n + 3 < p.N ? *reinterpret_cast<const float4 *>(crow + n)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int n = n_base + c * 32;
                if (p.c_vec4 && n + 3 < p.N) {
                    float4 o;
                    o.x = alpha * acc.at(ti, c * 4 + 0);
                    o.y = alpha * acc.at(ti, c * 4 + 1);
                    o.z = alpha * acc.at(ti, c * 4 + 2);
                    o.w = alpha * acc.at(ti, c * 4 + 3);
                    if (beta != 0.0f) {
                        const float4 cv = cvr[c];
                        o.x = __fmaf_rn(beta, cv.x, o.x);
                        o.y = __fmaf_rn(beta, cv.y, o.y);
                        o.z = __fmaf_rn(beta, cv.z, o.z);
                        o.w = __fmaf_rn(beta, cv.w, o.w);
                    }
                    if (p.epi.bias || p.epi.act) {
                        o.x = apply_epilogue(o.x, p.epi, n + 0);
                        o.y = apply_epilogue(o.y, p.epi, n + 1);
                        o.z = apply_epilogue(o.z, p.epi, n + 2);
                        o.w = apply_epilogue(o.w, p.epi, n + 3);
                    }
                    *reinterpret_cast<float4 *>(crow + n) = o;
                } else {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        if (n + jj < p.N) {
                            float o = alpha * acc.at(ti, c * 4 + jj);
                            if (beta != 0.0f) o = __fmaf_rn(beta, crow[n + jj], o);
                            crow[n + jj] = apply_epilogue(o, p.epi, n + jj);
                        }
                    }
                }
            }
        }
    }
}

// Partial tiles use a thread-linear layout: float4 number e4 of thread tid
// sits at slot[(e4 * NT + tid) * 4], element order (row ti, columns c*4..).
template <int FM, int TM>
__device__ __forceinline__ void write_partial(float *slot, Acc<FM, TM> &acc, int tid) {
    constexpr int NT = Cfg<TM>::NT;
#pragma unroll
    for (int e4 = 0; e4 < TILE_FLOATS / NT / 4; ++e4) {
        const int ti = e4 >> 1, c = e4 & 1;
        const float4 v = make_float4(acc.at(ti, c * 4 + 0), acc.at(ti, c * 4 + 1),
                                     acc.at(ti, c * 4 + 2), acc.at(ti, c * 4 + 3));
        __stcg(reinterpret_cast<float4 *>(slot) + e4 * NT + tid, v);
    }
}

__device__ __forceinline__ int partial_slot(const TileParams &p, int cta, int t_sk) {
    const int tile_start = t_sk * p.kt_total;
    const int k0 = max(cta * p.sk_share, tile_start) - tile_start;
    return 2 * cta + (k0 == 0 ? 1 : 0);
}

// The stream-K fix-up: the pieces of tile t_sk (CTAs c_first .. c_last,
// every one of them, this CTA's included, already in its partial slot) are
// added in CTA order and C is written.  In a slot, float4 number e4 of thread
// t sits at [(e4 * NT + t) * 4], so thread t sums and stores exactly the
// elements it would have held in registers.

// From L2, for a unit whose ring still holds copies in flight.
template <int TM>
__device__ __forceinline__ void fixup_from_l2(const TileParams &p, int tm, int tn, int t_sk,
                                              int c_first, int c_last, int tid) {
    constexpr int NT = Cfg<TM>::NT;
#pragma unroll 1
    for (int e4 = 0; e4 < TILE_FLOATS / NT / 4; ++e4) {
        const int f = e4 * NT + tid;
        float4 s = __ldcg(reinterpret_cast<const float4 *>(
                              p.partials + (size_t)partial_slot(p, c_first, t_sk) * TILE_FLOATS) + f);
#pragma unroll 1
        for (int c = c_first + 1; c <= c_last; ++c) {
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(
                                        p.partials + (size_t)partial_slot(p, c, t_sk) * TILE_FLOATS) + f);
            s.x += x.x;
            s.y += x.y;
            s.z += x.z;
            s.w += x.w;
        }
        store_c4(p, tm * BM + acc_row(tid, e4 >> 1), tn * BN + acc_col(tid, e4 & 1), s);
    }
}

// Through the idle ring of a CTA's final unit: band by band (four float4 per
// thread, 16 KB per piece) the pieces come in with bulk copies.  Up to three
// bands are in flight at once, each on its own barrier (bars[0..2]: the
// fix-up barrier and the two partner-prefetch barriers, idle in a unit that
// takes this path), so the L2 round trips overlap the sums.  Takes up to
// ring capacity / 16 KB pieces.  Returns false (uniformly) if a copy did not
// arrive in time, after waiting (bounded) for every copy still in flight.
template <int TM, int STAGES>
__device__ __forceinline__ bool fixup_staged(const TileParams &p, int tm, int tn, int t_sk,
                                             int c_first, int c_last, int tid, float *ring,
                                             uint64_t *bars, uint32_t &phase) {
    constexpr int NT = Cfg<TM>::NT;
    constexpr int BAND = 4 * NT * 4;  // floats of one band of one piece
    constexpr int NBANDS = TILE_FLOATS / BAND;
    constexpr int RING_BANDS = STAGES * STAGE_FLOATS / BAND;
    const int n = c_last - c_first + 1;
    const int nslots = min(3, RING_BANDS / n);  // >= 1: the caller checks n <= RING_BANDS
    const uint32_t ph0 = phase;                // bars[1] and bars[2] are at phase 0
    // Parity of the wait for band b: slot b % nslots, its (b / nslots)-th use.
    auto parity = [&](int b) -> uint32_t {
        return ((b % nslots == 0 ? ph0 : 0u) + (uint32_t)(b / nslots)) & 1u;
    };
    auto issue = [&](int b) {  // thread 0
        const int s = b % nslots;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        fence_proxy_async_global();
        mbar_arrive_expect_tx(&bars[s], uint32_t(n) * BAND * 4);
        for (int j = 0; j < n; ++j)
            bulk_load(ring + (s * n + j) * BAND,
                      p.partials + (size_t)partial_slot(p, c_first + j, t_sk) * TILE_FLOATS +
                          b * BAND,
                      BAND * 4, &bars[s]);
    };
    __syncthreads();  // the ring's previous contents are read
    const int first = min(nslots, NBANDS);
    if (tid == 0)
        for (int b = 0; b < first; ++b) issue(b);
    int issued = first;
#pragma unroll 1
    for (int band = 0; band < NBANDS; ++band) {
        const int s = band % nslots;
        const bool got = mbar_wait_bounded(&bars[s], parity(band), p.timeout_ns);
        if (__syncthreads_or(!got)) {
            if (tid == 0) {
                atomicOr(p.err, kErrWaitTimeout);
                for (int b = band; b < issued; ++b) {
                    if (!mbar_wait_bounded(&bars[b % nslots], parity(b), 1000000000ull)) {
                        atomicOr(p.err, kErrDrainTimeout);
                        break;
                    }
                }
            }
            __syncthreads();
            return false;
        }
        const float *slot = ring + s * n * BAND;
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
            const int f = k * NT + tid;
            float4 sum = ld_shared_f4(slot + f * 4);
#pragma unroll 1
            for (int j = 1; j < n; ++j) {
                const float4 x = ld_shared_f4(slot + j * BAND + f * 4);
                sum.x += x.x;
                sum.y += x.y;
                sum.z += x.z;
                sum.w += x.w;
            }
            const int e4 = band * 4 + k;
            store_c4(p, tm * BM + acc_row(tid, e4 >> 1), tn * BN + acc_col(tid, e4 & 1), sum);
        }
        __syncthreads();  // slot s is read by every thread
        if (band + nslots < NBANDS) {
            if (tid == 0) issue(band + nslots);
            ++issued;
        }
    }
    phase = ph0 ^ (uint32_t)(((NBANDS + nslots - 1) / nslots) & 1);  // bars[0]'s uses
    return true;
}

template <int FM, int STAGES, int TM>
__global__ void __launch_bounds__(Cfg<TM>::NT, 1)
    sgemm_tile_kernel(const __grid_constant__ CUtensorMap mapA,
                      const __grid_constant__ CUtensorMap mapB, const TileParams p) {
    using L = SmemLayout<FM, STAGES>;
    using C = Cfg<TM>;
    extern __shared__ __align__(1024) uint8_t smem[];
    float *stages = reinterpret_cast<float *>(smem);
    float *at_buf = reinterpret_cast<float *>(smem + L::at_off);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L::bar_off);
    uint64_t *red_bar = reinterpret_cast<uint64_t *>(smem + L::redbar_off);
    uint64_t *pre_bar = reinterpret_cast<uint64_t *>(smem + L::prebar_off);
    uint32_t red_phase = 0;
    bool prefetched = false;  // the partner prefetch was issued (uniform)
    volatile int *flags = reinterpret_cast<volatile int *>(smem + L::flag_off);
    constexpr int AT_FLOATS = BK * AtRow<FM>::value;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp / C::WARPS_N, wn = warp % C::WARPS_N;
    const int ty = lane >> 3, tx = lane & 7;
    const int G = gridDim.x, cta = blockIdx.x;

    // Number of k-iterations this CTA runs, over all its units.
    const int n_dp = cta < p.dp_tiles ? (p.dp_tiles - 1 - cta) / G + 1 : 0;
    const int sk_total = p.sk_tiles * p.kt_total;
    const int sk_begin = min(cta * p.sk_share, sk_total);
    const int sk_end = min(sk_begin + p.sk_share, sk_total);
    const int q_total = n_dp * p.kt_total + (sk_end - sk_begin);
    if (q_total == 0) return;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
        mbar_init(red_bar, 1);
        mbar_init(&pre_bar[0], 1);
        mbar_init(&pre_bar[1], 1);
        flags[1] = 0;
        fence_barrier_init();
        prefetch_tensormap(&mapA);
        prefetch_tensormap(&mapB);
    }
    __syncthreads();

    // ---- copy producer state: used by thread 0 only, so it lives in shared
    // memory rather than in every thread's registers ----
    ProducerState &ps = *reinterpret_cast<ProducerState *>(smem + L::prod_off);
    UnitIter &prod = ps.it;
    int &pq = ps.pq, &p_tm = ps.tm, &p_tn = ps.tn, &p_k = ps.k, &p_k1 = ps.k1;
    if (tid == 0) {
        prod.init(p, cta);
        pq = p_tm = p_tn = p_k = p_k1 = 0;
    }
    auto issue_next = [&]() {
        if (pq >= q_total) return;
        if (p.skip_loads_from >= 0 && pq >= p.skip_loads_from) return;
        if (p_k >= p_k1) {
            int tile;
            prod.next(p, G, tile, p_k, p_k1);
            tile_coords(p, tile, p_tm, p_tn);
        }
        const int s = pq % STAGES;
        float *sa = stages + s * STAGE_FLOATS;
        float *sb = sa + A_STAGE_FLOATS;
        mbar_arrive_expect_tx(&full[s], STAGE_TX_BYTES);
        tma_load_2d(sa, &mapA, &full[s], p_k * BK, p_tm * BM);
        tma_load_2d(sb, &mapB, &full[s], p_tn * BN, p_k * BK);
        ++p_k;
        ++pq;
    };
    if (tid == 0)
        for (int s = 0; s < STAGES; ++s) issue_next();

    // ---- consumers (all threads) ----
    UnitIter cons;
    cons.init(p, cta);
    int q = 0;
    bool aborted = false;
    int timed_out = 0;  // made uniform over the CTA by __syncthreads_or

    if (!mbar_wait_bounded(&full[0], 0, p.timeout_ns)) {
        timed_out = 1;
        atomicOr(p.err, kErrWaitTimeout);
    }
    transpose_slice<FM>(stages, at_buf, tid);
    if (__syncthreads_or(timed_out)) aborted = true;

    int tile, k0, k1;
    while (!aborted && cons.next(p, G, tile, k0, k1)) {
        int tm, tn;
        tile_coords(p, tile, tm, tn);
        Acc<FM, TM> acc;
        acc_zero<FM, TM>(acc);

        // A two-piece stream-K tile whose head piece is this CTA's final
        // unit: the partner's piece is its first unit and normally finished
        // long ago.  If its ticket is already in at the start of the last
        // slice, its partial tile is prefetched into the ring stages that are
        // already idle, and this CTA finishes the tile without writing a
        // partial or taking a ticket.  (The sum is the same: this CTA's piece
        // is the first in CTA order.)
        const bool whole = (k0 == 0 && k1 == p.kt_total);
        const int t_sk = tile - p.dp_tiles;
        bool predict = false;
        if (STAGES == 3 && !whole && k0 == 0 && q + (k1 - k0) == q_total) {
            const int cf = (t_sk * p.kt_total) / p.sk_share;
            const int cl = (t_sk * p.kt_total + p.kt_total - 1) / p.sk_share;
            predict = (cf == cta && cl == cta + 1);
        }

        for (int kt = k0; kt < k1; ++kt, ++q) {
            const int s = q % STAGES;
            if (q + 1 < q_total) {
                const int s1 = (q + 1) % STAGES;
                if (!mbar_wait_bounded(&full[s1], ((q + 1) / STAGES) & 1, p.timeout_ns)) {
                    timed_out = 1;
                    atomicOr(p.err, kErrWaitTimeout);
                }
                transpose_slice<FM>(stages + s1 * STAGE_FLOATS, at_buf + ((q + 1) & 1) * AT_FLOATS,
                                    tid);
            }
            if (predict && kt == k1 - 1 && tid == 0) {
                // Last slice: stage s is in use; the other two are idle.
                const int arrived = ld_acquire_gpu(p.counters + t_sk);
                flags[2] = arrived == 1;
                if (arrived == 1) {
                    fence_proxy_async_global();
                    const char *src = reinterpret_cast<const char *>(
                        p.partials + (size_t)partial_slot(p, cta + 1, t_sk) * TILE_FLOATS);
                    constexpr uint32_t kStage = STAGE_FLOATS * 4;
                    mbar_arrive_expect_tx(&pre_bar[0], 2 * kStage);
                    bulk_load(stages + ((s + 1) % STAGES) * STAGE_FLOATS, src, kStage, &pre_bar[0]);
                    bulk_load(stages + ((s + 2) % STAGES) * STAGE_FLOATS, src + kStage, kStage,
                              &pre_bar[0]);
                }
            }
            compute_slice<FM, TM>(at_buf + (q & 1) * AT_FLOATS,
                                  stages + s * STAGE_FLOATS + A_STAGE_FLOATS, acc, wm, wn, ty, tx);
            if (__syncthreads_or(timed_out)) {
                if (predict && kt == k1 - 1 && flags[2]) prefetched = true;
                aborted = true;
                ++q;
                break;
            }
            if (tid == 0) issue_next();
        }
        if (aborted) break;

        if (predict && flags[2]) {
            // The last stage is idle now: bring in the rest of the partner's
            // partial (the first two stages' worth is already on its way).
            prefetched = true;
            const int s_last = (q - 1) % STAGES;
            constexpr uint32_t kStage = STAGE_FLOATS * 4;
            constexpr uint32_t kRest = TILE_FLOATS * 4 - 2 * kStage;
            if (tid == 0) {
                const char *src = reinterpret_cast<const char *>(
                    p.partials + (size_t)partial_slot(p, cta + 1, t_sk) * TILE_FLOATS);
                mbar_arrive_expect_tx(&pre_bar[1], kRest);
                bulk_load(stages + s_last * STAGE_FLOATS, src + 2 * kStage, kRest, &pre_bar[1]);
            }
            bool ok = mbar_wait_bounded(&pre_bar[0], 0, p.timeout_ns);
            ok = mbar_wait_bounded(&pre_bar[1], 0, p.timeout_ns) && ok;
            if (!ok) atomicOr(p.err, kErrWaitTimeout);
            // The partner's partial tile now fills the ring in the order
            // stages s_last + 1, s_last + 2, s_last; this CTA's piece is the
            // first in CTA order.
            constexpr int NT = Cfg<TM>::NT;
            constexpr int PER_STAGE = STAGE_FLOATS / 4 / NT;  // float4 rows per stage
#pragma unroll 1
            for (int e4 = 0; e4 < TILE_FLOATS / NT / 4; ++e4) {
                const float *part = stages + ((s_last + 1 + e4 / PER_STAGE) % STAGES) * STAGE_FLOATS;
                const float4 x = ld_shared_f4(part + ((e4 % PER_STAGE) * NT + tid) * 4);
                float4 v = acc_f4(acc, e4);
                v.x += x.x;
                v.y += x.y;
                v.z += x.z;
                v.w += x.w;
                store_c4(p, tm * BM + acc_row(tid, e4 >> 1), tn * BN + acc_col(tid, e4 & 1), v);
            }
            if (tid == 0) p.counters[t_sk] = 0;
        } else if (whole) {
            store_tile<FM, TM>(acc, p, tm, tn, wm, wn, ty, tx);
        } else {
            float *slot = p.partials + (size_t)partial_slot(p, cta, t_sk) * TILE_FLOATS;
            write_partial<FM, TM>(slot, acc, tid);
            __threadfence();
            __syncthreads();
            const int c_first = (t_sk * p.kt_total) / p.sk_share;
            const int c_last = (t_sk * p.kt_total + p.kt_total - 1) / p.sk_share;
            if (tid == 0) {
                const int old = atomicAdd(&p.counters[t_sk], 1);
                flags[1] = (old == c_last - c_first) ? 1 : 0;
            }
            __syncthreads();
            if (flags[1]) {
                __threadfence();
                // Every piece, this CTA's included, is in its slot.  The
                // final unit's ring is idle (every copy issued has been
                // consumed): stage the pieces there.
                constexpr int kRingPieces = STAGES * STAGE_FLOATS / (4 * Cfg<TM>::NT * 4);
                if (q == q_total && c_last - c_first + 1 <= kRingPieces) {
                    // red_bar and the two pre_bar barriers follow each other
                    // (waits on them are bounded; a timeout drains inside).
                    fixup_staged<TM, STAGES>(p, tm, tn, t_sk, c_first, c_last, tid, stages, red_bar,
                                             red_phase);
                } else {
                    fixup_from_l2<TM>(p, tm, tn, t_sk, c_first, c_last, tid);
                }
                if (tid == 0) p.counters[t_sk] = 0;
            }
        }
    }

    if (aborted && tid == 0) {
        // Wait (bounded) for every copy issued but not yet consumed, so none
        // lands in shared memory after this CTA has exited.  q is the first
        // position not yet transposed; positions [q, pq) may be in flight.
        if (prefetched && !mbar_wait_bounded(&pre_bar[0], 0, 1000000000ull))
            atomicOr(p.err, kErrDrainTimeout);
        for (int j = q; j < pq; ++j) {
            if (!mbar_wait_bounded(&full[j % STAGES], (j / STAGES) & 1, 1000000000ull)) {
                atomicOr(p.err, kErrDrainTimeout);
                break;
            }
        }
    }
}

template <int FM, int STAGES, int TM>
cudaError_t launch_impl(const CUtensorMap &mapA, const CUtensorMap &mapB, const TileParams &p,
                        int grid, cudaStream_t stream) {
    using L = SmemLayout<FM, STAGES>;
    sgemm_tile_kernel<FM, STAGES, TM><<<grid, Cfg<TM>::NT, L::total, stream>>>(mapA, mapB, p);
    return cudaGetLastError();
}

template <int FM, int STAGES, int TM>
cudaError_t configure_impl() {
    using L = SmemLayout<FM, STAGES>;
    return cudaFuncSetAttribute(sgemm_tile_kernel<FM, STAGES, TM>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::total);
}

// The instantiated configurations: (multiply-add form, ring stages, micro-tile rows).
// (8-row micro-tiles with 4 warps per scheduler measured slower on GB300 and
// spill at their 128-register limit, so they are not instantiated.)
#define SGEMM_TILE_CONFIGS(X)       \
    X(kFmaScalar, 3, 16)            \
    X(kFmaPairMovA, 3, 16)          \
    X(kFmaPairDupA, 3, 16)          \
    X(kFmaPairMovB, 3, 16)          \
    X(kFmaPairMovB, 4, 16)

constexpr int config_key(int fm, int st, int tm) { return (fm * 10 + st) * 100 + tm; }

}  // namespace

size_t tile_smem_bytes(int fma_mode, int stages, int tm) {
#define SGEMM_SMEM(FM, S, TM) \
    if (config_key(fma_mode, stages, tm) == config_key(FM, S, TM)) return SmemLayout<FM, S>::total;
    SGEMM_TILE_CONFIGS(SGEMM_SMEM)
#undef SGEMM_SMEM
    return 0;
}

int tile_threads(int tm) { return tm == 8 ? Cfg<8>::NT : Cfg<16>::NT; }

cudaError_t launch_tile(int fma_mode, int stages, int tm, const CUtensorMap &mapA,
                        const CUtensorMap &mapB, const TileParams &p, int grid,
                        cudaStream_t stream) {
#define SGEMM_LAUNCH(FM, S, TM)                                       \
    if (config_key(fma_mode, stages, tm) == config_key(FM, S, TM)) \
        return launch_impl<FM, S, TM>(mapA, mapB, p, grid, stream);
    SGEMM_TILE_CONFIGS(SGEMM_LAUNCH)
#undef SGEMM_LAUNCH
    return cudaErrorInvalidValue;
}

cudaError_t tile_configure(int fma_mode, int stages, int tm) {
#define SGEMM_CONF(FM, S, TM)                                         \
    if (config_key(fma_mode, stages, tm) == config_key(FM, S, TM)) \
        return configure_impl<FM, S, TM>();
    SGEMM_TILE_CONFIGS(SGEMM_CONF)
#undef SGEMM_CONF
    return cudaErrorInvalidValue;
}

}  // namespace sgemm
