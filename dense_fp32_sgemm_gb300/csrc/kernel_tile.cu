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
// (k / 4) mod 8, so both the fill and the inner-loop reads are free of bank
// conflicts.
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
                        const float4 cv = *reinterpret_cast<const float4 *>(crow + n);
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

// Sum the pieces of stream-K tile t_sk, CTAs c_first..c_last, in CTA order;
// this CTA's own piece is taken from registers.
template <int FM, int TM>
__device__ __forceinline__ void reduce_pieces(Acc<FM, TM> &acc, const TileParams &p, int cta,
                                              int t_sk, int c_first, int c_last, int tid) {
    constexpr int NT = Cfg<TM>::NT;
#pragma unroll
    for (int e4 = 0; e4 < TILE_FLOATS / NT / 4; ++e4) {
        const int ti = e4 >> 1, c = e4 & 1;
        const float4 own = make_float4(acc.at(ti, c * 4 + 0), acc.at(ti, c * 4 + 1),
                                       acc.at(ti, c * 4 + 2), acc.at(ti, c * 4 + 3));
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int cc = c_first; cc <= c_last; ++cc) {
            float4 v;
            if (cc == cta) {
                v = own;
            } else {
                const float *slot =
                    p.partials + (size_t)partial_slot(p, cc, t_sk) * TILE_FLOATS;
                v = __ldcg(reinterpret_cast<const float4 *>(slot) + e4 * NT + tid);
            }
            if (cc == c_first) {
                s = v;
            } else {
                s.x += v.x;
                s.y += v.y;
                s.z += v.z;
                s.w += v.w;
            }
        }
        acc.at(ti, c * 4 + 0) = s.x;
        acc.at(ti, c * 4 + 1) = s.y;
        acc.at(ti, c * 4 + 2) = s.z;
        acc.at(ti, c * 4 + 3) = s.w;
    }
}

// The same sum for a CTA's final unit, when its TMA ring is idle: the other
// pieces' partial tiles are pulled into the ring with bulk asynchronous
// copies (one L2 round trip per round, no registers), then added from
// shared memory in CTA order.  ROUNDS splits the tile so that all other
// pieces of a round fit the ring: 1 other piece -> 1 round, 2 -> 2, 3 or 4
// -> 4.  Returns false if a copy did not arrive in time (the error word is
// set; the caller still waits for the copies before exiting).
template <int FM, int TM, int ROUNDS>
__device__ __forceinline__ bool reduce_pieces_staged(Acc<FM, TM> &acc, const TileParams &p,
                                                     int cta, int t_sk, int c_first, int c_last,
                                                     int tid, float *ring, uint64_t *bar,
                                                     uint32_t &phase) {
    constexpr int NT = Cfg<TM>::NT;
    constexpr int E4 = TILE_FLOATS / NT / 4;
    constexpr int E = E4 / ROUNDS;                    // float4 per thread per round
    constexpr uint32_t CHUNK = uint32_t(E) * NT * 16;  // bytes per piece per round
    const int others = c_last - c_first;
    bool ok = true;
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
        if (tid == 0) {
            fence_proxy_async_global();
            mbar_arrive_expect_tx(bar, CHUNK * others);
            int j = 0;
            for (int cc = c_first; cc <= c_last; ++cc) {
                if (cc == cta) continue;
                const char *slot = reinterpret_cast<const char *>(
                    p.partials + (size_t)partial_slot(p, cc, t_sk) * TILE_FLOATS);
                bulk_load(reinterpret_cast<char *>(ring) + j * CHUNK, slot + r * CHUNK, CHUNK, bar);
                ++j;
            }
        }
        if (!mbar_wait_bounded(bar, phase, p.timeout_ns)) {
            atomicOr(p.err, kErrWaitTimeout);
            ok = false;
        }
        phase ^= 1u;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int e4 = r * E + e, ti = e4 >> 1, cg = e4 & 1;
            const float4 own = make_float4(acc.at(ti, cg * 4 + 0), acc.at(ti, cg * 4 + 1),
                                           acc.at(ti, cg * 4 + 2), acc.at(ti, cg * 4 + 3));
            float4 sum = own;
            int j = 0;
            for (int cc = c_first; cc <= c_last; ++cc) {
                float4 x;
                if (cc == cta) {
                    x = own;
                } else {
                    x = ld_shared_f4(ring + (size_t)j * (CHUNK / 4) + (e * NT + tid) * 4);
                    ++j;
                }
                if (cc == c_first) {
                    sum = x;
                } else {
                    sum.x += x.x;
                    sum.y += x.y;
                    sum.z += x.z;
                    sum.w += x.w;
                }
            }
            acc.at(ti, cg * 4 + 0) = sum.x;
            acc.at(ti, cg * 4 + 1) = sum.y;
            acc.at(ti, cg * 4 + 2) = sum.z;
            acc.at(ti, cg * 4 + 3) = sum.w;
        }
        __syncthreads();  // the ring is read before the next round overwrites it
    }
    return ok;
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
                int arrived;
                asm volatile("ld.acquire.gpu.global.b32 %0, [%1];"
                             : "=r"(arrived)
                             : "l"(p.counters + t_sk)
                             : "memory");
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
            const float *part[3] = {stages + ((s_last + 1) % STAGES) * STAGE_FLOATS,
                                    stages + ((s_last + 2) % STAGES) * STAGE_FLOATS,
                                    stages + s_last * STAGE_FLOATS};
            constexpr int NT = Cfg<TM>::NT;
            constexpr int PER_STAGE = STAGE_FLOATS / 4 / NT;  // float4 rows per stage
#pragma unroll
            for (int e4 = 0; e4 < TILE_FLOATS / NT / 4; ++e4) {
                const int ti = e4 >> 1, cg = e4 & 1;
                const float4 x =
                    ld_shared_f4(part[e4 / PER_STAGE] + ((e4 % PER_STAGE) * NT + tid) * 4);
                acc.at(ti, cg * 4 + 0) += x.x;
                acc.at(ti, cg * 4 + 1) += x.y;
                acc.at(ti, cg * 4 + 2) += x.z;
                acc.at(ti, cg * 4 + 3) += x.w;
            }
            if (tid == 0) p.counters[t_sk] = 0;
            store_tile<FM, TM>(acc, p, tm, tn, wm, wn, ty, tx);
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
                const int others = c_last - c_first;
                // The final unit's ring is idle (every copy issued has been
                // consumed): stage the other pieces there.
                bool staged_ok = true;
                if (q == q_total && others <= 4) {
                    if (others == 1)
                        staged_ok = reduce_pieces_staged<FM, TM, 1>(acc, p, cta, t_sk, c_first, c_last,
                                                                    tid, stages, red_bar, red_phase);
                    else if (others == 2)
                        staged_ok = reduce_pieces_staged<FM, TM, 2>(acc, p, cta, t_sk, c_first, c_last,
                                                                    tid, stages, red_bar, red_phase);
                    else
                        staged_ok = reduce_pieces_staged<FM, TM, 4>(acc, p, cta, t_sk, c_first, c_last,
                                                                    tid, stages, red_bar, red_phase);
                    if (!staged_ok && tid == 0 &&
                        !mbar_wait_bounded(red_bar, red_phase ^ 1u, 1000000000ull))
                        atomicOr(p.err, kErrDrainTimeout);
                } else {
                    reduce_pieces<FM, TM>(acc, p, cta, t_sk, c_first, c_last, tid);
                }
                if (tid == 0) p.counters[t_sk] = 0;
                store_tile<FM, TM>(acc, p, tm, tn, wm, wn, ty, tx);
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
