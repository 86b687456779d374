// Split-K SIMT FP32 GEMM for sm_103a: C = alpha * A * B + beta * C, row-major,
// for products with few tiles (the whole output fits about one wave of 64 x
// 128 tiles) and operands of any alignment.
//
// "Optimizing Matrix Multiply on CUDA, Part 2", section "Selecting Among Three
// Kernels", keeps a split-K variant beside the two tile sizes: K is cut into
// pieces so that more SMs get work when there are few tiles, and the pieces
// are added afterwards.  On GB300 that combination through global memory (a
// partial tile written, a ticket, the last piece's CTA reading the others
// back) costs several microseconds per tile, which is as much as a small
// product's whole main loop.  Here the split stays inside one CTA: one CTA of
// 256 threads owns a 64 x 128 tile (four groups of 64 threads) or a 64 x 64
// tile (eight groups of one warp); each group takes its part of every slice of
// kKsBK k, and at the end the groups' sums meet in shared memory and are
// added in group order.  The SM then holds eight warps of independent
// multiply-adds (two per scheduler) for one tile, where a 64 x 128 tile of 64
// threads would hold two; the 64 x 64 tile spreads small products over twice
// as many SMs.
//
// Each thread keeps a 16 x 8 micro-tile of the tile's sums (warps of 64 x 64,
// lanes 4 x 8, rows in groups of four 16 apart, columns in two groups of four
// 32 apart), updated per k from four 128-bit shared loads of A and two of B by
// 64 packed FP32 fma (__ffma2_rn, pairs along m), as in the mid-size kernel.
//
// Global -> shared staging is a ring of kKsStages slices filled by cp.async
// ("Part 2", section "Overlapping Loads and Computation"); any alignment and
// leading dimension works without a copy pass:
//   - A in 4-byte copies straight to a k-major tile ("Optimizing CUDA matmul,
//     steps 4 to 6", section "Two ladders, one kernel": the transposed tile).
//     A warp copies 32 k of one row (four 32-byte sectors, each used whole);
//     the shared-memory side is written one sector at a time, so the 16-byte
//     chunk of row k is XOR-ed with k mod 8 and the eight k of a sector land
//     in eight different bank groups.
//   - B in 16-byte copies when its rows are 16-byte aligned, else in 4-byte
//     copies; a warp copies consecutive columns of one row.
//   Elements outside the matrices are zero-filled by the copy itself, which
//   adds exact zeros ("Part 1", section "Small and Odd Sizes").  In the last
//   slice a group multiplies only the k that exist.
//
// The only waits are on the CTA's own copies (cp.async.wait_group) and its own
// barriers; no CTA depends on another, and the sums are added in a fixed order,
// so the result does not depend on timing.

#include "device_common.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

constexpr int BM = kKsBM;
constexpr int BK = kKsBK;
constexpr int ST = kKsStages;
constexpr int NT = kKsThreads;              // 256
constexpr int A_FLOATS = BK * BM;           // k-major: row k holds BM values
constexpr int A_HALVES = BK / 32;           // 32-k halves of an A row per slice
static_assert(BM == 64 && (BK == 32 || BK == 64) && NT == 256, "the copy and fragment maps");

// A tile of BM x BN (BN = 128 or 64): each k-group holds one 16 x 8 micro-tile
// of the whole tile per thread, so a group is BM * BN / 128 threads (two
// warps or one) and there are NT / that many groups (four or eight).
template <int BN_>
struct KsCfg {
    static constexpr int BN = BN_;
    static constexpr int GT = BM * BN / (16 * 8);  // threads per group: 64 or 32
    static constexpr int KG = NT / GT;             // groups: 4 or 8
    static constexpr int GK = BK / KG;             // k of a slice per group
    static constexpr int WARPS_N = BN / 64;        // warp columns of a group
    static constexpr int B_FLOATS = BK * BN;
    static constexpr int STAGE_FLOATS = A_FLOATS + B_FLOATS;
    static constexpr int TILE_F4 = BM * BN / 4;    // float4 of one tile
    static constexpr int ROW_F4 = BN / 4;          // float4 of one tile row
    static constexpr size_t RING_BYTES = size_t(ST) * STAGE_FLOATS * 4;
    static constexpr size_t SUMS_BYTES = size_t(KG) * TILE_F4 * 16;  // the groups' sums
    static constexpr size_t SMEM_BYTES = RING_BYTES > SUMS_BYTES ? RING_BYTES : SUMS_BYTES;
    static_assert(BN == 128 || BN == 64, "tile widths");
    static_assert(GK % 8 == 0 && KG * GT == NT, "group layout");
    static_assert(SMEM_BYTES <= 232448, "exceeds the 227 KB of shared memory a CTA may use");
};

// Offset (floats) of A element (m, k) in a k-major slice of BM rows.
__device__ __forceinline__ int ks_a_off(int m, int k) {
    return k * BM + (((m >> 2) ^ (k & 7)) << 2) + (m & 3);
}

__device__ __forceinline__ void ks_tile_coords(const MidParams &p, int t, int &tm, int &tn) {
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int rows = min(p.tiles_m - first_m, p.group_m);
    const int r = t - g * per_group;
    tm = first_m + r % rows;
    tn = r / rows;
}

// Copies of k-slice ks of tile (tm, tn) into stage `st`.
template <int BVEC, int BN>
__device__ __forceinline__ void ks_issue(const MidParams &p, float *st, int tm, int tn, int ks,
                                         int tid) {
    float *sa = st;
    float *sb = st + A_FLOATS;
    const int k_base = ks * BK;
    // A: thread t copies k = t % 32 (+ 32 h) of rows t / 32 + 8 j (j < 8).
#pragma unroll
    for (int h = 0; h < A_HALVES; ++h) {
        const int kin = (tid & 31) + 32 * h;
        const int m_in = tid >> 5;
        const int gm0 = tm * BM + m_in;
        const bool k_ok = k_base + kin < p.K;
        const float *src = p.A + (long long)gm0 * p.lda + k_base + kin;
        const long long step = 8LL * p.lda;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const bool ok = k_ok && gm0 + 8 * j < p.M;
            cp_async4(sa + ks_a_off(m_in + 8 * j, kin), ok ? src : p.A, ok ? 4u : 0u);
            src += step;
        }
    }
    const int n_base = tn * BN;
    if (BVEC == 4) {
        // BK * BN / 4 chunks of 16 bytes, CPR to a row; chunk t + 256 q is
        // row t / CPR + (256 / CPR) q, columns 4 (t % CPR) .. + 3.
        constexpr int CPR = BN / 4;
        constexpr int RPQ = NT / CPR;
        const int n4 = (tid % CPR) * 4;
        const int cols = min(4, p.N - (n_base + n4));
        const int kin0 = tid / CPR;
        const float *src = p.B + (long long)(k_base + kin0) * p.ldb + n_base + n4;
        const long long step = (long long)RPQ * p.ldb;
#pragma unroll
        for (int q = 0; q < BK * BN / 4 / NT; ++q) {
            const bool ok = k_base + kin0 + RPQ * q < p.K && cols > 0;
            cp_async16(sb + (kin0 + RPQ * q) * BN + n4, ok ? src : p.B,
                       ok ? uint32_t(cols) * 4u : 0u);
            src += step;
        }
    } else {
        // BK * BN elements; element t + 256 q is row t / BN + (256 / BN) q,
        // column t % BN.
        constexpr int RPQ = NT / BN;
        const int n = tid % BN;
        const bool n_ok = n_base + n < p.N;
        const int kin0 = tid / BN;
        const float *src = p.B + (long long)(k_base + kin0) * p.ldb + n_base + n;
        const long long step = (long long)RPQ * p.ldb;
#pragma unroll
        for (int q = 0; q < BK * BN / NT; ++q) {
            const bool ok = n_ok && k_base + kin0 + RPQ * q < p.K;
            cp_async4(sb + (kin0 + RPQ * q) * BN + n, ok ? src : p.B, ok ? 4u : 0u);
            src += step;
        }
    }
}

// A thread's sums: v[ip][j] = (C[2ip][j], C[2ip+1][j]) over its sixteen rows
// r * 16 + ty * 4 + (0..3) and eight columns wn * 64 + c * 32 + tx * 4 + (0..3).
struct KsAcc {
    float2 v[8][8];
};

// Fragment addresses of one thread: the four A bases (one per k mod 4, the
// XOR of row chunk ty with k mod 4) and the B base, as shared-window bytes.
template <int BN>
struct KsFrag {
    uint32_t pa[4];
    uint32_t pb;
    uint32_t a0;  // the stage's A tile
    int ty;
    // Row k0 + k of the stage, k0 a multiple of 8 and k known at compile
    // time (unrolled loops), so that k mod 8 picks the swizzle statically.
    __device__ __forceinline__ void load(int k0, int k, float4 (&a)[4], float4 (&b)[2]) const {
        // Rows r * 16 + ty * 4 .. + 3 sit in chunk 4 r + ty of row kk, XOR-ed
        // with kk mod 8 = k mod 8: (4 r) ^ (k & 4) plus ty ^ (k & 3).
        const int kk = k0 + k;
#pragma unroll
        for (int r = 0; r < 4; ++r)
            a[r] = lds128(pa[k & 3] + 4u * (kk * BM + (((4 * r) ^ (k & 4)) << 2)));
        b[0] = lds128(pb + 4u * (kk * BN));
        b[1] = lds128(pb + 4u * (kk * BN + 32));
    }
    // kk known only at run time.
    __device__ __forceinline__ void load_dyn(int kk, float4 (&a)[4], float4 (&b)[2]) const {
#pragma unroll
        for (int r = 0; r < 4; ++r)
            a[r] = lds128(a0 + 4u * (kk * BM + (((4 * r + ty) ^ (kk & 7)) << 2)));
        b[0] = lds128(pb + 4u * (kk * BN));
        b[1] = lds128(pb + 4u * (kk * BN + 32));
    }
};

__device__ __forceinline__ void ks_fma(KsAcc &acc, const float4 (&a)[4], const float4 (&b)[2]) {
#pragma unroll
    for (int ip = 0; ip < 8; ++ip) {
        const float4 &av = a[ip >> 1];
        const float2 a2 = (ip & 1) ? make_float2(av.z, av.w) : make_float2(av.x, av.y);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 &bv = b[j >> 2];
            const float bj = (j & 3) == 0 ? bv.x : (j & 3) == 1 ? bv.y : (j & 3) == 2 ? bv.z : bv.w;
            acc.v[ip][j] = __ffma2_rn(a2, make_float2(bj, bj), acc.v[ip][j]);
        }
    }
}

// The group's GK k (k0 .. k0 + GK - 1 of the stage whose fragment bases are
// in `f`), fully unrolled with fragments double-buffered in registers.
template <int GK, int BN>
__device__ __forceinline__ void ks_compute_full(const KsFrag<BN> &f, int k0, KsAcc &acc) {
    float4 fa[2][4], fb[2][2];
    f.load(k0, 0, fa[0], fb[0]);
#pragma unroll
    for (int k = 0; k < GK; ++k) {
        if (k + 1 < GK) f.load(k0, k + 1, fa[(k + 1) & 1], fb[(k + 1) & 1]);
        ks_fma(acc, fa[k & 1], fb[k & 1]);
    }
}

// The first `kc` (< GK) of the group's k, one at a time (the last slice).
template <int BN>
__device__ __forceinline__ void ks_compute_part(const KsFrag<BN> &f, int k0, int kc, KsAcc &acc) {
#pragma unroll 1
    for (int k = 0; k < kc; ++k) {
        float4 a[4], b[2];
        f.load_dyn(k0 + k, a, b);
        ks_fma(acc, a, b);
    }
}

// Float4 number e4 (0..31) of a thread's sums: row e4 / 2 of its sixteen,
// columns (e4 % 2) * 32 + tx * 4 .. + 3.  Called with e4 known after
// unrolling, the switch folds away and the sums stay in registers.
__device__ __forceinline__ float4 ks_f4(const KsAcc &acc, int e4) {
    switch (e4) {
#define SGEMM_KS_E4(E)                                                                     \
    case E: {                                                                              \
        const int ip = (E) >> 2, hi = ((E) >> 1) & 1, j0 = ((E)&1) * 4;                    \
        return hi ? make_float4(acc.v[ip][j0].y, acc.v[ip][j0 + 1].y, acc.v[ip][j0 + 2].y, \
                                acc.v[ip][j0 + 3].y)                                       \
                  : make_float4(acc.v[ip][j0].x, acc.v[ip][j0 + 1].x, acc.v[ip][j0 + 2].x, \
                                acc.v[ip][j0 + 3].x);                                      \
    }
        SGEMM_KS_E4(0) SGEMM_KS_E4(1) SGEMM_KS_E4(2) SGEMM_KS_E4(3) SGEMM_KS_E4(4)
        SGEMM_KS_E4(5) SGEMM_KS_E4(6) SGEMM_KS_E4(7) SGEMM_KS_E4(8) SGEMM_KS_E4(9)
        SGEMM_KS_E4(10) SGEMM_KS_E4(11) SGEMM_KS_E4(12) SGEMM_KS_E4(13) SGEMM_KS_E4(14)
        SGEMM_KS_E4(15) SGEMM_KS_E4(16) SGEMM_KS_E4(17) SGEMM_KS_E4(18) SGEMM_KS_E4(19)
        SGEMM_KS_E4(20) SGEMM_KS_E4(21) SGEMM_KS_E4(22) SGEMM_KS_E4(23) SGEMM_KS_E4(24)
        SGEMM_KS_E4(25) SGEMM_KS_E4(26) SGEMM_KS_E4(27) SGEMM_KS_E4(28) SGEMM_KS_E4(29)
        SGEMM_KS_E4(30) SGEMM_KS_E4(31)
#undef SGEMM_KS_E4
    }
    return make_float4(0.f, 0.f, 0.f, 0.f);
}

// C = alpha * s (+ beta C, epilogue) for columns n .. n+3 of row m.
__device__ __forceinline__ void ks_store4(const MidParams &p, int m, int n, float4 s) {
    if (m >= p.M || n >= p.N) return;
    float *crow = p.C + (long long)m * p.ldc;
    float o[4] = {p.alpha * s.x, p.alpha * s.y, p.alpha * s.z, p.alpha * s.w};
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

template <int BVEC, int BN>
__global__ void __launch_bounds__(NT, 1) sgemm_ksplit_kernel(const __grid_constant__ MidParams p) {
    using Cf = KsCfg<BN>;
    constexpr int GK = Cf::GK, KG = Cf::KG, STAGE_FLOATS = Cf::STAGE_FLOATS;
    constexpr int TILE_F4 = Cf::TILE_F4, ROW_F4 = Cf::ROW_F4;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    float *ring = reinterpret_cast<float *>(smem_raw);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int grp = warp / Cf::WARPS_N;  // k-group
    const int wn = warp % Cf::WARPS_N;   // warp column (64 wide) within the tile
    const int ty = lane >> 3, tx = lane & 7;

    int tm, tn;
    ks_tile_coords(p, blockIdx.x, tm, tn);
    const int n_slices = p.kt_total;

#pragma unroll
    for (int s = 0; s < ST - 1; ++s) {
        if (s < n_slices) ks_issue<BVEC, BN>(p, ring + s * STAGE_FLOATS, tm, tn, s, tid);
        cp_async_commit();
    }
    KsAcc acc;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc.v[i][j] = make_float2(0.f, 0.f);

    // Fragment bases relative to stage 0; a stage adds s * STAGE_FLOATS * 4.
    KsFrag<BN> f0;
#pragma unroll
    for (int x = 0; x < 4; ++x) f0.pa[x] = smem_addr(ring + ((ty ^ x) << 2));
    f0.pb = smem_addr(ring + A_FLOATS + wn * 64 + tx * 4);
    f0.a0 = smem_addr(ring);
    f0.ty = ty;
    const int k_grp = grp * GK;                        // the group's first k in a slice
    const int full = p.K / BK;                         // slices with every k present
    const int k_last = p.K - full * BK - k_grp;        // the group's k in the last slice
    const int kc_last = k_last < 0 ? 0 : (k_last > GK ? GK : k_last);

#pragma unroll 1
    for (int i = 0; i < n_slices; ++i) {
        cp_async_wait<ST - 2>();  // this thread's copies of slice i are in
        __syncthreads();          // everyone's are; slice i - 1 is consumed
        if (i + ST - 1 < n_slices)
            ks_issue<BVEC, BN>(p, ring + ((i + ST - 1) % ST) * STAGE_FLOATS, tm, tn, i + ST - 1,
                               tid);
        cp_async_commit();
        KsFrag<BN> f = f0;
        const uint32_t so = 4u * (uint32_t)((i % ST) * STAGE_FLOATS);
#pragma unroll
        for (int x = 0; x < 4; ++x) f.pa[x] += so;
        f.pb += so;
        f.a0 += so;
        if (i < full)
            ks_compute_full<GK>(f, k_grp, acc);
        else if (kc_last > 0)
            ks_compute_part(f, k_grp, kc_last, acc);
    }
    cp_async_wait<0>();
    __syncthreads();  // every group is done with the ring

    // The groups' sums, float4 (row, c4) of group g at S[g][row * ROW_F4 + c4].
    // (Unrolled: each store takes its sums straight from registers; through
    // the rolled switch of ks_f4 the write took 2.6 us at 1023 x 1025 x 513,
    // unrolled 0.5 us.)
    float4 *S = reinterpret_cast<float4 *>(ring);
#pragma unroll
    for (int e4 = 0; e4 < 32; ++e4) {
        const int ri = e4 >> 1;  // r * 4 + i
        const int row = (ri >> 2) * 16 + ty * 4 + (ri & 3);
        const int c4 = wn * 16 + (e4 & 1) * 8 + tx;
        S[grp * TILE_F4 + row * ROW_F4 + c4] = ks_f4(acc, e4);
    }
    __syncthreads();
    // Thread t adds float4 t + 256 q of the groups in group order and stores
    // it: consecutive threads cover consecutive columns of a row.
    const int m0 = tm * BM, n0 = tn * BN;
#pragma unroll 1
    for (int q = 0; q < TILE_F4 / NT; ++q) {
        const int f = tid + NT * q;
        float4 s = S[f];
#pragma unroll
        for (int g = 1; g < KG; ++g) {
            const float4 x = S[g * TILE_F4 + f];
            s.x += x.x;
            s.y += x.y;
            s.z += x.z;
            s.w += x.w;
        }
        ks_store4(p, m0 + f / ROW_F4, n0 + (f % ROW_F4) * 4, s);
    }
}

template <int BVEC, int BN>
cudaError_t launch_impl(const MidParams &p, int grid, cudaStream_t stream) {
    sgemm_ksplit_kernel<BVEC, BN><<<grid, NT, KsCfg<BN>::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

template <int BVEC, int BN>
cudaError_t configure_impl() {
    cudaError_t e = cudaFuncSetAttribute(sgemm_ksplit_kernel<BVEC, BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)KsCfg<BN>::SMEM_BYTES);
    // No carveout preference: the driver's choice leaves L1 more room than
    // the largest shared-memory carveout, and the 4-byte copies (cp.async.ca)
    // pass through L1 (1023^3 63.5 -> 59.4-60.1 us, 1025^3 71.7 -> 67.6-68.3).
    return e;
}

// The instantiated forms: (B copy width, tile width).
#define SGEMM_KS_FORMS(X) X(4, 128) X(1, 128) X(4, 64) X(1, 64)

}  // namespace

cudaError_t launch_ksplit(int b_vec, int bn, const MidParams &p, int grid, cudaStream_t stream) {
#define SGEMM_KS_LAUNCH(BV, BN_) \
    if (b_vec == BV && bn == BN_) return launch_impl<BV, BN_>(p, grid, stream);
    SGEMM_KS_FORMS(SGEMM_KS_LAUNCH)
#undef SGEMM_KS_LAUNCH
    return cudaErrorInvalidValue;
}

cudaError_t ksplit_configure(int b_vec, int bn) {
#define SGEMM_KS_CONF(BV, BN_) \
    if (b_vec == BV && bn == BN_) return configure_impl<BV, BN_>();
    SGEMM_KS_FORMS(SGEMM_KS_CONF)
#undef SGEMM_KS_CONF
    return cudaErrorInvalidValue;
}

}  // namespace sgemm
