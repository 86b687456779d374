// Mid-size SIMT FP32 GEMM for sm_103a: C = alpha * A * B + beta * C,
// row-major, for products too small to fill GB300 with 128 x 256 tiles and
// for operands whose rows the TMA cannot map (a base or a leading dimension
// off 16 bytes).
//
// "Optimizing Matrix Multiply on CUDA, Part 2", sections "Choosing Tiles" and
// "Selecting Among Three Kernels": a 128 x 128 tile of 128 threads with a
// 16 x 8 patch each is the mid-size choice next to the large 128 x 256 one,
// and small sizes want smaller tiles so that more SMs get work.  Here one CTA
// of BM threads (BM = 128 or 64) owns a BM x 128 tile and walks K in slices
// of 16; each thread keeps a 16 x 8 micro-tile of sums (warps of 64 x 64, as
// in the tiled kernel), updated per k from four 128-bit shared loads of A and
// two of B by 64 packed FP32 fma (__ffma2_rn, pairs along m).  Several CTAs
// share an SM (two at BM = 128, four at BM = 64), so that one CTA's copies,
// barriers and epilogue overlap another's multiply-adds.
//
// Global -> shared staging is a ring of kMidStages slices filled by cp.async
// ("Part 2", section "Overlapping Loads and Computation"):
//   - A goes in 4-byte copies that write each element straight to its place
//     in a k-major tile, so a thread's four A values of one k are adjacent
//     ("Optimizing CUDA matmul, steps 4 to 6", section "Two ladders, one
//     kernel": the transposed tile).  A warp's copy covers 16 k of two rows
//     (four 32-byte sectors, each used whole).  The shared-memory side of
//     such a copy is written sector by sector, so the 16-byte chunk index of
//     row k is XOR-ed with (k mod 8): the eight k of a sector land in eight
//     different bank groups, and the inner-loop reads of four chunks stay
//     conflict-free.  (Measured: copies of one row per thread, 32 sectors per
//     instruction, wrote shared memory one sector at a time and kept its
//     pipe 74 % busy.)
//   - B goes in 16-byte copies when its rows are 16-byte aligned, else in
//     4-byte copies; either way a warp covers consecutive columns.
//   Elements outside the matrices are filled with zeros by the copy itself
//   (source size 0 or short), which adds exact zeros ("Part 1", section
//   "Small and Odd Sizes").  No alignment beyond 4 bytes is needed, so no
//   operand is ever copied to aligned rows first.
//
// Work distribution is that of the tiled kernel: a persistent grid computes
// the first dp_tiles tiles whole, round-robin, then shares the k-slices of
// the rest evenly (stream-K, "Part 2", section "Distributing the Partially
// Filled Wave").  Each unit (a tile, or a CTA's range of one) fills and
// drains its own copy pipeline.  A CTA whose range covers part of a tile
// writes its sums to a fixed slot and takes a ticket; the last to arrive adds
// the pieces in CTA order and applies the epilogue, so no CTA waits for
// another and the result does not depend on timing.  It brings the pieces in
// through its then idle ring with cp.async, several copies in flight, each
// thread fetching exactly the sums it adds.  The only waits are on the CTA's
// own copies (cp.async.wait_group) and its own barriers.

#include "device_common.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

constexpr int MBN = kMidBN;
constexpr int MBK = kMidBK;
constexpr int MST = kMidStages;
static_assert(MBK == 16 && MBN == 128, "the copy and fragment maps assume 16 x 128 slices");

template <int BM_>
struct MidCfg {
    static constexpr int BM = BM_;
    static constexpr int NT = BM;                   // 16 x 8 per thread over BM x 128
    static constexpr int WARPS_N = MBN / 64;        // warps of 64 x 64
    static constexpr int A_FLOATS = MBK * BM;       // k-major: row k holds BM values
    static constexpr int B_FLOATS = MBK * MBN;
    static constexpr int STAGE_FLOATS = A_FLOATS + B_FLOATS;
    static constexpr int A_COPIES = A_FLOATS / NT;  // 4-byte copies per thread: 16
    static constexpr int ROW_STEP = NT / 16;        // rows between a thread's copies
    static constexpr int TILE_FLOATS = BM * MBN;
    static constexpr int E4 = TILE_FLOATS / NT / 4;  // float4 of sums per thread: 32
    static constexpr int RING_FLOATS = MST * STAGE_FLOATS;
    static constexpr size_t smem_bytes = size_t(RING_FLOATS) * 4;
    // Fix-up through the ring: a thread's sums in FIX_GROUPS groups of
    // FIX_E4 float4, one group of one piece per ring region.
    static constexpr int FIX_GROUPS = 4;
    static constexpr int FIX_E4 = E4 / FIX_GROUPS;
    static constexpr int FIX_REGION = FIX_E4 * NT * 4;  // floats
    static constexpr int FIX_REGIONS = 4;                // three copies in flight
    static_assert(A_COPIES == 16 && BM / 4 >= 8, "A copy map");
    static_assert(BM % 64 == 0, "warp rows");
    static_assert(FIX_REGIONS * FIX_REGION <= RING_FLOATS, "fix-up regions fit the ring");
};

// Offset (floats) of A element (m, k) in a k-major slice of BM rows: the
// 16-byte chunk m / 4 of row k is XOR-ed with k mod 8.  A copy instruction
// covers 16 k of two rows, and the shared-memory side of a 4-byte cp.async
// is written per 32-byte global sector: the eight k of one sector then land
// in eight different bank groups.
template <int BM>
__device__ __forceinline__ int a_off(int m, int k) {
    return k * BM + (((m >> 2) ^ (k & 7)) << 2) + (m & 3);
}

__device__ __forceinline__ void mid_tile_coords(const MidParams &p, int t, int &tm, int &tn) {
    const int per_group = p.group_m * p.tiles_n;
    const int g = t / per_group;
    const int first_m = g * p.group_m;
    const int rows = min(p.tiles_m - first_m, p.group_m);
    const int r = t - g * per_group;
    tm = first_m + r % rows;
    tn = r / rows;
}

// The units (tile, k-slice range) of one CTA: its round-robin share of the
// whole tiles, then its contiguous range of stream-K slices.  Position `pos`
// of the CTA (its pos-th slice over all units) lies in the unit returned:
// tile, the slice k of that tile, and the end of the CTA's range in it.
struct MidRange {
    int n_dp;      // whole tiles of this CTA
    int sk_begin;  // first stream-K slice (over all stream-K tiles)
    int sk_end;
    __device__ __forceinline__ void unit_of(const MidParams &p, int cta, int G, int pos,
                                            int &tile, int &k, int &kend) const {
        const int dp_pos = n_dp * p.kt_total;
        if (pos < dp_pos) {
            const int u = pos / p.kt_total;
            tile = cta + u * G;
            k = pos - u * p.kt_total;
            kend = p.kt_total;
        } else {
            const int su = sk_begin + (pos - dp_pos);
            const int t = su / p.kt_total;
            tile = p.dp_tiles + t;
            k = su - t * p.kt_total;
            kend = min(p.kt_total, k + (sk_end - su));
        }
    }
};

// Copies of one slice (tile row tm, tile column tn, k-slice ks) into `st`.
template <int BM, int BVEC>
__device__ __forceinline__ void issue_slice(const MidParams &p, float *st, int tm, int tn, int ks,
                                            int tid) {
    using Cf = MidCfg<BM>;
    float *sa = st;
    float *sb = st + Cf::A_FLOATS;
    const int k_base = ks * MBK;
    // A: thread t copies k = t % 16 of rows t / 16 + ROW_STEP * j (j < 16):
    // a warp's copy covers 16 k of two rows (four 32-byte sectors).
    {
        const int kin = tid & 15;
        const int m_in = tid >> 4;
        const int gm0 = tm * BM + m_in;
        const bool k_ok = k_base + kin < p.K;
        const float *src = p.A + (long long)gm0 * p.lda + k_base + kin;
        const long long step = (long long)Cf::ROW_STEP * p.lda;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const bool ok = k_ok && gm0 + Cf::ROW_STEP * j < p.M;
            cp_async4(sa + a_off<BM>(m_in + Cf::ROW_STEP * j, kin), ok ? src : p.A, ok ? 4u : 0u);
            src += step;
        }
    }
    // B: row-major 16 x 128 slice.
    const int n_base = tn * MBN;
    if (BVEC == 4) {
        // 512 chunks of 16 bytes; chunk tid + NT * q is row (tid / 32) +
        // (NT / 32) * q, columns 4 * (tid % 32) .. + 3.
        constexpr int ROWS_PER_Q = Cf::NT / 32;
        const int n4 = (tid & 31) * 4;
        const int cols = min(4, p.N - (n_base + n4));
        const int kin0 = tid >> 5;
        const float *col = p.B + (long long)(k_base + kin0) * p.ldb + n_base + n4;
#pragma unroll
        for (int q = 0; q < 512 / Cf::NT; ++q) {
            const int kin = kin0 + ROWS_PER_Q * q;
            const bool ok = k_base + kin < p.K && cols > 0;
            cp_async16(sb + kin * MBN + n4, ok ? col : p.B, ok ? uint32_t(cols) * 4u : 0u);
            col += (long long)ROWS_PER_Q * p.ldb;
        }
    } else {
        // 2048 elements; element e = tid + NT * q is row e / 128, column e % 128.
        constexpr int ROWS_PER_Q = Cf::NT / MBN;  // rows one round of copies covers (0: part)
        const int n = tid & 127;
        const bool n_ok = n_base + n < p.N;
        const int kin0 = tid >> 7;
        const float *col = p.B + (long long)(k_base + kin0) * p.ldb + n_base + n;
#pragma unroll
        for (int q = 0; q < MBK * MBN / Cf::NT; ++q) {
            const int kin = ROWS_PER_Q > 0 ? kin0 + ROWS_PER_Q * q : (tid + Cf::NT * q) >> 7;
            const int nn = ROWS_PER_Q > 0 ? n : (tid + Cf::NT * q) & 127;
            const bool ok = k_base + kin < p.K && (ROWS_PER_Q > 0 ? n_ok : n_base + nn < p.N);
            const float *src =
                ok ? (ROWS_PER_Q > 0 ? col + (long long)(ROWS_PER_Q * q) * p.ldb
                                     : p.B + (long long)(k_base + kin) * p.ldb + n_base + nn)
                   : p.B;
            cp_async4(sb + kin * MBN + nn, src, ok ? 4u : 0u);
        }
    }
}

// Sums of one thread: v[ip][j] = (C[2ip][j], C[2ip+1][j]) over its sixteen
// rows r * 16 + ty * 4 + (0..3) (r = 0..3; pairs along m) and eight columns
// c * 32 + tx * 4 + (0..3) (c = 0, 1) of its warp's 64 x 64 block.
struct MidAcc {
    float2 v[8][8];
    __device__ __forceinline__ float at(int i, int j) const {
        return (i & 1) ? v[i >> 1][j].y : v[i >> 1][j].x;
    }
};

// One K slice (16 k) of outer products from the stage `st`, fully unrolled:
// fragments are double-buffered in registers (the loads for k + 1 are issued
// before the multiply-adds of k).  (Measured: two passes of an 8-k body, half
// the code, were 1-5 % slower at every size, the smallest included.)
template <int BM>
__device__ __forceinline__ void compute_slice(const float *st, MidAcc &acc, int wm, int wn, int ty,
                                              int tx) {
    const float *sa = st;
    const float *sb = st + MidCfg<BM>::A_FLOATS;
    // Rows r * 16 + ty * 4 .. + 3 sit in chunk wm * 16 + 4 r + ty of row k,
    // XOR-ed with k mod 8: (4 r) ^ (k & 4) plus ty ^ (k & 3), the second
    // part one of four per-thread offsets.  Shared-window byte addresses (32
    // bits) keep the four bases cheap.
    uint32_t pa[4];
#pragma unroll
    for (int x = 0; x < 4; ++x) pa[x] = smem_addr(sa + wm * 64 + ((ty ^ x) << 2));
    const uint32_t pb = smem_addr(sb + (wn * 64 + tx * 4));  // columns c * 32 + tx * 4 .. + 3
    float4 fa[2][4], fb[2][2];
    auto load = [&](int k, float4(&a)[4], float4(&b)[2]) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
            a[r] = lds128(pa[k & 3] + 4u * (k * BM + (((4 * r) ^ (k & 4)) << 2)));
        b[0] = lds128(pb + 4u * (k * MBN));
        b[1] = lds128(pb + 4u * (k * MBN + 32));
    };
    load(0, fa[0], fb[0]);
#pragma unroll
    for (int k = 0; k < MBK; ++k) {
        if (k + 1 < MBK) load(k + 1, fa[(k + 1) & 1], fb[(k + 1) & 1]);
        const float4(&a)[4] = fa[k & 1];
        const float4(&b)[2] = fb[k & 1];
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
}

// Float4 number e4 (0..31) of a thread's sums: row e4 / 2 of its sixteen,
// columns (e4 % 2) * 32 + tx * 4 .. + 3.  Called with e4 known after
// unrolling, the switch folds away and the sums stay in registers.
__device__ __forceinline__ float4 mid_f4(const MidAcc &acc, int e4) {
    switch (e4) {
#define SGEMM_MID_E4(E)                                                                     \
    case E:                                                                                 \
        return make_float4(acc.at((E) >> 1, ((E)&1) * 4 + 0), acc.at((E) >> 1, ((E)&1) * 4 + 1), \
                           acc.at((E) >> 1, ((E)&1) * 4 + 2), acc.at((E) >> 1, ((E)&1) * 4 + 3));
        SGEMM_MID_E4(0) SGEMM_MID_E4(1) SGEMM_MID_E4(2) SGEMM_MID_E4(3) SGEMM_MID_E4(4)
        SGEMM_MID_E4(5) SGEMM_MID_E4(6) SGEMM_MID_E4(7) SGEMM_MID_E4(8) SGEMM_MID_E4(9)
        SGEMM_MID_E4(10) SGEMM_MID_E4(11) SGEMM_MID_E4(12) SGEMM_MID_E4(13) SGEMM_MID_E4(14)
        SGEMM_MID_E4(15) SGEMM_MID_E4(16) SGEMM_MID_E4(17) SGEMM_MID_E4(18) SGEMM_MID_E4(19)
        SGEMM_MID_E4(20) SGEMM_MID_E4(21) SGEMM_MID_E4(22) SGEMM_MID_E4(23) SGEMM_MID_E4(24)
        SGEMM_MID_E4(25) SGEMM_MID_E4(26) SGEMM_MID_E4(27) SGEMM_MID_E4(28) SGEMM_MID_E4(29)
        SGEMM_MID_E4(30) SGEMM_MID_E4(31)
#undef SGEMM_MID_E4
    }
    return make_float4(0.f, 0.f, 0.f, 0.f);
}

// Tile coordinates of float4 e4 of thread t.
template <int BM>
__device__ __forceinline__ int mid_row(int t, int e4) {
    const int warp = t >> 5, wm = warp / MidCfg<BM>::WARPS_N, ty = (t & 31) >> 3;
    const int ri = e4 >> 1;  // r * 4 + i
    return wm * 64 + (ri >> 2) * 16 + ty * 4 + (ri & 3);
}
template <int BM>
__device__ __forceinline__ int mid_col(int t, int e4) {
    const int warp = t >> 5, wn = warp % MidCfg<BM>::WARPS_N, tx = t & 7;
    return wn * 64 + (e4 & 1) * 32 + tx * 4;
}

// C = alpha * s (+ beta C, epilogue) for columns n .. n+3 of row m.
__device__ __forceinline__ void mid_store4(const MidParams &p, int m, int n, float4 s) {
    if (m >= p.M) return;
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

__device__ __forceinline__ int mid_slot(const MidParams &p, int cta, int t_sk) {
    const int tile_start = t_sk * p.kt_total;
    const int k0 = max(cta * p.sk_share, tile_start) - tile_start;
    return 2 * cta + (k0 == 0 ? 1 : 0);
}

template <int BM, int BVEC>
__global__ void __launch_bounds__(MidCfg<BM>::NT, mid_ctas_per_sm(BM))
    sgemm_mid_kernel(const __grid_constant__ MidParams p) {
    using Cf = MidCfg<BM>;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    float *ring = reinterpret_cast<float *>(smem_raw);
    __shared__ int last_flag;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp / Cf::WARPS_N, wn = warp % Cf::WARPS_N;
    const int ty = lane >> 3, tx = lane & 7;
    const int G = gridDim.x, cta = blockIdx.x;

    MidRange rg;
    rg.n_dp = cta < p.dp_tiles ? (p.dp_tiles - 1 - cta) / G + 1 : 0;
    const int sk_total = p.sk_tiles * p.kt_total;
    rg.sk_begin = min(cta * p.sk_share, sk_total);
    rg.sk_end = min(rg.sk_begin + p.sk_share, sk_total);
    const int q_total = rg.n_dp * p.kt_total + (rg.sk_end - rg.sk_begin);

    int q = 0;
#pragma unroll 1
    while (q < q_total) {
        int tile, k0, k1, tm, tn;
        rg.unit_of(p, cta, G, q, tile, k0, k1);
        mid_tile_coords(p, tile, tm, tn);
        const int n = k1 - k0;
        q += n;

        // The unit's own copy pipeline.  The barrier keeps the previous
        // unit's last reads of the ring ahead of these copies.
        __syncthreads();
#pragma unroll
        for (int s = 0; s < MST - 1; ++s) {
            if (s < n) issue_slice<BM, BVEC>(p, ring + s * Cf::STAGE_FLOATS, tm, tn, k0 + s, tid);
            cp_async_commit();
        }
        MidAcc acc;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc.v[i][j] = make_float2(0.f, 0.f);

#pragma unroll 1
        for (int i = 0; i < n; ++i) {
            cp_async_wait<MST - 2>();  // this thread's copies of slice i are in
            __syncthreads();           // everyone's are; slice i - 1 is consumed
            if (i + MST - 1 < n)
                issue_slice<BM, BVEC>(p, ring + ((i + MST - 1) % MST) * Cf::STAGE_FLOATS, tm, tn,
                                      k0 + i + MST - 1, tid);
            cp_async_commit();
            compute_slice<BM>(ring + (i % MST) * Cf::STAGE_FLOATS, acc, wm, wn, ty, tx);
        }

        const int m0 = tm * BM, n0 = tn * MBN;
        // The thread's sums go to its own part of the idle ring (float4 e4
        // at e4 * NT + t, unrolled, straight from registers) and leave from
        // there in rolled loops: a rolled loop over the registers needs a
        // switch per float4 (2.6 us for a 64 x 128 tile in the split-K
        // kernel), and fully unrolled stores make long code that runs once.
        // No copy is in flight; the barrier waits for the last slice's reads.
        __syncthreads();
        float4 *own = reinterpret_cast<float4 *>(ring) + tid;
        static_assert(Cf::TILE_FLOATS <= Cf::RING_FLOATS, "a tile of sums fits the ring");
#pragma unroll
        for (int e4 = 0; e4 < Cf::E4; ++e4) own[e4 * Cf::NT] = mid_f4(acc, e4);
        if (k0 == 0 && k1 == p.kt_total) {
            // Whole tile: store.  (The next unit's barrier keeps these reads
            // ahead of its copies.)
#pragma unroll 1
            for (int e4 = 0; e4 < Cf::E4; ++e4)
                mid_store4(p, m0 + mid_row<BM>(tid, e4), n0 + mid_col<BM>(tid, e4), own[e4 * Cf::NT]);
            continue;
        }
        // Part of a stream-K tile: publish the piece (float4 e4 of thread t
        // at e4 * NT + t), take a ticket; the last CTA to arrive adds every
        // piece in CTA order.
        const int t_sk = tile - p.dp_tiles;
        float4 *slot = reinterpret_cast<float4 *>(p.partials +
                                                  (size_t)mid_slot(p, cta, t_sk) * Cf::TILE_FLOATS);
#pragma unroll 1
        for (int e4 = 0; e4 < Cf::E4; ++e4) __stcg(slot + e4 * Cf::NT + tid, own[e4 * Cf::NT]);
        __threadfence();
        __syncthreads();  // also: every thread is done with the ring
        const int c_first = (t_sk * p.kt_total) / p.sk_share;
        const int c_last = (t_sk * p.kt_total + p.kt_total - 1) / p.sk_share;
        if (tid == 0) {
            const int old = atomicAdd(&p.counters[t_sk], 1);
            last_flag = (old == c_last - c_first) ? 1 : 0;
        }
        __syncthreads();
        if (!last_flag) continue;
        __threadfence();
        // Copy (group g of piece c) goes to ring region idx % FIX_REGIONS,
        // idx = g * P + (c - c_first); three copies stay in flight.
        const int P = c_last - c_first + 1;
        const int total = Cf::FIX_GROUPS * P;
        auto issue_fix = [&](int idx) {
            if (idx < total) {
                const int g = idx / P, c = c_first + (idx - g * P);
                const float *src = p.partials + (size_t)mid_slot(p, c, t_sk) * Cf::TILE_FLOATS +
                                   ((size_t)g * Cf::FIX_E4 * Cf::NT + tid) * 4;
                float *dst = ring + (idx % Cf::FIX_REGIONS) * Cf::FIX_REGION + tid * 4;
#pragma unroll
                for (int e = 0; e < Cf::FIX_E4; ++e)
                    cp_async16(dst + e * Cf::NT * 4, src + (size_t)e * Cf::NT * 4, 16u);
            }
            cp_async_commit();
        };
        issue_fix(0);
        issue_fix(1);
        issue_fix(2);
        float4 sum[Cf::FIX_E4];
#pragma unroll 1
        for (int idx = 0; idx < total; ++idx) {
            issue_fix(idx + 3);
            cp_async_wait<3>();  // copy idx is in (each thread reads only its own)
            const int g = idx / P, ci = idx - g * P;
            const float *src = ring + (idx % Cf::FIX_REGIONS) * Cf::FIX_REGION + tid * 4;
#pragma unroll
            for (int e = 0; e < Cf::FIX_E4; ++e) {
                const float4 x = ld_shared_f4(src + e * Cf::NT * 4);
                if (ci == 0) {
                    sum[e] = x;
                } else {
                    sum[e].x += x.x;
                    sum[e].y += x.y;
                    sum[e].z += x.z;
                    sum[e].w += x.w;
                }
            }
            if (ci == P - 1) {
#pragma unroll
                for (int e = 0; e < Cf::FIX_E4; ++e) {
                    const int e4 = g * Cf::FIX_E4 + e;
                    mid_store4(p, m0 + mid_row<BM>(tid, e4), n0 + mid_col<BM>(tid, e4), sum[e]);
                }
            }
        }
        if (tid == 0) p.counters[t_sk] = 0;
    }
    cp_async_wait<0>();  // no copy may land after the CTA has exited
}

template <int BM, int BVEC>
cudaError_t launch_impl(const MidParams &p, int grid, cudaStream_t stream) {
    sgemm_mid_kernel<BM, BVEC><<<grid, MidCfg<BM>::NT, MidCfg<BM>::smem_bytes, stream>>>(p);
    return cudaGetLastError();
}

template <int BM, int BVEC>
cudaError_t configure_impl() {
    cudaError_t e = cudaFuncSetAttribute(sgemm_mid_kernel<BM, BVEC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)MidCfg<BM>::smem_bytes);
    // No carveout preference: the driver's choice leaves L1 more room than
    // the largest shared-memory carveout, and A's 4-byte copies
    // (cp.async.ca) pass through L1 (3000 x 300 x 5000 219.1 -> 215.0-215.8 us).
    return e;
}

// The instantiated forms: (tile rows, B copy width).
#define SGEMM_MID_FORMS(X) X(128, 4) X(128, 1) X(64, 4) X(64, 1)

}  // namespace

cudaError_t launch_mid(int bm, int b_vec, const MidParams &p, int grid, cudaStream_t stream) {
#define SGEMM_MID_LAUNCH(BM, BV) \
    if (bm == BM && b_vec == BV) return launch_impl<BM, BV>(p, grid, stream);
    SGEMM_MID_FORMS(SGEMM_MID_LAUNCH)
#undef SGEMM_MID_LAUNCH
    return cudaErrorInvalidValue;
}

cudaError_t mid_configure(int bm, int b_vec) {
#define SGEMM_MID_CONF(BM, BV) \
    if (bm == BM && b_vec == BV) return configure_impl<BM, BV>();
    SGEMM_MID_FORMS(SGEMM_MID_CONF)
#undef SGEMM_MID_CONF
    return cudaErrorInvalidValue;
}

}  // namespace sgemm
