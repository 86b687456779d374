// Kernel parameter blocks and launch wrappers shared by the host planner
// (api.cu) and the kernel translation units.  Host-visible only: no device
// code here.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sgemm {

// ---------------------------------------------------------------------------
// Epilogue applied by every kernel after alpha * acc + beta * c: a bias per
// column of C, then an activation.
// ---------------------------------------------------------------------------
enum : int { kActNone = 0, kActRelu = 1 };

struct Epilogue {
    const float *bias;  // N floats, or nullptr
    int act;            // kActNone or kActRelu
};

// ---------------------------------------------------------------------------
// Tiled FFMA kernel (TMA + mbarrier pipeline, in-CTA transposed A tile).
// Block tile BM x BN = 128 x 256, K slice BK = 32; each thread a TM x 8
// micro-tile.
// ---------------------------------------------------------------------------
constexpr int kTileBM = 128;
constexpr int kTileBN = 256;
constexpr int kTileBK = 32;

// Inner-product form of the micro-tile update (see kernel_tile.cu).
enum FmaMode : int {
    kFmaScalar = 0,    // one FFMA per product
    kFmaPairMovA = 1,  // packed pairs along n, A value duplicated in registers
    kFmaPairDupA = 2,  // packed pairs along n, A stored duplicated in shared memory
    kFmaPairMovB = 3,  // packed pairs along m, B value duplicated in registers
};

struct TileParams {
    int M, N, K;
    int tiles_m, tiles_n;
    int kt_total;       // ceil(K / BK): k-iterations of a whole tile
    int dp_tiles;       // tiles [0, dp_tiles) are computed whole, round-robin
    int sk_tiles;       // tiles [dp_tiles, dp_tiles + sk_tiles) are stream-K
    int sk_share;       // k-iterations each CTA takes in the stream-K region
    int group_m;        // tile rasterisation: tiles_m grouped by this many rows
    float alpha, beta;
    float *C;
    long long ldc;
    int c_vec4;         // C and ldc allow 16-byte accesses
    Epilogue epi;
    float *partials;    // 2 * gridDim.x slots of BM*BN floats (stream-K)
    int *counters;      // one arrival counter per stream-K tile, zero at rest
    int *err;           // device error word
    unsigned long long timeout_ns;
    int skip_loads_from;  // testing hook, -1 = off
};

// tm: micro-tile rows, 16 (256 threads, 2 warps per scheduler) or 8 (512
// threads, 4 warps per scheduler); both cover the 128 x 256 tile.
cudaError_t launch_tile(int fma_mode, int stages, int tm, const CUtensorMap &mapA,
                        const CUtensorMap &mapB, const TileParams &p, int grid,
                        cudaStream_t stream);
size_t tile_smem_bytes(int fma_mode, int stages, int tm);
cudaError_t tile_configure(int fma_mode, int stages, int tm);
int tile_threads(int tm);

// ---------------------------------------------------------------------------
// Generic kernel: any alignment and leading dimension, bounds-checked loads.
// ---------------------------------------------------------------------------
constexpr int kGenBM = 64;
constexpr int kGenBN = 64;
constexpr int kGenBK = 16;

struct GenericParams {
    int M, N, K;
    float alpha, beta;
    const float *A;
    long long lda;
    const float *B;
    long long ldb;
    float *C;
    long long ldc;
    Epilogue epi;
};

cudaError_t launch_generic(const GenericParams &p, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Mid-size kernel: BM x 128 tiles (BM = 128 or 64) fed by cp.async copies of
// 4 bytes (A, and B when it is not 16-byte aligned) or 16 bytes (aligned B),
// so any alignment and leading dimension works without a copy pass; A lands
// k-major with an XOR swizzle; 8 x 8 micro-tiles on packed FFMA2; 2 * BM
// threads, several CTAs per SM; data-parallel tiles, then a stream-K tail
// with the same deterministic fix-up as the tiled kernel.
// ---------------------------------------------------------------------------
constexpr int kMidBN = 128;
constexpr int kMidBK = 16;
constexpr int kMidStages = 4;

struct MidParams {
    int M, N, K;
    int tiles_m, tiles_n;
    int kt_total;       // ceil(K / kMidBK)
    int dp_tiles, sk_tiles, sk_share;
    int group_m;
    float alpha, beta;
    const float *A;
    long long lda;
    const float *B;
    long long ldb;
    float *C;
    long long ldc;
    int c_vec4;
    Epilogue epi;
    float *partials;    // 2 * gridDim.x slots of BM * 128 floats (stream-K)
    int *counters;      // one per stream-K tile, zero at rest
};

// bm: 128 or 64; b_vec: 4 (B 16-byte aligned, ldb % 4 == 0) or 1.
cudaError_t launch_mid(int bm, int b_vec, const MidParams &p, int grid, cudaStream_t stream);
cudaError_t mid_configure(int bm, int b_vec);
constexpr int mid_ctas_per_sm(int bm) { return bm == 64 ? 4 : 2; }

// ---------------------------------------------------------------------------
// Split-K-in-CTA kernel: one CTA of 256 threads per 64 x BN tile (BN = 128:
// four groups of 64 threads; BN = 64: eight groups of one warp); group g
// takes the g-th part of every kKsBK-k slice and keeps a 16 x 8 micro-tile
// of sums of the whole tile per thread; the groups' sums are added in
// shared memory in group order.  Copies as in the mid-size kernel (cp.async
// of 4 or 16 bytes, any alignment), a ring of kKsStages slices.
// Data-parallel: one tile per CTA, one CTA per SM.  Takes MidParams
// (tiles_m, tiles_n, kt_total = ceil(K / kKsBK), group_m; the stream-K
// fields are unused).
// ---------------------------------------------------------------------------
constexpr int kKsBM = 64;
constexpr int kKsBK = 64;
constexpr int kKsStages = 4;
constexpr int kKsThreads = 256;

// b_vec: 4 (B 16-byte aligned, ldb % 4 == 0) or 1; bn: 128 or 64.
cudaError_t launch_ksplit(int b_vec, int bn, const MidParams &p, int grid, cudaStream_t stream);
cudaError_t ksplit_configure(int b_vec, int bn);

// ---------------------------------------------------------------------------
// Narrow kernel: N <= kNarrowMaxN columns (also the last few columns of C
// beside the tiled kernel).  A warp per row of A, lanes over K; B's columns
// staged transposed in shared memory in chunks of kch k (a multiple of 128;
// all of K when nn * (kch + 4) floats fit kNarrowSmemBytes); CTAs own
// contiguous ranges of rows_per_cta rows.  nn: columns the kernel is built
// for (1, 2 or 4, at least N); a_vec: 4 when A's rows are 16-byte aligned.
// The bias of the epilogue is indexed from the first column of C passed.
// ---------------------------------------------------------------------------
constexpr int kNarrowMaxN = 4;
constexpr size_t kNarrowSmemBytes = 96 * 1024;  // two CTAs per SM fit with it
// Chunk of K staged at once for nn columns.
constexpr int narrow_kch(long long K, int nn) {
    const long long fit = ((long long)kNarrowSmemBytes / 4 / nn - 4) / 128 * 128;
    const long long want = (K + 127) / 128 * 128;
    return (int)(want < fit ? want : fit);
}

struct NarrowParams {
    int M, N, K;
    float alpha, beta;
    const float *A;
    long long lda;
    const float *B;
    long long ldb;
    float *C;
    long long ldc;
    Epilogue epi;
    int rows_per_cta;
    int kch;  // narrow_kch(K, nn)
};

cudaError_t launch_narrow(int nn, int a_vec, const NarrowParams &p, int grid, cudaStream_t stream);
// Lets the form (nn, a_vec) use kNarrowSmemBytes of dynamic shared memory.
cudaError_t narrow_configure(int nn, int a_vec);

// ---------------------------------------------------------------------------
// Small-product kernel: one CTA of 256 threads per 32 x 32 tile, four groups
// of 64 threads each taking a quarter of every kSmallBK-k slice (4 x 4 sums
// per thread), sums added in shared memory in group order; a 3-stage cp.async
// ring of 16 KiB slices, up to four CTAs per SM.  Takes MidParams (tiles_m,
// tiles_n, kt_total = ceil(K / kSmallBK); tile t is row t / tiles_n, column
// t % tiles_n).
// ---------------------------------------------------------------------------
constexpr int kSmallBM = 32;
constexpr int kSmallBN = 32;
constexpr int kSmallBK = 64;
constexpr int kSmallStages = 3;
constexpr int kSmallCtasPerSm = 4;

cudaError_t launch_small(int b_vec, const MidParams &p, int grid, cudaStream_t stream);
cudaError_t small_configure(int b_vec);

// Copies of operands the TMA cannot map: rows x cols at src (leading
// dimension ld, any 4-byte alignment) to dst with 16-byte-aligned rows of
// ldp floats (ldp a multiple of 4, dst 16-byte aligned).  Up to two copies in
// one launch.
struct PackJob {
    const float *src;
    long long ld;
    int rows, cols;
    float *dst;
    long long ldp;
};
// Grids are capped at a few CTAs per SM of the device (num_sms).
cudaError_t launch_pack(const PackJob *jobs, int njobs, int num_sms, cudaStream_t stream);

// C = act(beta * C + bias) (beta == 0 does not read C).
cudaError_t launch_scale(int M, int N, float beta, float *C, long long ldc, const Epilogue &epi,
                         int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Skinny-M kernel (M <= 32): streams B once through a TMA ring together with
// the matching 32-column slices of A (128-byte swizzled), stream-K over
// (column slab, k) with a fixed-order reduction.  The A tensor map must use
// CU_TENSOR_MAP_SWIZZLE_128B.
// ---------------------------------------------------------------------------
constexpr int kSkinnyBN = 256;   // columns per slab
constexpr int kSkinnyBK = 32;    // B rows per TMA stage
constexpr int kSkinnyMaxM = 32;  // rows of C the kernel covers (tiles of 8, 16 or 32 rows)
// Warps per CTA: 8 (one CTA per SM, 6 ring stages) or 4 (two CTAs per SM, 3
// stages each).  A build constant so that both can be timed; 8 measured
// faster on GB300 (its warps share one ring, so no CTA of an SM falls behind
// the other).
#ifndef SGEMM_SKINNY_WARPS
#define SGEMM_SKINNY_WARPS 8
#endif
constexpr int kSkinnyWarps = SGEMM_SKINNY_WARPS;
static_assert(kSkinnyWarps == 4 || kSkinnyWarps == 8, "skinny kernel: 4 or 8 warps");
constexpr int kSkinnyThreads = 32 * kSkinnyWarps;
constexpr int kSkinnyCtasPerSm = kSkinnyWarps == 4 ? 2 : 1;
constexpr int kSkinnyStages = kSkinnyWarps == 4 ? 3 : 6;
// Ring stages of the kernel with an m_tile-row A tile: the 32-row tile's
// stages are 36 KiB, five of them fit beside the reduction buffers.
constexpr int skinny_stages(int m_tile) { return m_tile == 32 ? 5 : kSkinnyStages; }

constexpr int kSkinnyMaxGrid = 160;  // CTAs a skinny launch may use
// A unit end in the middle of a CTA's range (a reduction over the warps, a
// partial written and a ticket taken while the ring keeps streaming) costs
// about this many positions of streaming time on GB300; the planner shortens
// such ranges by it.  (Measured 16 x 8192 x 8192, CUDA events: 3 -> 59.5 us,
// 4 -> 59.4, 5 -> 57.8, 6 -> 57.5, 8 -> 59.4.)
constexpr int kSkinnyUnitEndCost = 6;

struct SkinnyParams {
    int M, N, K;
    int slabs;            // ceil(N / BN)
    int kt_total;         // ceil(K / BK)
    // CTA c takes positions [starts[c], starts[c + 1]) of the (slab, k) plane
    // (position u is slab u / kt_total, k-step u % kt_total); starts[grid] is
    // slabs * kt_total.
    int starts[kSkinnyMaxGrid + 1];
    float alpha, beta;
    const float *A;
    long long lda;
    float *C;
    long long ldc;
    int c_vec4;
    Epilogue epi;
    float *partials;      // 2 * gridDim.x slots of m_tile * BN floats
    int *counters;        // one per slab
    int *err;
    unsigned long long timeout_ns;
    int skip_loads_from;
};

cudaError_t launch_skinny(int m_tile, const CUtensorMap &mapA, const CUtensorMap &mapB,
                          const SkinnyParams &p, int grid, cudaStream_t stream);
size_t skinny_smem_bytes(int m_tile, int share);
cudaError_t skinny_configure(int m_tile);

// ---------------------------------------------------------------------------
// Testing hooks set through sgemm_set_wait_timeout_ns (api.cu): the limit of
// every bounded device wait (the default, one second, when none is set) and
// the k-iteration of each CTA from which copy producers stop issuing loads
// (-1 = never).
// ---------------------------------------------------------------------------
void wait_hooks(unsigned long long *timeout_ns, int *skip_loads_from);

// ---------------------------------------------------------------------------
// Measurement probes (same library, used by the benchmark).
// ---------------------------------------------------------------------------
cudaError_t launch_ffma_probe(int paired, long long iters, int blocks, float *sink,
                              cudaStream_t stream);
cudaError_t launch_read_probe(const float4 *buf, long long n4, float *sink, int blocks,
                              cudaStream_t stream);
cudaError_t launch_hold(unsigned long long ns, cudaStream_t stream);

}  // namespace sgemm
