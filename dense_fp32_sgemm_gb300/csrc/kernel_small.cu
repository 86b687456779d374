// Small-product SIMT FP32 GEMM for sm_103a: C = alpha * A * B + beta * C,
// row-major, for products so small that the time is the launch, the first
// copies and the store (128^3 is 2 M multiply-adds: 0.1 us of the GPU's FP32
// rate).
//
// "Optimizing Matrix Multiply on CUDA, Part 1", section "Small and Odd
// Sizes": a small product gives few tiles, so small tiles spread it over more
// SMs; "Part 2", section "Selecting Among Three Kernels": a split-K variant
// gives more SMs work when there are few tiles.  Here one CTA of 256 threads
// owns a 32 x 32 tile and splits K inside itself: four groups of 64 threads
// each take a quarter of every 64-k slice with a 4 x 4 micro-tile of the
// whole tile per thread, and add their sums in shared memory in group order.
// A 3-stage cp.async ring (16 KiB a slice, so that four CTAs fit an SM)
// brings A in 4-byte copies straight to a k-major tile (the 16-byte chunk of
// row k XOR-ed with k mod 8: the eight k of a copied 32-byte sector land in
// eight bank groups) and B in 16- or 4-byte copies, zero-filled outside the
// matrices, so any alignment works.  In the last slice a group multiplies
// only the k that exist.  The only waits are on the CTA's own copies and
// barriers; the sums are added in a fixed order.

#include "device_common.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

constexpr int SM_ = kSmallBM;   // tile rows
constexpr int SN = kSmallBN;    // tile columns
constexpr int SK = kSmallBK;    // k per slice
constexpr int SST = kSmallStages;
constexpr int SNT = 256;
constexpr int SKG = 4;                       // k-groups
constexpr int SGK = SK / SKG;                // k of a slice per group: 16
constexpr int A_FL = SK * SM_;               // k-major A slice
constexpr int B_FL = SK * SN;
constexpr int STAGE_FL = A_FL + B_FL;
constexpr int TILE = SM_ * SN;
static_assert(SM_ == 32 && SN == 32 && SK == 64, "the copy and fragment maps");
static_assert(SKG * 64 == SNT && TILE / 16 == 64, "a group of 64 threads of 4 x 4 covers the tile");
static_assert(SKG * TILE <= SST * STAGE_FL, "the groups' sums fit the idle ring");

__device__ __forceinline__ int sm_a_off(int m, int k) {
    return k * SM_ + (((m >> 2) ^ (k & 7)) << 2) + (m & 3);
}

// Copies of k-slice ks of tile (tm, tn) into stage `st`.
template <int BVEC>
__device__ __forceinline__ void small_issue(const MidParams &p, float *st, int tm, int tn, int ks,
                                            int tid) {
    float *sa = st;
    float *sb = st + A_FL;
    const int k_base = ks * SK;
    // A: thread t copies k = t % 32 (+ 32 h) of rows t / 32 + 8 j (j < 4):
    // a warp copies 32 consecutive k of one row.
#pragma unroll
    for (int h = 0; h < SK / 32; ++h) {
        const int kin = (tid & 31) + 32 * h;
        const int m_in = tid >> 5;
        const int gm0 = tm * SM_ + m_in;
        const bool k_ok = k_base + kin < p.K;
        const float *src = p.A + (long long)gm0 * p.lda + k_base + kin;
#pragma unroll
        for (int j = 0; j < SM_ / 8; ++j) {
            const bool ok = k_ok && gm0 + 8 * j < p.M;
            cp_async4(sa + sm_a_off(m_in + 8 * j, kin), ok ? src : p.A, ok ? 4u : 0u);
            src += 8LL * p.lda;
        }
    }
    const int n_base = tn * SN;
    if (BVEC == 4) {
        // 512 chunks of 16 bytes, 8 to a row: chunk t + 256 q is row
        // t / 8 + 32 q, columns 4 (t % 8) .. + 3.
        const int n4 = (tid & 7) * 4;
        const int cols = min(4, p.N - (n_base + n4));
        const int kin0 = tid >> 3;
#pragma unroll
        for (int q = 0; q < SK * SN / 4 / SNT; ++q) {
            const int kin = kin0 + 32 * q;
            const bool ok = k_base + kin < p.K && cols > 0;
            cp_async16(sb + kin * SN + n4, ok ? p.B + (long long)(k_base + kin) * p.ldb + n_base + n4
                                              : p.B,
                       ok ? uint32_t(cols) * 4u : 0u);
        }
    } else {
        // 2048 elements: element t + 256 q is row t / 32 + 8 q, column t % 32.
        const int n = tid & 31;
        const bool n_ok = n_base + n < p.N;
        const int kin0 = tid >> 5;
#pragma unroll
        for (int q = 0; q < SK * SN / SNT; ++q) {
            const int kin = kin0 + 8 * q;
            const bool ok = n_ok && k_base + kin < p.K;
            cp_async4(sb + kin * SN + n, ok ? p.B + (long long)(k_base + kin) * p.ldb + n_base + n : p.B,
                      ok ? 4u : 0u);
        }
    }
}

// C = alpha * s (+ beta C, epilogue) for columns n .. n+3 of row m.
__device__ __forceinline__ void small_store4(const MidParams &p, int m, int n, float4 s) {
    if (m >= p.M || n >= p.N) return;
    float *crow = p.C + (long long)m * p.ldc;
    const float o[4] = {p.alpha * s.x, p.alpha * s.y, p.alpha * s.z, p.alpha * s.w};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        if (n + jj < p.N) {
            float v = o[jj];
            if (p.beta != 0.0f) v = __fmaf_rn(p.beta, crow[n + jj], v);
            crow[n + jj] = apply_epilogue(v, p.epi, n + jj);
        }
    }
}

template <int BVEC>
__global__ void __launch_bounds__(SNT, 4) sgemm_small_kernel(const __grid_constant__ MidParams p) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    float *ring = reinterpret_cast<float *>(smem_raw);
    const int tid = threadIdx.x;
    const int grp = tid >> 6, gt = tid & 63;
    const int ty = gt >> 3, tx = gt & 7;  // rows ty * 4 .. + 3, columns tx * 4 .. + 3
    const int tm = blockIdx.x / p.tiles_n, tn = blockIdx.x - (blockIdx.x / p.tiles_n) * p.tiles_n;
    const int n_slices = p.kt_total;

#pragma unroll
    for (int s = 0; s < SST - 1; ++s) {
        if (s < n_slices) small_issue<BVEC>(p, ring + s * STAGE_FL, tm, tn, s, tid);
        cp_async_commit();
    }
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    const int k_grp = grp * SGK;
    const int full = p.K / SK;
    const int k_last = p.K - full * SK - k_grp;
    const int kc_last = k_last < 0 ? 0 : (k_last > SGK ? SGK : k_last);

#pragma unroll 1
    for (int i = 0; i < n_slices; ++i) {
        cp_async_wait<SST - 2>();  // this thread's copies of slice i are in
        __syncthreads();           // everyone's are; slice i - 1 is consumed
        if (i + SST - 1 < n_slices)
            small_issue<BVEC>(p, ring + ((i + SST - 1) % SST) * STAGE_FL, tm, tn, i + SST - 1, tid);
        cp_async_commit();
        const float *sa = ring + (i % SST) * STAGE_FL;
        const float *sb = sa + A_FL;
        const int kc = i < full ? SGK : kc_last;
#pragma unroll 4
        for (int k = 0; k < kc; ++k) {
            const int kk = k_grp + k;
            const float4 a = ld_shared_f4(sa + kk * SM_ + ((ty ^ (kk & 7)) << 2));
            const float4 b = ld_shared_f4(sb + kk * SN + tx * 4);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = __fmaf_rn(av[r], bv[c], acc[r][c]);
        }
    }
    cp_async_wait<0>();
    __syncthreads();  // every group is done with the ring

    // The groups' sums at S[g][row][col]; thread t then adds float4 t of the
    // tile (row t / 8, columns 4 (t % 8) ..) over the groups in group order.
    float *S = ring;
#pragma unroll
    for (int r = 0; r < 4; ++r)
        st_shared_f4(S + grp * TILE + (ty * 4 + r) * SN + tx * 4,
                     make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]));
    __syncthreads();
    const int row = tid >> 3, c4 = (tid & 7) * 4;
    float4 s = ld_shared_f4(S + row * SN + c4);
#pragma unroll
    for (int g = 1; g < SKG; ++g) {
        const float4 x = ld_shared_f4(S + g * TILE + row * SN + c4);
        s.x += x.x;
        s.y += x.y;
        s.z += x.z;
        s.w += x.w;
    }
    small_store4(p, tm * SM_ + row, tn * SN + c4, s);
}

constexpr size_t SMALL_SMEM = size_t(SST) * STAGE_FL * 4;

template <int BVEC>
cudaError_t launch_impl(const MidParams &p, int grid, cudaStream_t stream) {
    sgemm_small_kernel<BVEC><<<grid, SNT, SMALL_SMEM, stream>>>(p);
    return cudaGetLastError();
}

template <int BVEC>
cudaError_t configure_impl() {
    return cudaFuncSetAttribute(sgemm_small_kernel<BVEC>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMALL_SMEM);
}

}  // namespace

cudaError_t launch_small(int b_vec, const MidParams &p, int grid, cudaStream_t stream) {
    if (b_vec == 4) return launch_impl<4>(p, grid, stream);
    if (b_vec == 1) return launch_impl<1>(p, grid, stream);
    return cudaErrorInvalidValue;
}

cudaError_t small_configure(int b_vec) {
    if (b_vec == 4) return configure_impl<4>();
    if (b_vec == 1) return configure_impl<1>();
    return cudaErrorInvalidValue;
}

}  // namespace sgemm
