// Parameter block and launch wrappers of the 3xTF32 tensor-core variant,
// shared by the host entry point (api.cu) and kernel_3xtf32.cu.  Host-visible
// only: no device code here.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace sgemm {

// ---------------------------------------------------------------------------
// 3xTF32 variant on the tensor cores (tcgen05, accumulator in tensor memory).
// A split pass writes each operand as TF32 hi and lo parts, K-major, zero
// padded: A as (2 * Mp) x Kp rows (hi rows [0, Mp), lo rows [Mp, 2 Mp)), B
// transposed as (2 * Np) x Kp rows.  The MMA kernel takes one 128 x bn tile
// of C per CTA and sums hi*hi + hi*lo + lo*hi over K.
// ---------------------------------------------------------------------------
constexpr int kX3BM = 128;
constexpr int kX3BN = 256;
constexpr int kX3MinK = 64;  // shorter products run the FFMA kernels
constexpr int kX3MinBN = 64;  // narrowest tile (small products fill more SMs)

// Tile width for an M x N product on num_sms SMs (one tile per CTA, one CTA
// per SM): the multiple of 16 in [64, 256] whose whole number of waves
// costs least, a wave costing its width plus 32 (the A tile every CTA loads
// whatever its width); ties go to the wider tile.
inline int x3_tile_width(long long M, long long N, int num_sms) {
    int best = kX3BN;
    long long best_cost = -1;
    for (int bn = kX3BN; bn >= kX3MinBN; bn -= 16) {
        const long long tiles = ((M + kX3BM - 1) / kX3BM) * ((N + bn - 1) / bn);
        const long long cost = ((tiles + num_sms - 1) / num_sms) * (bn + 32);
        if (best_cost < 0 || cost < best_cost) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

struct X3Params {
    int M, N, K;
    int bn;                // tile width: a multiple of 16 in [64, 256]
    int tiles_m, tiles_n;
    int kt_total;          // ceil(K / BK)
    int a_lo_row;          // Mp: first row of A's lo part in the split buffer
    int b_lo_row;          // Np: first row of B's lo part
    float alpha, beta;
    float *C;
    long long ldc;
    int c_tma;             // mapC covers C (16-byte aligned, ldc a multiple of 4)
    int *err;
    unsigned long long timeout_ns;
    int skip_loads_from;   // testing hook, -1 = off
};

// bk: 32 (128-byte swizzled rows) or 16 (64-byte swizzled rows).
// a_raw: mapA covers A itself (FP32, M x K) and the kernel splits each A
// tile in shared memory; otherwise mapA covers the split pass's A buffer.
int x3_stages(int bk);
size_t x3_smem_bytes(int bk);
cudaError_t x3_configure(int bk, bool a_raw);
// mapC: C as M x N FP32, 32 x 32 boxes, used when beta != 0 and p.c_tma.
cudaError_t launch_x3(int bk, bool a_raw, const CUtensorMap &mapA, const CUtensorMap &mapB,
                      const CUtensorMap &mapC, const X3Params &p, cudaStream_t stream);
// Split A (M x K, lda; skipped when A is null) and B (K x N, ldb) into the
// buffers above.  Kp is a multiple of 4; Mp and Np multiples of the tile
// sizes.
cudaError_t launch_x3_split(const float *A, long long lda, int M, const float *B, long long ldb,
                            int N, int K, float *splitA, int Mp, float *splitB, int Np, int Kp,
                            int num_sms, cudaStream_t stream);

}  // namespace sgemm
