// Parameter block and launch wrappers of the 3xTF32 tensor-core variant,
// shared by the host entry point (api.cu) and kernel_3xtf32.cu.  Host-visible
// only: no device code here.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"  // Epilogue

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
constexpr int kX3MaxSplits = 8;  // K ranges per tile (deep products with few tiles)

// Tile width and K split for an M x N x (kt_total K slices) product on
// num_sms SMs (one tile and K range per CTA, one CTA per SM).  Cost of a
// choice, in units of one K slice of one tile column (about 1.75 ns on
// GB300): whole waves x (width + 32, the A tile every CTA loads whatever its
// width) x (slices per split + 8, a tile's fill and epilogue), plus for a
// split the extra launch and the bytes its reduction moves.  Widths are the
// multiples of 16 in [64, 256]; a split keeps at least 16 slices per range.
// Ties go to the wider tile, then to fewer splits.  forced_splits > 0 fixes
// the split count (the nearest feasible one).
inline void x3_plan(long long M, long long N, int kt_total, int num_sms, int forced_splits,
                    int *bn_out, int *splits_out) {
    int best_bn = kX3BN, best_s = 1;
    double best = -1.0;
    for (int bn = kX3BN; bn >= kX3MinBN; bn -= 16) {
        const long long tiles = ((M + kX3BM - 1) / kX3BM) * ((N + bn - 1) / bn);
        for (int sp = 1; sp <= kX3MaxSplits; ++sp) {
            const int kps = (kt_total + sp - 1) / sp;
            if (sp > 1 && (kps < 16 || (long long)(sp - 1) * kps >= kt_total)) continue;
            if (forced_splits > 0 && sp != forced_splits && !(sp == 1 && forced_splits == 1))
                continue;
            const long long rounds = (tiles * sp + num_sms - 1) / num_sms;
            double cost = (double)rounds * (bn + 32) * (kps + 8);
            if (sp > 1) cost += 1700.0 + (double)(sp + 2) * (double)M * (double)N / 2625.0;
            if (best < 0 || cost < best) {
                best = cost;
                best_bn = bn;
                best_s = sp;
            }
        }
    }
    if (best < 0) {  // the forced split count is not feasible for this K
        x3_plan(M, N, kt_total, num_sms, 0, bn_out, splits_out);
        return;
    }
    *bn_out = best_bn;
    *splits_out = best_s;
}

struct X3Params {
    int M, N, K;
    int bn;                // tile width: a multiple of 16 in [64, 256]
    int tiles_m, tiles_n;
    int kt_total;          // ceil(K / BK)
    int splits;            // K ranges per tile; CTA blockIdx / tiles takes range
    int kt_per_split;      //   [split * kt_per_split, + kt_per_split) of the slices
    float *part;           // splits > 1: raw sums, slice s at part + s * part_stride
    long long part_stride; //   (floats), row m of a slice at m * part_ld
    long long part_ld;
    int a_lo_row;          // Mp: first row of A's lo part in the split buffer
    int b_lo_row;          // Np: first row of B's lo part
    float alpha, beta;
    float *C;
    long long ldc;
    int c_tma;             // mapC covers C (16-byte aligned, ldc a multiple of 4)
    Epilogue epi;          // bias / activation after alpha and beta (none for K splits)
    int *err;
    unsigned long long timeout_ns;
    int skip_loads_from;   // testing hook, -1 = off
};

// Kernel forms (bk = K slice, stages = ring depth): 16 x 4 and 32 x 2 run
// one CTA per SM; 16 x 2 runs two CTAs per SM.
// a_raw: mapA covers A itself (FP32, M x K) and the kernel splits each A
// tile in shared memory; otherwise mapA covers the split pass's A buffer.
// mapC: C as M x N FP32, 32 x 32 boxes, used when beta != 0 and p.c_tma (one
// CTA per SM forms only; the two-CTA form reads C directly).
bool x3_form_valid(int bk, int stages);
cudaError_t x3_configure(int bk, int stages, bool a_raw);
cudaError_t launch_x3(int bk, int stages, bool a_raw, const CUtensorMap &mapA,
                      const CUtensorMap &mapB, const CUtensorMap &mapC, const X3Params &p,
                      cudaStream_t stream);
// C = act(alpha * (part[0] + ... + part[splits - 1]) + beta * C + bias), the
// slices added in order (deterministic).
cudaError_t launch_x3_reduce(const float *part, int splits, long long stride, long long ld_part,
                             int M, int N, float alpha, float beta, float *C, long long ldc,
                             const Epilogue &epi, int num_sms, cudaStream_t stream);
// Split A (M x K, lda; skipped when A is null) and B (K x N, ldb) into the
// buffers above.  Kp is a multiple of 4; Mp and Np multiples of the tile
// sizes.
cudaError_t launch_x3_split(const float *A, long long lda, int M, const float *B, long long ldb,
                            int N, int K, float *splitA, int Mp, float *splitB, int Np, int Kp,
                            int num_sms, cudaStream_t stream);

// Rate probe of tcgen05.mma kind::tf32 (M 128, N 256, K 8): `blocks` CTAs, one
// per SM, each issuing iters * 4 MMAs; 2^21 * iters * blocks flops per launch.
// A bounded wait that gives up sets `err`.
cudaError_t tf32_probe_configure();
cudaError_t launch_tf32_probe(long long iters, int blocks, int *err, unsigned long long timeout_ns,
                              cudaStream_t stream);

}  // namespace sgemm
