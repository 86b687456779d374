// Generic FP32 GEMM for operands the TMA path cannot map (pointers or leading
// dimensions that break 16-byte alignment, or products too small for the
// tiled kernel), the C = beta * C kernel for the alpha == 0 / K == 0 quick
// return, and the copy of unaligned operands to aligned rows that lets larger
// products take the tiled kernel.
//
// 64 x 64 block tile, K slice 16, 256 threads with a 4 x 4 micro-tile each
// ("Optimizing Matrix Multiply on CUDA, Part 1", section "Stage 3: Register
// Tiling": the outer product per k from a shared-memory tile).  Loads are
// scalar and bounds-checked, so any alignment and any leading dimension work;
// out-of-range elements are loaded as zero ("Part 1", section "Small and Odd
// Sizes": lanes outside the matrix supply zeros).  The next slice is fetched
// into registers while the current one is consumed.

#include "device_common.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

constexpr int GBM = kGenBM, GBN = kGenBN, GBK = kGenBK;
constexpr int GNT = 256;
constexpr int APAD = 4;  // keeps 16-byte rows, staggers banks of the k-major A tile

__global__ void __launch_bounds__(GNT) sgemm_generic_kernel(const GenericParams p) {
    __shared__ __align__(16) float As[GBK][GBM + APAD];
    __shared__ __align__(16) float Bs[GBK][GBN];

    const int tid = threadIdx.x;
    const int ty = tid >> 4, tx = tid & 15;
    const int m0 = blockIdx.y * GBM, n0 = blockIdx.x * GBN;

    // Each thread copies 4 elements of each slice: element e = tid + 256*q.
    float ra[4], rb[4];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = tid + GNT * q;
            const int am = e / GBK, ak = e % GBK;  // A slice: 64 rows x 16 k
            const int gm = m0 + am, gk = k0 + ak;
            ra[q] = (gm < p.M && gk < p.K) ? p.A[(long long)gm * p.lda + gk] : 0.0f;
            const int bk = e / GBN, bn = e % GBN;  // B slice: 16 k x 64 columns
            const int gk2 = k0 + bk, gn = n0 + bn;
            rb[q] = (gk2 < p.K && gn < p.N) ? p.B[(long long)gk2 * p.ldb + gn] : 0.0f;
        }
    };
    auto stash = [&]() {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = tid + GNT * q;
            As[e % GBK][e / GBK] = ra[q];
            Bs[e / GBN][e % GBN] = rb[q];
        }
    };

    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    fetch(0);
    for (int k0 = 0; k0 < p.K; k0 += GBK) {
        __syncthreads();
        stash();
        __syncthreads();
        if (k0 + GBK < p.K) fetch(k0 + GBK);
#pragma unroll
        for (int k = 0; k < GBK; ++k) {
            const float4 a = *reinterpret_cast<const float4 *>(&As[k][ty * 4]);
            const float4 b = *reinterpret_cast<const float4 *>(&Bs[k][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
        }
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= p.M) continue;
        float *crow = p.C + (long long)m * p.ldc;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= p.N) continue;
            float o = p.alpha * acc[i][j];
            if (p.beta != 0.0f) o = __fmaf_rn(p.beta, crow[n], o);
            crow[n] = apply_epilogue(o, p.epi, n);
        }
    }
}

__global__ void sgemm_scale_kernel(int M, int N, float beta, float *C, long long ldc,
                                   const Epilogue epi) {
    const long long total = (long long)M * N;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long m = e / N, n = e - m * N;
        float *c = C + m * ldc + n;
        *c = apply_epilogue((beta == 0.0f) ? 0.0f : beta * *c, epi, (int)n);
    }
}

struct PackJobs {
    PackJob job[2];
};

// Job blockIdx.y, in passes of 256 / w rows a block (w = 256, or the
// smallest of 128, 64, 32 that holds a row of ldp floats): w threads copy
// consecutive elements of a row with 4-byte loads and stores, so every warp
// instruction reads and writes 128 consecutive bytes whatever the source
// alignment, and write zeros in the padding columns [cols, ldp).  Each thread
// keeps kPackUnroll loads in flight.  (An earlier form with one 16-byte store
// per thread, four scalar loads 16 bytes apart and a 64-bit division per
// element read 1.7 TB/s at 2047^3; 16 loads a thread, one round for rows of
// up to 4096 floats, made 2047^3 and 1535^3 3-4 us slower.)
constexpr int kPackUnroll = 8;
constexpr int kPackThreads = 256;

__host__ __device__ inline int pack_width(long long ldp) {
    int w = kPackThreads;
    while (w > 32 && w / 2 >= ldp) w /= 2;
    return w;
}

__global__ void __launch_bounds__(kPackThreads) sgemm_pack_kernel(const PackJobs jobs) {
    const PackJob j = blockIdx.y == 0 ? jobs.job[0] : jobs.job[1];
    const int ldp = (int)j.ldp;
    const int w = pack_width(ldp);
    const int per_pass = kPackThreads / w;
    const int sub = threadIdx.x / w, col = threadIdx.x % w;
    for (long long r = (long long)blockIdx.x * per_pass + sub; r < j.rows;
         r += (long long)gridDim.x * per_pass) {
        const float *src = j.src + r * j.ld;
        float *dst = j.dst + r * j.ldp;
        for (int c0 = col; c0 < ldp; c0 += kPackUnroll * w) {
            float v[kPackUnroll];
#pragma unroll
            for (int u = 0; u < kPackUnroll; ++u) {
                const int c = c0 + u * w;
                v[u] = c < j.cols ? __ldg(src + c) : 0.0f;
            }
#pragma unroll
            for (int u = 0; u < kPackUnroll; ++u) {
                const int c = c0 + u * w;
                if (c < ldp) dst[c] = v[u];
            }
        }
    }
}

}  // namespace

cudaError_t launch_pack(const PackJob *jobs, int njobs, int num_sms, cudaStream_t stream) {
    if (njobs < 1 || njobs > 2) return cudaErrorInvalidValue;
    PackJobs pj = {};
    long long most = 0;
    for (int i = 0; i < njobs; ++i) {
        pj.job[i] = jobs[i];
        if (jobs[i].ldp > INT32_MAX || jobs[i].cols > jobs[i].ldp) return cudaErrorInvalidValue;
        const long long per_pass = kPackThreads / pack_width(jobs[i].ldp);
        const long long b = (jobs[i].rows + per_pass - 1) / per_pass;
        if (b > most) most = b;
    }
    // At most eight blocks per SM at a time.
    long long blocks = most;
    if (blocks > (long long)num_sms * 8) blocks = (long long)num_sms * 8;
    if (blocks < 1) blocks = 1;
    sgemm_pack_kernel<<<dim3((unsigned)blocks, (unsigned)njobs), kPackThreads, 0, stream>>>(pj);
    return cudaGetLastError();
}

cudaError_t launch_generic(const GenericParams &p, cudaStream_t stream) {
    const dim3 grid((p.N + GBN - 1) / GBN, (p.M + GBM - 1) / GBM);
    if (grid.y > 65535) return cudaErrorInvalidValue;
    sgemm_generic_kernel<<<grid, GNT, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_scale(int M, int N, float beta, float *C, long long ldc, const Epilogue &epi,
                         int num_sms, cudaStream_t stream) {
    const long long total = (long long)M * N;
    long long blocks = (total + 255) / 256;
    if (blocks > (long long)num_sms * 16) blocks = (long long)num_sms * 16;
    if (blocks < 1) blocks = 1;
    sgemm_scale_kernel<<<(int)blocks, 256, 0, stream>>>(M, N, beta, C, ldc, epi);
    return cudaGetLastError();
}

}  // namespace sgemm
