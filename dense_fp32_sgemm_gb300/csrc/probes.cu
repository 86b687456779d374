// Measurement probes for the roofline denominators, run in the same process
// as the GEMM ("Optimizing CUDA matmul, steps 4 to 6" measures its FMA peak in
// the same run; "Optimizing Matrix Multiply on CUDA, Part 2", section "Power
// Throttling": the sustained clock under load sets the real peak).
//
// - FFMA probe: every thread runs 16 independent multiply-add chains, either
//   as 16 scalar FFMA or 8 packed pairs per iteration; 2 flops per product.
// - Read probe: a grid-stride 128-bit streaming read of a buffer, summed so
//   the loads cannot be dropped.
// - Hold: one thread that sleeps on the GPU global timer for a fixed time,
//   so that the host can queue the next launches behind it and the device
//   never waits for the host between them.

#include "device_common.cuh"
#include "kernels.h"

namespace sgemm {
namespace {

__global__ void __launch_bounds__(512) ffma_probe_kernel(long long iters, float *sink) {
    const float seed = 1.0f + 1e-7f * (float)(threadIdx.x + 37 * blockIdx.x);
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = seed + 0.01f * i;
    const float a = 0.99999f + 1e-9f * threadIdx.x, b = 1e-5f * seed;
#pragma unroll 1
    for (long long it = 0; it < iters; ++it) {
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = __fmaf_rn(x[i], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) s += x[i];
    if (s == 1234.5f) sink[blockIdx.x] = s;  // practically never true; keeps the chains live
}

__global__ void __launch_bounds__(512) ffma2_probe_kernel(long long iters, float *sink) {
    const float seed = 1.0f + 1e-7f * (float)(threadIdx.x + 37 * blockIdx.x);
    float2 x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = make_float2(seed + 0.01f * i, seed - 0.01f * i);
    const float a0 = 0.99999f + 1e-9f * threadIdx.x;
    const float2 a = make_float2(a0, a0 - 1e-6f), b = make_float2(1e-5f * seed, 2e-5f * seed);
#pragma unroll 1
    for (long long it = 0; it < iters; ++it) {
#pragma unroll
        for (int r = 0; r < 8; ++r)
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] = __ffma2_rn(x[i], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += x[i].x + x[i].y;
    if (s == 1234.5f) sink[blockIdx.x] = s;
}

__global__ void read_probe_kernel(const float4 *__restrict__ buf, long long n4, float *sink) {
    float s = 0.f;
    const long long stride = (long long)gridDim.x * blockDim.x;
    long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n4; i += 4 * stride) {
        const float4 v0 = __ldcs(buf + i);
        const float4 v1 = __ldcs(buf + i + stride);
        const float4 v2 = __ldcs(buf + i + 2 * stride);
        const float4 v3 = __ldcs(buf + i + 3 * stride);
        s += (v0.x + v0.y + v0.z + v0.w) + (v1.x + v1.y + v1.z + v1.w) +
             (v2.x + v2.y + v2.z + v2.w) + (v3.x + v3.y + v3.z + v3.w);
    }
    for (; i < n4; i += stride) {
        const float4 v = __ldcs(buf + i);
        s += v.x + v.y + v.z + v.w;
    }
    if (s == 1234.5f) sink[blockIdx.x] = s;
}

__global__ void hold_kernel(unsigned long long ns) {
    const unsigned long long t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) __nanosleep(2000);
}

}  // namespace

// Products per thread per iteration: 8 rounds x 16 chains = 128 FMA.
cudaError_t launch_ffma_probe(int paired, long long iters, int blocks, float *sink,
                              cudaStream_t stream) {
    if (paired)
        ffma2_probe_kernel<<<blocks, 512, 0, stream>>>(iters, sink);
    else
        ffma_probe_kernel<<<blocks, 512, 0, stream>>>(iters, sink);
    return cudaGetLastError();
}

cudaError_t launch_read_probe(const float4 *buf, long long n4, float *sink, int blocks,
                              cudaStream_t stream) {
    read_probe_kernel<<<blocks, 512, 0, stream>>>(buf, n4, sink);
    return cudaGetLastError();
}

cudaError_t launch_hold(unsigned long long ns, cudaStream_t stream) {
    hold_kernel<<<1, 1, 0, stream>>>(ns);
    return cudaGetLastError();
}

}  // namespace sgemm
