// sgemm_run_skinny_noalloc: the skinny-M product without any device
// allocation, for callers that cannot call cudaMalloc.
//
// Who needs it: code that runs while a framework's caching allocator owns all
// device memory (a cudaMalloc there can fail or fragment the pool), loops that
// must not allocate once they are set up (latency-critical decode loops,
// code checked to allocate only at start-up), and code paths where the
// allocation would be a synchronising call in the middle of queued work.
// sgemm_run allocates its stream-K workspace with cudaMalloc on first use;
// this entry point instead takes the partial sums, the arrival tickets and its
// error word from one fixed buffer that is part of the library image: a
// file-scope __device__ array, created by the CUDA runtime on each GPU that
// loads the library and held there until the process exits.
//
// Limits: M <= 16, at most kMaxSlabs slabs of 256 columns (N <= 1,048,576),
// A and B 16-byte aligned with leading dimensions that are multiples of 4.
// Anything else is rejected with SGEMM_ERR_SCRATCH_LIMIT before any work is
// queued.  The plan uses at most kMaxGrid = 160 CTAs in total
// (kSkinnyCtasPerSm per SM, so 160 / kSkinnyCtasPerSm SMs): a GPU with more
// SMs than that leaves the rest idle rather than outgrowing the buffer.
//
// A bounded device wait that gives up (a TMA copy that never lands) sets the
// buffer's own error word; sgemm_skinny_noalloc_status() reads and clears it.
// The calls themselves never clear it, so a timeout stays visible until it
// has been read.
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sgemm.h"
#include "kernels.h"
#include "plan.h"

namespace sgemm {
namespace {

constexpr int kMaxGrid = kSkinnyMaxGrid;
constexpr int kMaxM = 16;  // rows this entry point takes (tiles of 8 or 16 rows)
constexpr int kMaxSlabs = 4096;
constexpr int kMaxDevices = 64;
// The skinny kernel gives each CTA two partial slots of m_tile x 256 floats
// (at most 16 KiB here).
constexpr size_t kSlotFloats = size_t(kMaxM) * kSkinnyBN;
constexpr size_t kPartialBytes = 2 * size_t(kMaxGrid) * kSlotFloats * sizeof(float);
constexpr size_t kCounterBytes = size_t(kMaxSlabs) * sizeof(int);
constexpr size_t kErrOffset = kPartialBytes + kCounterBytes;
constexpr size_t kScratchBytes = kErrOffset + 256;  // 5 MiB + 16 KiB + 256 B with one CTA per SM

// The fixed scratch.  In host code this name is a host-side stand-in, not a
// device address: the host only ever passes the address cudaGetSymbolAddress
// returns for the current device.
static __device__ __align__(256) unsigned char g_skinny_scratch[kScratchBytes];

struct DeviceSetup {
    bool done = false;
    bool ok = false;
    int num_sms = 0;
    unsigned char *scratch = nullptr;  // device address of g_skinny_scratch
    bool configured8 = false, configured16 = false;
};
DeviceSetup g_setup[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode_fn = nullptr;

sgemm_status_t encode(CUtensorMap *map, const float *base, int64_t rows, int64_t cols, int64_t ld,
                      int box_cols, int box_rows,
                      CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode_fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                                   const_cast<float *>(base), dims, strides, box, estr,
                                   CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SGEMM_OK : SGEMM_ERR_TMA;
}

// Once per device, with that device current: check the architecture, look up
// the device address of the scratch array and fetch the TMA encoder.  Runs on
// the first call on each device; it queues no work, but the first call should
// still come before any stream capture.
sgemm_status_t setup_current_device(DeviceSetup **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return SGEMM_ERR_NO_DEVICE;
    DeviceSetup &s = g_setup[dev];
    if (!s.done) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SGEMM_ERR_NO_DEVICE;
        s.ok = (major == 10 && minor == 3);
        s.num_sms = sms;
        if (s.ok) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_skinny_scratch) != cudaSuccess || ptr == nullptr)
                return SGEMM_ERR_LAUNCH;
            s.scratch = static_cast<unsigned char *>(ptr);
        }
        s.done = true;
    }
    if (!s.ok) return SGEMM_ERR_NO_DEVICE;
    *out = &s;
    return SGEMM_OK;
}

sgemm_status_t setup_with_encoder(DeviceSetup **out) {
    DeviceSetup *s = nullptr;
    const sgemm_status_t st = setup_current_device(&s);
    if (st != SGEMM_OK) return st;
    if (!g_encode_fn) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return SGEMM_ERR_TMA;
        g_encode_fn = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = s;
    return SGEMM_OK;
}

}  // namespace
}  // namespace sgemm

using namespace sgemm;

extern "C" sgemm_status_t sgemm_run_skinny_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                                   const float *A, int64_t lda, const float *B,
                                                   int64_t ldb, float beta, float *C,
                                                   int64_t ldc, void *stream) {
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
        return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (!C || (reinterpret_cast<uintptr_t>(C) & 3u)) return SGEMM_ERR_INVALID_ARG;
    const bool product = K > 0 && alpha != 0.0f;
    if (product && (!A || !B || (reinterpret_cast<uintptr_t>(A) & 3u) ||
                    (reinterpret_cast<uintptr_t>(B) & 3u)))
        return SGEMM_ERR_INVALID_ARG;
    // Sizes and layouts this fixed buffer and kernel cannot take.
    if (M > kMaxM) return SGEMM_ERR_SCRATCH_LIMIT;
    if ((N + kSkinnyBN - 1) / kSkinnyBN > kMaxSlabs) return SGEMM_ERR_SCRATCH_LIMIT;
    if (product && ((reinterpret_cast<uintptr_t>(A) & 15u) || (reinterpret_cast<uintptr_t>(B) & 15u) ||
                    lda % 4 != 0 || ldb % 4 != 0))
        return SGEMM_ERR_SCRATCH_LIMIT;
    // Sizes no kernel of the library takes (the same answer sgemm_run gives).
    if (K > INT32_MAX / 2 || N > INT32_MAX / 2) return SGEMM_ERR_INVALID_ARG;

    DeviceSetup *dev = nullptr;
    sgemm_status_t s = setup_with_encoder(&dev);
    if (s != SGEMM_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!product) {
        const cudaError_t e = launch_scale((int)M, (int)N, beta, C, ldc, Epilogue{nullptr, kActNone},
                                           dev->num_sms, st);
        return e == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH;
    }

    PlanInput in;
    in.M = M; in.N = N; in.K = K; in.lda = lda; in.ldb = ldb; in.ldc = ldc;
    in.a_addr = reinterpret_cast<uintptr_t>(A);
    in.b_addr = reinterpret_cast<uintptr_t>(B);
    in.c_addr = reinterpret_cast<uintptr_t>(C);
    in.alpha = alpha; in.beta = beta;
    in.num_sms = dev->num_sms;
    in.force_variant = kVarSkinny;
    in.force_splits = 0;
    Plan pl;
    // The checks above leave only a (slab, k) plane too large for the
    // kernel's int positions (K of about 2^18 rows per slab and more), which
    // the skinny plan declines: no kernel here takes it.
    if (make_plan(in, &pl) != 0 || pl.variant != kVarSkinny) return SGEMM_ERR_UNSUPPORTED;
    if (pl.grid > kMaxGrid || pl.slabs > kMaxSlabs) return SGEMM_ERR_SCRATCH_LIMIT;

    bool &configured = pl.m_tile == 8 ? dev->configured8 : dev->configured16;
    if (!configured) {
        if (skinny_configure(pl.m_tile) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        configured = true;
    }
    CUtensorMap mapA, mapB;
    s = encode(&mapA, A, M, K, lda, kSkinnyBK, pl.m_tile, CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != SGEMM_OK) return s;
    s = encode(&mapB, B, K, N, ldb, kSkinnyBN, kSkinnyBK);
    if (s != SGEMM_OK) return s;

    int *counters = reinterpret_cast<int *>(dev->scratch + kPartialBytes);
    int *err = reinterpret_cast<int *>(dev->scratch + kErrOffset);
    // The buffer keeps the previous call's contents: the tickets must start
    // at zero (a call that gave up a wait may have left some taken).  The
    // error word is left alone, so an earlier timeout stays visible to
    // sgemm_skinny_noalloc_status().
    if (cudaMemsetAsync(counters, 0, (size_t)pl.slabs * sizeof(int), st) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;

    SkinnyParams sp;
    sp.M = (int)M; sp.N = (int)N; sp.K = (int)K;
    sp.slabs = pl.slabs; sp.kt_total = pl.kt_total;
    for (int c = 0; c <= pl.grid; ++c) sp.starts[c] = pl.sk_starts[c];
    sp.alpha = alpha; sp.beta = beta;
    sp.A = A; sp.lda = lda; sp.C = C; sp.ldc = ldc; sp.c_vec4 = 0;
    sp.epi = Epilogue{nullptr, kActNone};
    sp.partials = reinterpret_cast<float *>(dev->scratch);
    sp.counters = counters;
    sp.err = err;
    wait_hooks(&sp.timeout_ns, &sp.skip_loads_from);
    return launch_skinny(pl.m_tile, mapA, mapB, sp, pl.grid, st) == cudaSuccess ? SGEMM_OK
                                                                                 : SGEMM_ERR_LAUNCH;
}

extern "C" sgemm_status_t sgemm_skinny_noalloc_status(void *stream) {
    DeviceSetup *dev = nullptr;
    const sgemm_status_t s = setup_current_device(&dev);
    if (s != SGEMM_OK) return s;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    int *err = reinterpret_cast<int *>(dev->scratch + kErrOffset);
    int word = 0;
    if (cudaMemcpy(&word, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    if (word == 0) return SGEMM_OK;
    // Clear the word; the tickets are cleared by the next call itself.
    if (cudaMemset(err, 0, sizeof(int)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    return SGEMM_ERR_DEVICE_TIMEOUT;
}
