// C ABI of the SGEMM library (declared in include/sgemm.h): argument checks,
// per-device state, workspace, TMA descriptors and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <set>
#include <utility>

#include "../../include/sgemm.h"
#include "../../include/sgemm_probe.h"
#include "kernels.h"
#include "kernels_3xtf32.h"
#include "plan.h"

namespace sgemm {
namespace {

constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // one second

std::atomic<int> g_force_variant{-1};
std::atomic<int> g_force_splits{0};
std::atomic<unsigned long long> g_timeout_ns{0};
std::atomic<int> g_skip_loads_from{-1};
std::atomic<int> g_fma_mode{kFmaPairMovB};
std::atomic<int> g_stages{3};
std::atomic<int> g_micro_m{16};
std::atomic<int> g_x3_bk{16};
std::atomic<int> g_x3_a_in_kernel{-1};  // -1: chosen per call
std::atomic<int> g_x3_splits{0};         // 0: chosen per call
std::atomic<int> g_x3_ctas_per_sm{0};    // 0: chosen per call

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct Workspace {
    float *partials = nullptr;
    size_t partial_bytes = 0;
    int *counters = nullptr;
    size_t counter_count = 0;
    float *pack = nullptr;  // aligned copies of unaligned operands
    size_t pack_bytes = 0;
    float *split = nullptr;  // 3xTF32 hi / lo operand copies
    size_t split_bytes = 0;
};

struct HostBuffers {
    float *A = nullptr, *B = nullptr, *C = nullptr;
    size_t a_bytes = 0, b_bytes = 0, c_bytes = 0;
};

// Streams and events of the host entry point's copy / compute pipeline.
constexpr int kHostMaxBlocks = 8;
struct HostPipeline {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in[kHostMaxBlocks] = {}, done[kHostMaxBlocks] = {};
};

struct DeviceState {
    HostPipeline pipe;
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    int *err = nullptr;  // device error word
    std::map<cudaStream_t, Workspace> ws;
    HostBuffers host;
    unsigned configured = 0;            // skinny configurations set up
    std::set<int> x3_configured;        // 3xTF32 kernel forms set up
    std::set<int> configured_tiles;     // tile configurations set up
    bool tf32_probe_configured = false;
    // Second stream for the thin edges beside the tiled kernel, forked from
    // and joined back to the caller's stream with the two events.
    cudaStream_t side = nullptr;
    cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
};

std::mutex g_mu;
std::map<int, DeviceState> g_dev;
EncodeTiledFn g_encode = nullptr;

sgemm_status_t status_from(cudaError_t e) { return e == cudaSuccess ? SGEMM_OK : SGEMM_ERR_LAUNCH; }

// Per-device state, created on first use with that device current.
sgemm_status_t device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_NO_DEVICE;
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SGEMM_ERR_NO_DEVICE;
        d.supported = (major == 10 && minor == 3);
        d.num_sms = sms;
        if (d.supported) {
            if (cudaMalloc(&d.err, sizeof(int)) != cudaSuccess) return SGEMM_ERR_ALLOC;
            if (cudaMemset(d.err, 0, sizeof(int)) != cudaSuccess) return SGEMM_ERR_ALLOC;
        }
        d.ready = true;
    }
    if (!d.supported) return SGEMM_ERR_NO_DEVICE;
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return SGEMM_ERR_TMA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    *out = &d;
    return SGEMM_OK;
}

sgemm_status_t ensure_workspace(DeviceState &d, cudaStream_t stream, size_t partial_bytes,
                                size_t counters, Workspace **out) {
    Workspace &w = d.ws[stream];
    if (w.partial_bytes < partial_bytes) {
        if (w.partials) cudaFree(w.partials);
        w.partials = nullptr;
        w.partial_bytes = 0;
        if (cudaMalloc(&w.partials, partial_bytes) != cudaSuccess) return SGEMM_ERR_ALLOC;
        w.partial_bytes = partial_bytes;
    }
    if (w.counter_count < counters) {
        if (w.counters) cudaFree(w.counters);
        w.counters = nullptr;
        w.counter_count = 0;
        if (cudaMalloc(&w.counters, counters * sizeof(int)) != cudaSuccess) return SGEMM_ERR_ALLOC;
        if (cudaMemset(w.counters, 0, counters * sizeof(int)) != cudaSuccess) return SGEMM_ERR_ALLOC;
        w.counter_count = counters;
    }
    *out = &w;
    return SGEMM_OK;
}

sgemm_status_t ensure_pack(DeviceState &d, cudaStream_t stream, size_t bytes, float **out) {
    Workspace &w = d.ws[stream];
    if (w.pack_bytes < bytes) {
        if (w.pack) cudaFree(w.pack);
        w.pack = nullptr;
        w.pack_bytes = 0;
        if (cudaMalloc(&w.pack, bytes) != cudaSuccess) return SGEMM_ERR_ALLOC;
        w.pack_bytes = bytes;
    }
    *out = w.pack;
    return SGEMM_OK;
}

// Row-major rows x cols FP32 matrix with leading dimension ld (elements),
// box of box_rows x box_cols, zero fill outside the matrix.
sgemm_status_t encode_2d(CUtensorMap *map, const float *base, int64_t rows, int64_t cols,
                         int64_t ld, int box_cols, int box_rows,
                         CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
    const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base),
                                dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SGEMM_OK : SGEMM_ERR_TMA;
}

sgemm_status_t validate(int64_t M, int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                        const float *B, int64_t ldb, float beta, const float *C, int64_t ldc) {
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
        return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (!C || (reinterpret_cast<uintptr_t>(C) & 3u)) return SGEMM_ERR_INVALID_ARG;
    if (K > 0 && alpha != 0.0f) {
        if (!A || !B) return SGEMM_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(A) & 3u) || (reinterpret_cast<uintptr_t>(B) & 3u))
            return SGEMM_ERR_INVALID_ARG;
    }
    (void)beta;
    return SGEMM_OK;
}

// Partial-sum workspace the skinny plan `pl` needs.
size_t skinny_partial_bytes(const Plan &pl) {
    return (size_t)2 * pl.grid * pl.m_tile * kSkinnyBN * sizeof(float);
}

// The skinny kernel on the plan `pl` (A and B 16-byte aligned, M <= 32), with
// the workspace `w` (at least skinny_partial_bytes(pl) and pl.slabs counters).
sgemm_status_t run_skinny(DeviceState &d, const Plan &pl, int64_t M, int64_t N, int64_t K,
                          float alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                          float beta, float *C, int64_t ldc, const Epilogue &epi, Workspace *w,
                          cudaStream_t stream) {
    const unsigned bit = 1u << (24 + pl.m_tile / 8);  // m_tile 8, 16, 32: bits 25, 26, 28
    if (!(d.configured & bit)) {
        if (skinny_configure(pl.m_tile) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        d.configured |= bit;
    }
    CUtensorMap mapA, mapB;
    sgemm_status_t s = encode_2d(&mapA, A, M, K, lda, kSkinnyBK, pl.m_tile,
                                 CU_TENSOR_MAP_SWIZZLE_128B);
    if (s != SGEMM_OK) return s;
    s = encode_2d(&mapB, B, K, N, ldb, kSkinnyBN, kSkinnyBK);
    if (s != SGEMM_OK) return s;
    SkinnyParams sp;
    sp.M = (int)M; sp.N = (int)N; sp.K = (int)K;
    sp.slabs = pl.slabs; sp.kt_total = pl.kt_total;
    for (int c = 0; c <= pl.grid; ++c) sp.starts[c] = pl.sk_starts[c];
    sp.alpha = alpha; sp.beta = beta;
    sp.A = A; sp.lda = lda; sp.C = C; sp.ldc = ldc; sp.c_vec4 = 0;
    sp.epi = epi;
    sp.err = d.err;
    const unsigned long long to = g_timeout_ns.load();
    sp.timeout_ns = to ? to : kDefaultTimeoutNs;
    sp.skip_loads_from = g_skip_loads_from.load();
    sp.partials = w->partials;
    sp.counters = w->counters;
    return status_from(launch_skinny(pl.m_tile, mapA, mapB, sp, pl.grid, stream));
}

// The narrow kernel over rows [0, M) and N <= kNarrowMaxN columns.
sgemm_status_t run_narrow(DeviceState &d, int nn, int a_vec, int grid, int rows_per_cta, int64_t M,
                          int64_t N, int64_t K, float alpha, const float *A, int64_t lda,
                          const float *B, int64_t ldb, float beta, float *C, int64_t ldc,
                          const Epilogue &epi, cudaStream_t stream) {
    const int key = 4000 + nn * 10 + a_vec;
    if (!d.configured_tiles.count(key)) {
        if (narrow_configure(nn, a_vec) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        d.configured_tiles.insert(key);
    }
    NarrowParams np;
    np.M = (int)M; np.N = (int)N; np.K = (int)K;
    np.alpha = alpha; np.beta = beta;
    np.A = A; np.lda = lda; np.B = B; np.ldb = ldb; np.C = C; np.ldc = ldc;
    np.epi = epi;
    np.rows_per_cta = rows_per_cta;
    np.kch = narrow_kch(K, nn);
    return status_from(launch_narrow(nn, a_vec, np, grid, stream));
}

sgemm_status_t run_locked(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                          int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                          int64_t ldc, const Epilogue &epi, cudaStream_t stream, DeviceState &d) {
    PlanInput in;
    in.M = M; in.N = N; in.K = K; in.lda = lda; in.ldb = ldb; in.ldc = ldc;
    in.a_addr = reinterpret_cast<uintptr_t>(A);
    in.b_addr = reinterpret_cast<uintptr_t>(B);
    in.c_addr = reinterpret_cast<uintptr_t>(C);
    in.alpha = alpha; in.beta = beta;
    in.num_sms = d.num_sms;
    in.force_variant = g_force_variant.load();
    in.force_splits = g_force_splits.load();
    Plan pl;
    if (make_plan(in, &pl) != 0) return SGEMM_ERR_INVALID_ARG;

    switch (pl.variant) {
        case kVarNone:
            return SGEMM_OK;
        case kVarScale:
            return status_from(launch_scale((int)M, (int)N, beta, C, ldc, epi, d.num_sms, stream));
        case kVarGeneric: {
            GenericParams gp;
            gp.M = (int)M; gp.N = (int)N; gp.K = (int)K;
            gp.alpha = alpha; gp.beta = beta;
            gp.A = A; gp.lda = lda; gp.B = B; gp.ldb = ldb; gp.C = C; gp.ldc = ldc;
            gp.epi = epi;
            return status_from(launch_generic(gp, stream));
        }
        case kVarTile:
        case kVarStreamK: {
            const int fm = g_fma_mode.load(), st = g_stages.load(), tm = g_micro_m.load();
            const int key = (fm * 10 + st) * 100 + tm;
            if (!d.configured_tiles.count(key)) {
                if (tile_configure(fm, st, tm) != cudaSuccess) return SGEMM_ERR_LAUNCH;
                d.configured_tiles.insert(key);
            }
            const float *Ause = A, *Buse = B;
            int64_t lda_use = lda, ldb_use = ldb;
            if (pl.pack_a || pl.pack_b) {
                // Copy the unaligned operand(s) to 16-byte-aligned rows first.
                const size_t a_floats = pl.pack_a ? (size_t)M * pl.lda_packed : 0;
                const size_t a_span = (a_floats + 63) / 64 * 64;  // keeps B's copy 256-byte aligned
                const size_t b_floats = pl.pack_b ? (size_t)K * pl.ldb_packed : 0;
                float *buf = nullptr;
                sgemm_status_t s = ensure_pack(d, stream, (a_span + b_floats) * sizeof(float), &buf);
                if (s != SGEMM_OK) return s;
                PackJob jobs[2];
                int n = 0;
                if (pl.pack_a) {
                    jobs[n++] = PackJob{A, lda, (int)M, (int)K, buf, pl.lda_packed};
                    Ause = buf;
                    lda_use = pl.lda_packed;
                }
                if (pl.pack_b) {
                    jobs[n++] = PackJob{B, ldb, (int)K, (int)N, buf + a_span, pl.ldb_packed};
                    Buse = buf + a_span;
                    ldb_use = pl.ldb_packed;
                }
                if (launch_pack(jobs, n, d.num_sms, stream) != cudaSuccess) return SGEMM_ERR_LAUNCH;
            }
            // Thin edges left to the skinny (last edge_m rows) and narrow (last
            // edge_n columns) kernels: the tiles cover M0 x N0.
            const int64_t M0 = M - pl.edge_m, N0 = N - pl.edge_n;
            Plan edge_plan = {};
            if (pl.edge_m > 0) {
                PlanInput ein = in;
                ein.M = pl.edge_m;
                ein.N = N0;
                ein.lda = lda_use;
                ein.ldb = ldb_use;
                ein.a_addr = reinterpret_cast<uintptr_t>(Ause + M0 * lda_use);
                ein.b_addr = reinterpret_cast<uintptr_t>(Buse);
                ein.c_addr = reinterpret_cast<uintptr_t>(C + M0 * ldc);
                ein.force_variant = kVarSkinny;
                ein.force_splits = 0;
                if (make_plan(ein, &edge_plan) != 0 || edge_plan.variant != kVarSkinny)
                    return SGEMM_ERR_UNSUPPORTED;
            }
            CUtensorMap mapA, mapB;
            sgemm_status_t s = encode_2d(&mapA, Ause, M0, K, lda_use, kTileBK, kTileBM);
            if (s != SGEMM_OK) return s;
            s = encode_2d(&mapB, Buse, K, N0, ldb_use, kTileBN, kTileBK);
            if (s != SGEMM_OK) return s;
            TileParams tp;
            tp.M = (int)M0; tp.N = (int)N0; tp.K = (int)K;
            tp.tiles_m = pl.tiles_m; tp.tiles_n = pl.tiles_n; tp.kt_total = pl.kt_total;
            tp.dp_tiles = pl.dp_tiles; tp.sk_tiles = pl.sk_tiles; tp.sk_share = pl.sk_share;
            tp.group_m = pl.group_m;
            tp.alpha = alpha; tp.beta = beta; tp.C = C; tp.ldc = ldc; tp.c_vec4 = pl.c_vec4;
            tp.epi = epi;
            tp.partials = nullptr; tp.counters = nullptr;
            tp.err = d.err;
            const unsigned long long to = g_timeout_ns.load();
            tp.timeout_ns = to ? to : kDefaultTimeoutNs;
            tp.skip_loads_from = g_skip_loads_from.load();
            // One workspace: the tiles' stream-K slots and counters first,
            // the bottom edge's after them (the two may run at once).
            Workspace *w = nullptr;
            const size_t tile_pbytes =
                pl.sk_tiles > 0 ? (size_t)2 * pl.grid * kTileBM * kTileBN * sizeof(float) : 0;
            const size_t tile_counters = (size_t)pl.sk_tiles;
            if (pl.sk_tiles > 0 || pl.edge_m > 0) {
                size_t pbytes = tile_pbytes, counters = tile_counters;
                if (pl.edge_m > 0) {
                    pbytes += skinny_partial_bytes(edge_plan);
                    counters += (size_t)edge_plan.slabs;
                }
                s = ensure_workspace(d, stream, pbytes, counters, &w);
                if (s != SGEMM_OK) return s;
                if (pl.sk_tiles > 0) {
                    tp.partials = w->partials;
                    tp.counters = w->counters;
                }
            }
            // The edges go to a second stream forked after the copies, so
            // that their CTAs take the SMs the tiles' last CTAs leave idle;
            // the caller's stream waits for them before anything it queues
            // next.  (During stream capture they stay on the caller's stream.)
            const bool edges = pl.edge_m > 0 || pl.edge_n > 0;
            cudaStream_t es = stream;
            if (edges) {
                cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
                if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return SGEMM_ERR_LAUNCH;
                if (cap == cudaStreamCaptureStatusNone) {
                    if (!d.side) {
                        if (cudaStreamCreateWithFlags(&d.side, cudaStreamNonBlocking) != cudaSuccess)
                            return SGEMM_ERR_LAUNCH;
                        if (cudaEventCreateWithFlags(&d.fork_ev, cudaEventDisableTiming) !=
                                cudaSuccess ||
                            cudaEventCreateWithFlags(&d.join_ev, cudaEventDisableTiming) !=
                                cudaSuccess)
                            return SGEMM_ERR_LAUNCH;
                    }
                    if (cudaEventRecord(d.fork_ev, stream) != cudaSuccess ||
                        cudaStreamWaitEvent(d.side, d.fork_ev, 0) != cudaSuccess)
                        return SGEMM_ERR_LAUNCH;
                    es = d.side;
                }
            }
            s = status_from(launch_tile(fm, st, tm, mapA, mapB, tp, pl.grid, stream));
            if (s != SGEMM_OK || !edges) return s;
            if (pl.edge_n > 0) {
                int grid = 0, rows = 0;
                narrow_grid(M, d.num_sms, &grid, &rows);
                Epilogue eepi = epi;
                if (eepi.bias) eepi.bias += N0;
                const int a_vec =
                    ((reinterpret_cast<uintptr_t>(Ause) & 15u) == 0 && lda_use % 4 == 0) ? 4 : 1;
                const int nn = pl.edge_n <= 1 ? 1 : pl.edge_n <= 2 ? 2 : 4;
                s = run_narrow(d, nn, a_vec, grid, rows, M, pl.edge_n, K, alpha, Ause, lda_use,
                               Buse + N0, ldb_use, beta, C + N0, ldc, eepi, es);
            }
            if (s == SGEMM_OK && pl.edge_m > 0) {
                Workspace ew = *w;
                ew.partials = reinterpret_cast<float *>(reinterpret_cast<char *>(w->partials) +
                                                        tile_pbytes);
                ew.counters = w->counters + tile_counters;
                s = run_skinny(d, edge_plan, pl.edge_m, N0, K, alpha, Ause + M0 * lda_use, lda_use,
                               Buse, ldb_use, beta, C + M0 * ldc, ldc, epi, &ew, es);
            }
            if (es != stream) {
                // Join even after a failed launch, so the caller's stream
                // never runs ahead of work already queued on the side.
                const bool joined = cudaEventRecord(d.join_ev, es) == cudaSuccess &&
                                    cudaStreamWaitEvent(stream, d.join_ev, 0) == cudaSuccess;
                if (s == SGEMM_OK && !joined) s = SGEMM_ERR_LAUNCH;
            }
            return s;
        }
        case kVarMid:
        case kVarMid64: {
            const int key = 1000 + pl.mid_bm * 10 + pl.b_vec;
            if (!d.configured_tiles.count(key)) {
                if (mid_configure(pl.mid_bm, pl.b_vec) != cudaSuccess) return SGEMM_ERR_LAUNCH;
                d.configured_tiles.insert(key);
            }
            MidParams mp;
            mp.M = (int)M; mp.N = (int)N; mp.K = (int)K;
            mp.tiles_m = pl.tiles_m; mp.tiles_n = pl.tiles_n; mp.kt_total = pl.kt_total;
            mp.dp_tiles = pl.dp_tiles; mp.sk_tiles = pl.sk_tiles; mp.sk_share = pl.sk_share;
            mp.group_m = pl.group_m;
            mp.alpha = alpha; mp.beta = beta;
            mp.A = A; mp.lda = lda; mp.B = B; mp.ldb = ldb; mp.C = C; mp.ldc = ldc;
            mp.c_vec4 = pl.c_vec4;
            mp.epi = epi;
            mp.partials = nullptr; mp.counters = nullptr;
            if (pl.sk_tiles > 0) {
                Workspace *w = nullptr;
                const size_t pbytes = (size_t)2 * pl.grid * pl.mid_bm * kMidBN * sizeof(float);
                const sgemm_status_t s = ensure_workspace(d, stream, pbytes, (size_t)pl.sk_tiles, &w);
                if (s != SGEMM_OK) return s;
                mp.partials = w->partials;
                mp.counters = w->counters;
            }
            return status_from(launch_mid(pl.mid_bm, pl.b_vec, mp, pl.grid, stream));
        }
        case kVarSmall: {
            const int key = 3000 + pl.b_vec;
            if (!d.configured_tiles.count(key)) {
                if (small_configure(pl.b_vec) != cudaSuccess) return SGEMM_ERR_LAUNCH;
                d.configured_tiles.insert(key);
            }
            MidParams mp = {};
            mp.M = (int)M; mp.N = (int)N; mp.K = (int)K;
            mp.tiles_m = pl.tiles_m; mp.tiles_n = pl.tiles_n; mp.kt_total = pl.kt_total;
            mp.dp_tiles = pl.dp_tiles; mp.sk_tiles = 0; mp.sk_share = 1;
            mp.group_m = 1;
            mp.alpha = alpha; mp.beta = beta;
            mp.A = A; mp.lda = lda; mp.B = B; mp.ldb = ldb; mp.C = C; mp.ldc = ldc;
            mp.c_vec4 = pl.c_vec4;
            mp.epi = epi;
            return status_from(launch_small(pl.b_vec, mp, pl.grid, stream));
        }
        case kVarKsplit:
        case kVarKsplit64: {
            const int key = 2000 + pl.ks_bn * 10 + pl.b_vec;
            if (!d.configured_tiles.count(key)) {
                if (ksplit_configure(pl.b_vec, pl.ks_bn) != cudaSuccess) return SGEMM_ERR_LAUNCH;
                d.configured_tiles.insert(key);
            }
            MidParams mp = {};
            mp.M = (int)M; mp.N = (int)N; mp.K = (int)K;
            mp.tiles_m = pl.tiles_m; mp.tiles_n = pl.tiles_n; mp.kt_total = pl.kt_total;
            mp.dp_tiles = pl.dp_tiles; mp.sk_tiles = 0; mp.sk_share = 1;
            mp.group_m = pl.group_m;
            mp.alpha = alpha; mp.beta = beta;
            mp.A = A; mp.lda = lda; mp.B = B; mp.ldb = ldb; mp.C = C; mp.ldc = ldc;
            mp.c_vec4 = pl.c_vec4;
            mp.epi = epi;
            return status_from(launch_ksplit(pl.b_vec, pl.ks_bn, mp, pl.grid, stream));
        }
        case kVarSkinny: {
            Workspace *w = nullptr;
            const sgemm_status_t s =
                ensure_workspace(d, stream, skinny_partial_bytes(pl), (size_t)pl.slabs, &w);
            if (s != SGEMM_OK) return s;
            return run_skinny(d, pl, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, epi, w, stream);
        }
        case kVarNarrow:
            return run_narrow(d, pl.narrow_nn, pl.a_vec, pl.grid, pl.narrow_rows, M, N, K, alpha, A,
                              lda, B, ldb, beta, C, ldc, epi, stream);
        default:
            return SGEMM_ERR_UNSUPPORTED;
    }
}

// The 3xTF32 entry point's choices for one call: whether the FFMA kernels
// take it, where A is split, the tile width, the K split and the kernel form.
struct X3Decision {
    bool ffma = false;  // K < 64, M <= 16 or alpha == 0: the FFMA kernels
    bool a_raw = false;
    int bk = 16, stages = 4, bn = kX3BN, splits = 1, kt_total = 0;
    int64_t ctas = 0;
};

X3Decision x3_decide(int64_t M, int64_t N, int64_t K, float alpha, uint64_t a_addr, int64_t lda,
                     int num_sms) {
    X3Decision x;
    if (K < kX3MinK || M <= 16 || alpha == 0.0f) {
        x.ffma = true;
        return x;
    }
    x.bk = g_x3_bk.load();
    // A split inside the kernel pays off only for large outputs whose A rows
    // start on 128-byte lines.  Measured on GB300 (TFLOP/s, split pass
    // against in-kernel split): 8192^3 270 / 281, 8192x6144x2048 227 / 238,
    // 6144x6144x2048 243 / 242, 4096x4096x8192 265 / 242, 4096^3 249 / 232,
    // 2048x8192x4096 254 / 221, 2048^3 194 / 190.
    const int a_mode = g_x3_a_in_kernel.load();
    x.a_raw = a_mode >= 0 ? a_mode != 0
                          : ((lda % 32) == 0 && !(a_addr & 127u) && M * N >= (int64_t)48 << 20);
    x.kt_total = (int)((K + x.bk - 1) / x.bk);
    x3_plan(M, N, x.kt_total, num_sms, g_x3_splits.load(), &x.bn, &x.splits);
    // Two CTAs per SM (K slice 16 only) overlap one tile's epilogue and
    // start-up with another's MMAs; they pay off once the launch has more
    // than one wave (measured on GB300: 3072^3 with 288 CTAs 230 -> 217 us,
    // 4092^3 520 -> 500 us, 8192^3 293 -> 308 TFLOP/s), while a single wave
    // would crowd onto half the SMs (2048^3: 80 -> 128 us).
    x.ctas = ((M + kX3BM - 1) / kX3BM) * ((N + x.bn - 1) / x.bn) * x.splits;
    const int cps = g_x3_ctas_per_sm.load();
    x.stages = x.bk == 32 ? 2 : (cps == 2 || (cps == 0 && x.ctas > (int64_t)num_sms)) ? 2 : 4;
    return x;
}

}  // namespace

void wait_hooks(unsigned long long *timeout_ns, int *skip_loads_from) {
    const unsigned long long to = g_timeout_ns.load();
    *timeout_ns = to ? to : kDefaultTimeoutNs;
    *skip_loads_from = g_skip_loads_from.load();
}

}  // namespace sgemm

using namespace sgemm;

extern "C" {

sgemm_status_t sgemm_run_epilogue(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                                  int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                                  int64_t ldc, const float *bias, int activation, void *stream) {
    const sgemm_status_t v = validate(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
    if (v != SGEMM_OK) return v;
    if (activation != SGEMM_ACT_NONE && activation != SGEMM_ACT_RELU) return SGEMM_ERR_INVALID_ARG;
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    const sgemm_status_t s = device_state(&d);
    if (s != SGEMM_OK) return s;
    Epilogue epi;
    epi.bias = bias;
    epi.act = activation == SGEMM_ACT_RELU ? kActRelu : kActNone;
    return run_locked(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, epi,
                      static_cast<cudaStream_t>(stream), *d);
}

sgemm_status_t sgemm_run(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                         int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                         int64_t ldc, void *stream) {
    return sgemm_run_epilogue(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, nullptr,
                              SGEMM_ACT_NONE, stream);
}

sgemm_status_t sgemm_run_3xtf32_epilogue(int64_t M, int64_t N, int64_t K, float alpha,
                                         const float *A, int64_t lda, const float *B, int64_t ldb,
                                         float beta, float *C, int64_t ldc, const float *bias,
                                         int activation, void *stream) {
    const sgemm_status_t v = validate(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
    if (v != SGEMM_OK) return v;
    if (activation != SGEMM_ACT_NONE && activation != SGEMM_ACT_RELU) return SGEMM_ERR_INVALID_ARG;
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    sgemm_status_t s = device_state(&d);
    if (s != SGEMM_OK) return s;
    Epilogue epi;
    epi.bias = bias;
    epi.act = activation == SGEMM_ACT_RELU ? kActRelu : kActNone;
    const X3Decision x = x3_decide(M, N, K, alpha, reinterpret_cast<uintptr_t>(A), lda,
                                   d->num_sms);
    if (x.ffma) return run_locked(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, epi, st, *d);
    if (M > (1 << 29) || N > (1 << 29) || K > (1 << 30) ||
        ((M + kX3BM - 1) / kX3BM) * ((N + kX3MinBN - 1) / kX3MinBN) * kX3MaxSplits > INT32_MAX)
        return SGEMM_ERR_INVALID_ARG;
    const int bk = x.bk, bn = x.bn, splits = x.splits, stages = x.stages, kt_total = x.kt_total;
    const bool a_raw = x.a_raw;
    const int form = bk * 100 + stages * 10 + (a_raw ? 1 : 0);
    if (!d->x3_configured.count(form)) {
        if (x3_configure(bk, stages, a_raw) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        d->x3_configured.insert(form);
    }
    const int64_t Mp = (M + kX3BM - 1) / kX3BM * kX3BM;
    const int64_t Np = (N + bn - 1) / bn * bn;
    const int64_t Kp = (K + 31) / 32 * 32;  // rows of whole 128-byte lines
    // Workspace: [A hi; A lo] (split pass only) | [B hi^T; B lo^T] | A copied
    // to 16-byte-aligned rows (A split in the kernel, when the TMA cannot
    // map A itself) | the K ranges' raw tiles (K split).
    const bool a_pack = a_raw && ((reinterpret_cast<uintptr_t>(A) & 15u) || (lda & 3));
    const int64_t ld_pack = (K + 3) / 4 * 4;
    const size_t a_floats = a_raw ? 0 : (size_t)(2 * Mp * Kp), b_floats = (size_t)(2 * Np * Kp);
    const size_t p_floats = a_pack ? (size_t)((M * ld_pack + 63) / 64 * 64) : 0;
    const size_t r_floats = splits > 1 ? (size_t)(splits * Mp * Np) : 0;
    Workspace &w = d->ws[st];
    const size_t bytes = (a_floats + b_floats + p_floats + r_floats) * sizeof(float);
    if (w.split_bytes < bytes) {
        if (w.split) cudaFree(w.split);
        w.split = nullptr;
        w.split_bytes = 0;
        if (cudaMalloc(&w.split, bytes) != cudaSuccess) return SGEMM_ERR_ALLOC;
        w.split_bytes = bytes;
    }
    // a_floats and b_floats are multiples of 64 floats (256 bytes)
    float *sa = w.split, *sb = w.split + a_floats, *pa = sb + b_floats, *pr = pa + p_floats;
    const float *a_map = A;
    int64_t lda_map = lda;
    if (a_pack) {
        const PackJob job{A, lda, (int)M, (int)K, pa, ld_pack};
        if (launch_pack(&job, 1, d->num_sms, st) != cudaSuccess) return SGEMM_ERR_LAUNCH;
        a_map = pa;
        lda_map = ld_pack;
    }
    if (launch_x3_split(a_raw ? nullptr : A, lda, (int)M, B, ldb, (int)N, (int)K, sa, (int)Mp, sb,
                        (int)Np, (int)Kp, d->num_sms, st) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    const CUtensorMapSwizzle sw = bk == 32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUtensorMap mapA, mapB;
    s = a_raw ? encode_2d(&mapA, a_map, M, K, lda_map, bk, kX3BM, sw)
              : encode_2d(&mapA, sa, 2 * Mp, Kp, Kp, bk, kX3BM, sw);
    if (s != SGEMM_OK) return s;
    s = encode_2d(&mapB, sb, 2 * Np, Kp, Kp, bk, bn, sw);
    if (s != SGEMM_OK) return s;
    X3Params p;
    p.M = (int)M; p.N = (int)N; p.K = (int)K;
    p.bn = bn;
    p.tiles_m = (int)(Mp / kX3BM); p.tiles_n = (int)(Np / bn);
    p.kt_total = kt_total;
    p.splits = splits;
    p.kt_per_split = (kt_total + splits - 1) / splits;
    p.part = pr; p.part_stride = Mp * Np; p.part_ld = Np;
    p.a_lo_row = (int)Mp; p.b_lo_row = (int)Np;
    // A K split writes raw sums; the reduction applies alpha and beta.
    p.alpha = splits > 1 ? 1.0f : alpha;
    p.beta = splits > 1 ? 0.0f : beta;
    p.C = C; p.ldc = ldc;
    p.epi = splits > 1 ? Epilogue{nullptr, kActNone} : epi;
    p.err = d->err;
    const unsigned long long to = g_timeout_ns.load();
    p.timeout_ns = to ? to : kDefaultTimeoutNs;
    p.skip_loads_from = g_skip_loads_from.load();
    CUtensorMap mapC = mapB;  // unused unless C is read through the TMA
    p.c_tma = 0;
    if (p.beta != 0.0f && !(reinterpret_cast<uintptr_t>(C) & 15u) && !(ldc & 3)) {
        s = encode_2d(&mapC, C, M, N, ldc, 32, 32);
        if (s != SGEMM_OK) return s;
        p.c_tma = 1;
    }
    if (launch_x3(bk, stages, a_raw, mapA, mapB, mapC, p, st) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    if (splits > 1 && launch_x3_reduce(pr, splits, Mp * Np, Np, (int)M, (int)N, alpha, beta, C,
                                       ldc, epi, d->num_sms, st) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    return SGEMM_OK;
}

sgemm_status_t sgemm_run_3xtf32(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                                int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                                int64_t ldc, void *stream) {
    return sgemm_run_3xtf32_epilogue(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, nullptr,
                                     SGEMM_ACT_NONE, stream);
}

// Host <-> device copy of `rows` rows of `width` floats; one contiguous copy
// when both pitches equal the row length.
cudaError_t copy_rows(float *dst, int64_t dpitch, const float *src, int64_t spitch, int64_t width,
                      int64_t rows, cudaMemcpyKind kind, cudaStream_t st) {
    if (dpitch == width && spitch == width)
        return cudaMemcpyAsync(dst, src, (size_t)(rows * width) * 4, kind, st);
    return cudaMemcpy2DAsync(dst, dpitch * 4, src, spitch * 4, width * 4, rows, kind, st);
}

sgemm_status_t sgemm_run_host(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                              int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                              int64_t ldc, void *stream) {
    sgemm_status_t v = validate(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc);
    if (v != SGEMM_OK) return v;
    if (M == 0 || N == 0) return SGEMM_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    sgemm_status_t s = device_state(&d);
    if (s != SGEMM_OK) return s;
    HostBuffers &hb = d->host;
    const bool need_ab = K > 0 && alpha != 0.0f;
    // Device copies use tight leading dimensions (the row lengths, rounded up
    // to 4 elements so rows stay 16-byte aligned).
    const int64_t dlda = (K + 3) / 4 * 4, dldb = (N + 3) / 4 * 4, dldc = (N + 3) / 4 * 4;
    auto grow = [](float **p, size_t *have, size_t want) -> bool {
        if (*have >= want) return true;
        if (*p) cudaFree(*p);
        *p = nullptr;
        *have = 0;
        if (cudaMalloc(p, want) != cudaSuccess) return false;
        *have = want;
        return true;
    };
    const size_t a_bytes = need_ab ? (size_t)M * dlda * 4 : 0;
    const size_t b_bytes = need_ab ? (size_t)K * dldb * 4 : 0;
    const size_t c_bytes = (size_t)M * dldc * 4;
    if (!grow(&hb.A, &hb.a_bytes, a_bytes ? a_bytes : 16) ||
        !grow(&hb.B, &hb.b_bytes, b_bytes ? b_bytes : 16) || !grow(&hb.C, &hb.c_bytes, c_bytes))
        return SGEMM_ERR_ALLOC;
    // Row blocks: copies of block i + 1 in and of block i - 1 out overlap the
    // product of block i (copy engines and SMs work at once).  B goes in
    // first, whole; small products are one block.
    // Each block must keep enough 128 x 256 x 32 slices per SM (24) for the
    // tiled kernel to stay efficient: measured at 2048^3, four 512-row
    // blocks took 416 us against 302 us for the whole product, two 1024-row
    // blocks about the whole product's time.
    int blocks = 1;
    int64_t rows = M;
    if (need_ab && M >= 1024) {
        const int64_t per_rows = ((N + 255) / 256) * ((K + 31) / 32);  // slices per 128 rows
        for (int cand = 4; cand >= 2; --cand) {
            const int64_t r = ((M + cand - 1) / cand + 127) / 128 * 128;
            if ((r / 128) * per_rows >= 24 * (int64_t)d->num_sms) {
                blocks = cand;
                rows = r;
                break;
            }
        }
        blocks = (int)((M + rows - 1) / rows);
    }
    if (blocks > 1) {
        HostPipeline &hp = d->pipe;
        if (!hp.ready) {
            bool ok = cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) == cudaSuccess &&
                      cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) == cudaSuccess &&
                      cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess &&
                      cudaEventCreateWithFlags(&hp.end, cudaEventDisableTiming) == cudaSuccess;
            for (int i = 0; ok && i < kHostMaxBlocks; ++i)
                ok = cudaEventCreateWithFlags(&hp.in[i], cudaEventDisableTiming) == cudaSuccess &&
                     cudaEventCreateWithFlags(&hp.done[i], cudaEventDisableTiming) == cudaSuccess;
            if (!ok) return SGEMM_ERR_LAUNCH;
            hp.ready = true;
        }
        // Everything already queued on `stream` comes first.
        if (cudaEventRecord(hp.start, st) != cudaSuccess ||
            cudaStreamWaitEvent(hp.h2d, hp.start, 0) != cudaSuccess ||
            cudaStreamWaitEvent(hp.d2h, hp.start, 0) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        if (copy_rows(hb.B, dldb, B, ldb, N, K, cudaMemcpyHostToDevice, hp.h2d) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        for (int i = 0; i < blocks; ++i) {
            const int64_t r0 = i * rows, mi = std::min<int64_t>(rows, M - r0);
            if (copy_rows(hb.A + r0 * dlda, dlda, A + r0 * lda, lda, K, mi, cudaMemcpyHostToDevice,
                          hp.h2d) != cudaSuccess)
                return SGEMM_ERR_LAUNCH;
            if (beta != 0.0f &&
                copy_rows(hb.C + r0 * dldc, dldc, C + r0 * ldc, ldc, N, mi, cudaMemcpyHostToDevice,
                          hp.h2d) != cudaSuccess)
                return SGEMM_ERR_LAUNCH;
            if (cudaEventRecord(hp.in[i], hp.h2d) != cudaSuccess ||
                cudaStreamWaitEvent(st, hp.in[i], 0) != cudaSuccess)
                return SGEMM_ERR_LAUNCH;
            s = run_locked(mi, N, K, alpha, hb.A + r0 * dlda, dlda, hb.B, dldb, beta,
                           hb.C + r0 * dldc, dldc, Epilogue{nullptr, kActNone}, st, *d);
            if (s != SGEMM_OK) return s;
            if (cudaEventRecord(hp.done[i], st) != cudaSuccess ||
                cudaStreamWaitEvent(hp.d2h, hp.done[i], 0) != cudaSuccess ||
                copy_rows(C + r0 * ldc, ldc, hb.C + r0 * dldc, dldc, N, mi, cudaMemcpyDeviceToHost,
                          hp.d2h) != cudaSuccess)
                return SGEMM_ERR_LAUNCH;
        }
        if (cudaEventRecord(hp.end, hp.d2h) != cudaSuccess ||
            cudaStreamWaitEvent(st, hp.end, 0) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
        return status_from(cudaStreamSynchronize(st));
    }
    if (need_ab) {
        if (copy_rows(hb.A, dlda, A, lda, K, M, cudaMemcpyHostToDevice, st) !=
                cudaSuccess ||
            copy_rows(hb.B, dldb, B, ldb, N, K, cudaMemcpyHostToDevice, st) !=
                cudaSuccess)
            return SGEMM_ERR_LAUNCH;
    }
    if (beta != 0.0f &&
        copy_rows(hb.C, dldc, C, ldc, N, M, cudaMemcpyHostToDevice, st) !=
            cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    s = run_locked(M, N, K, alpha, hb.A, dlda, hb.B, dldb, beta, hb.C, dldc, Epilogue{nullptr, kActNone},
                   st, *d);
    if (s != SGEMM_OK) return s;
    if (copy_rows(C, ldc, hb.C, dldc, N, M, cudaMemcpyDeviceToHost, st) !=
        cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    return status_from(cudaStreamSynchronize(st));
}

const char *sgemm_status_string(sgemm_status_t status) {
    switch (status) {
        case SGEMM_OK: return "SGEMM_OK";
        case SGEMM_ERR_INVALID_ARG: return "SGEMM_ERR_INVALID_ARG";
        case SGEMM_ERR_ALLOC: return "SGEMM_ERR_ALLOC";
        case SGEMM_ERR_TMA: return "SGEMM_ERR_TMA";
        case SGEMM_ERR_LAUNCH: return "SGEMM_ERR_LAUNCH";
        case SGEMM_ERR_DEVICE_TIMEOUT: return "SGEMM_ERR_DEVICE_TIMEOUT";
        case SGEMM_ERR_NO_DEVICE: return "SGEMM_ERR_NO_DEVICE";
        case SGEMM_ERR_UNSUPPORTED: return "SGEMM_ERR_UNSUPPORTED";
        case SGEMM_ERR_SCRATCH_LIMIT: return "SGEMM_ERR_SCRATCH_LIMIT";
        default: return "SGEMM_ERR_UNKNOWN";
    }
}

sgemm_status_t sgemm_device_status(void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    sgemm_status_t s = device_state(&d);
    if (s != SGEMM_OK) return s;
    if (cudaStreamSynchronize(st) != cudaSuccess) return SGEMM_ERR_LAUNCH;
    int word = 0;
    if (cudaMemcpy(&word, d->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return SGEMM_ERR_LAUNCH;
    if (word == 0) return SGEMM_OK;
    // A kernel gave up: clear the word and every arrival counter, so the
    // stream-K tickets of the abandoned call do not leak into the next one.
    if (cudaMemset(d->err, 0, sizeof(int)) != cudaSuccess) return SGEMM_ERR_LAUNCH;
    for (auto &kv : d->ws)
        if (kv.second.counters &&
            cudaMemset(kv.second.counters, 0, kv.second.counter_count * sizeof(int)) != cudaSuccess)
            return SGEMM_ERR_LAUNCH;
    if (cudaDeviceSynchronize() != cudaSuccess) return SGEMM_ERR_LAUNCH;
    return SGEMM_ERR_DEVICE_TIMEOUT;
}

sgemm_status_t sgemm_plan_describe(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                   int64_t ldc, uint64_t a_addr, uint64_t b_addr, uint64_t c_addr,
                                   float beta, int num_sms, char *buf, size_t len) {
    if (M < 0 || N < 0 || K < 0 || lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) ||
        ldc < (N > 1 ? N : 1) || !buf || len == 0)
        return SGEMM_ERR_INVALID_ARG;
    if (num_sms <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SGEMM_ERR_NO_DEVICE;
    }
    PlanInput in;
    in.M = M; in.N = N; in.K = K; in.lda = lda; in.ldb = ldb; in.ldc = ldc;
    in.a_addr = a_addr; in.b_addr = b_addr; in.c_addr = c_addr;
    in.alpha = 1.0f; in.beta = beta;
    in.num_sms = num_sms;
    in.force_variant = g_force_variant.load();
    in.force_splits = g_force_splits.load();
    Plan pl;
    if (make_plan(in, &pl) != 0) return SGEMM_ERR_INVALID_ARG;
    describe_plan(pl, buf, len);
    return SGEMM_OK;
}

sgemm_status_t sgemm_plan_describe_3xtf32(int64_t M, int64_t N, int64_t K, int64_t lda,
                                          uint64_t a_addr, int num_sms, char *buf, size_t len) {
    if (M < 0 || N < 0 || K < 0 || lda < (K > 1 ? K : 1) || !buf || len == 0)
        return SGEMM_ERR_INVALID_ARG;
    if (num_sms <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SGEMM_ERR_NO_DEVICE;
    }
    const X3Decision x = x3_decide(M, N, K, 1.0f, a_addr, lda, num_sms);
    if (x.ffma)
        snprintf(buf, len, "path=ffma");
    else
        snprintf(buf, len,
                 "path=tensor bk=%d stages=%d ctas_per_sm=%d a_in_kernel=%d tile_n=%d splits=%d "
                 "kt=%d ctas=%lld",
                 x.bk, x.stages, x.bk == 16 && x.stages == 2 ? 2 : 1, x.a_raw ? 1 : 0, x.bn,
                 x.splits, x.kt_total, (long long)x.ctas);
    return SGEMM_OK;
}

sgemm_status_t sgemm_set_plan_override(int variant, int splits) {
    if (variant < -1 || variant > SGEMM_VARIANT_SMALL || splits < 0) return SGEMM_ERR_INVALID_ARG;
    g_force_variant.store(variant);
    g_force_splits.store(splits);
    return SGEMM_OK;
}

sgemm_status_t sgemm_set_wait_timeout_ns(uint64_t timeout_ns, int skip_loads_from) {
    if (skip_loads_from < -1) return SGEMM_ERR_INVALID_ARG;
    g_timeout_ns.store(timeout_ns);
    g_skip_loads_from.store(skip_loads_from);
    return SGEMM_OK;
}

sgemm_status_t sgemm_set_tile_config(int fma_mode, int stages, int micro_m) {
    if (tile_smem_bytes(fma_mode, stages, micro_m) == 0) return SGEMM_ERR_INVALID_ARG;
    g_fma_mode.store(fma_mode);
    g_stages.store(stages);
    g_micro_m.store(micro_m);
    return SGEMM_OK;
}

sgemm_status_t sgemm_set_3xtf32_config(int bk, int a_in_kernel, int splits, int ctas_per_sm) {
    if ((bk != 16 && bk != 32) || a_in_kernel < -1 || a_in_kernel > 1 || splits < 0 ||
        splits > kX3MaxSplits || ctas_per_sm < 0 || ctas_per_sm > 2 ||
        (bk == 32 && ctas_per_sm == 2))
        return SGEMM_ERR_INVALID_ARG;
    g_x3_bk.store(bk);
    g_x3_a_in_kernel.store(a_in_kernel);
    g_x3_splits.store(splits);
    g_x3_ctas_per_sm.store(ctas_per_sm);
    return SGEMM_OK;
}

sgemm_status_t sgemm_release_workspace(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int prev = 0;
    cudaGetDevice(&prev);
    for (auto &kv : g_dev) {
        DeviceState &d = kv.second;
        if (!d.supported) continue;
        cudaSetDevice(kv.first);
        cudaDeviceSynchronize();
        for (auto &w : d.ws) {
            if (w.second.partials) cudaFree(w.second.partials);
            if (w.second.counters) cudaFree(w.second.counters);
            if (w.second.pack) cudaFree(w.second.pack);
            if (w.second.split) cudaFree(w.second.split);
        }
        d.ws.clear();
        if (d.side) cudaStreamDestroy(d.side);
        if (d.fork_ev) cudaEventDestroy(d.fork_ev);
        if (d.join_ev) cudaEventDestroy(d.join_ev);
        d.side = nullptr;
        d.fork_ev = d.join_ev = nullptr;
        if (d.host.A) cudaFree(d.host.A);
        if (d.host.B) cudaFree(d.host.B);
        if (d.host.C) cudaFree(d.host.C);
        d.host = HostBuffers();
    }
    cudaSetDevice(prev);
    return SGEMM_OK;
}

}  // extern "C"

extern "C" {

sgemm_status_t sgemm_probe_ffma(int paired, int64_t iters, int blocks, float *sink, void *stream) {
    if (iters < 1 || blocks < 1 || !sink) return SGEMM_ERR_INVALID_ARG;
    return status_from(launch_ffma_probe(paired, iters, blocks, sink,
                                         static_cast<cudaStream_t>(stream)));
}

sgemm_status_t sgemm_probe_read(const float *buf, int64_t n_floats, float *sink, int blocks,
                                void *stream) {
    if (!buf || !sink || blocks < 1 || n_floats < 4 || (n_floats & 3) ||
        (reinterpret_cast<uintptr_t>(buf) & 15u))
        return SGEMM_ERR_INVALID_ARG;
    return status_from(launch_read_probe(reinterpret_cast<const float4 *>(buf), n_floats / 4, sink,
                                         blocks, static_cast<cudaStream_t>(stream)));
}

sgemm_status_t sgemm_probe_tf32(int64_t iters, int blocks, void *stream) {
    // At most 2^18 iterations: about 80 ms, far inside the bounded wait.
    if (iters < 1 || iters > (int64_t(1) << 18) || blocks < 1) return SGEMM_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState *d = nullptr;
    const sgemm_status_t s = device_state(&d);
    if (s != SGEMM_OK) return s;
    if (!d->tf32_probe_configured) {
        if (tf32_probe_configure() != cudaSuccess) return SGEMM_ERR_LAUNCH;
        d->tf32_probe_configured = true;
    }
    unsigned long long timeout_ns = 0;
    int skip = -1;
    wait_hooks(&timeout_ns, &skip);
    return status_from(launch_tf32_probe((long long)iters, blocks, d->err, timeout_ns,
                                         static_cast<cudaStream_t>(stream)));
}

sgemm_status_t sgemm_probe_hold(int64_t ns, void *stream) {
    if (ns <= 0 || ns > 1000000000LL) return SGEMM_ERR_INVALID_ARG;
    return status_from(launch_hold((unsigned long long)ns, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
