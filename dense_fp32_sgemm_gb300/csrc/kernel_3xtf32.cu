// 3xTF32 SGEMM on the fifth-generation tensor cores (tcgen05, sm_103a).
//
// Why a tensor-core variant at all: "GEMM from Scratch", Module 07 ("Tensor
// Cores -- Why They Dominate Peak") puts the tensor units on a separate,
// much higher throughput ceiling than the FP32 cores, and "Optimizing Matrix
// Multiply on CUDA, Part 2", section "Looking Back", names lower-precision
// inputs on tensor cores as the route past FP32-core parity.  The same module
// warns that TF32 drops mantissa bits, which FP32 work cannot accept, and
// "Optimizing CUDA matmul, steps 4 to 6", section "The honest target", keeps
// the FP32 contract free of TF32.  So this variant is a separate entry point
// that must meet the FP32 error bound of the FFMA kernels, and gets there by
// split-precision emulation (the published 3xTF32 method: Markidis et al.
// 2018; Ootomo and Yokota 2022):
//
//   x = hi + lo + e,   hi = tf32(x),  lo = tf32(x - hi)   (round to nearest)
//   |x - hi| <= 2^-11 |x|,  |e| <= 2^-22 |x|
//   a * b ~= hi_a*hi_b + hi_a*lo_b + lo_a*hi_b      (lo_a*lo_b <= 2^-22 |ab| dropped)
//
// Each TF32 x TF32 product (11 x 11 significant bits) is exact in the FP32
// accumulator, so the result differs from the FP32 one only by the dropped
// terms and the accumulation order.
//
// Structure (one 128 x bn tile of C per CTA, 64 <= bn <= 256, 128 threads,
// one or two CTAs per SM; deep products with few tiles give each CTA one K
// range of a tile instead, and a reduction kernel adds the ranges' raw tiles
// in order):
//   split pass   A -> [A_hi; A_lo] (K-major rows), B -> [B_hi^T; B_lo^T]
//                (transposed to K-major), zero padded; an HBM-bound pass.
//                The MMA kernel is launched as its programmatic dependent:
//                its CTAs set up while the pass finishes, and the load
//                issuer waits for the pass's results before its first copy.
//   warp 0       one thread issues the TMA loads of the operand tiles of each
//                K slice into a ring of swizzled shared-memory stages.
//   warp 1       one thread issues tcgen05.mma (M 128, N bn, K 8) three
//                times per K step, accumulating in tensor memory, and
//                releases each stage with tcgen05.commit.
//   warp 2       allocates and frees the 256 tensor-memory columns.
//   warps 2, 3   (large outputs) split each FP32 A tile in shared memory
//                instead of the pass.
//   all 4 warps  epilogue: tcgen05.ld of their 32 accumulator lanes, through
//                shared memory to coalesced rows, alpha / beta, bias and
//                ReLU, store; with beta != 0 the one-CTA forms bring the
//                tile of C into the idle stages with the TMA first.
// Every wait is bounded; on a timeout the kernel flags the error word, waits
// (bounded) for its copies and MMAs in flight, frees tensor memory and exits.
#include <algorithm>

#include "device_common.cuh"
#include "kernels_3xtf32.h"

namespace sgemm {
namespace {

constexpr int BM = kX3BM;
constexpr int BN = kX3BN;
constexpr int THREADS = 128;
constexpr int TMEM_COLS = BN;  // FP32 accumulator: 128 lanes x 256 columns

// Kernel forms: K slice BK (16 or 32) and ring stages S.  16 x 4 and 32 x 2
// take about 193 KB of shared memory (one CTA per SM); 16 x 2 takes 97 KB, so
// two CTAs share an SM and one's epilogue and start-up overlap the other's
// MMAs (each holds 256 of the SM's 512 tensor-memory columns).
template <int BK, int S>
struct X3Cfg {
    static_assert(BK == 32 || BK == 16, "K slice of 32 (128-byte rows) or 16 (64-byte rows)");
    static constexpr int kRowBytes = BK * 4;                  // one swizzled row of K
    static constexpr uint32_t kA = BM * BK * 4;               // one A part (hi or lo)
    static constexpr uint32_t kB = BN * BK * 4;               // one B part (room for N 256)
    static constexpr uint32_t kStage = 2 * kA + 2 * kB;
    static constexpr int kStages = S;
    static constexpr uint32_t kAlign = 8 * kRowBytes;         // one swizzle atom
    static constexpr size_t kSmem = (size_t)kStages * kStage + 1024;
    static constexpr int kCtasPerSm = kSmem <= 112 * 1024 ? 2 : 1;
    // The epilogue's C tile (128 KB) and staging (17 KB) fit in the idle ring.
    static constexpr bool kCTile = (size_t)kStages * kStage >= 145 * 1024;
    // shared-memory descriptor layout type: 2 = 128-byte swizzle, 4 = 64-byte
    static constexpr uint64_t kLayout = BK == 32 ? 2 : 4;
};

// tcgen05 shared-memory matrix descriptor for a K-major operand stored as
// rows of BK FP32 values with the TMA's matching swizzle: start address,
// stride between 8-row groups (one swizzle atom), fixed version bits 46-47 =
// 1, layout type in bits 61-63.  The leading offset is unused for swizzled
// K-major operands.
template <int BK>
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    using L = X3Cfg<BK, 2>;
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;                       // leading byte offset 16 (unused)
    d |= (uint64_t)(L::kAlign >> 4) << 32;        // stride byte offset: 8 rows
    d |= (uint64_t)1 << 46;
    d |= L::kLayout << 61;
    return d;
}

// Instruction descriptor, kind::tf32: FP32 accumulator (bits 4-5 = 1), A and
// B TF32 (bits 7-9, 10-12 = 2), both K-major (bits 15, 16 = 0), N >> 3 in
// bits 17-22, M >> 4 in bits 24-28.  N is a multiple of 16 in [16, 256].
__host__ __device__ constexpr uint32_t make_idesc(int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on `bar` once every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::
                     "r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Whole-warp tensor-memory allocation; the column base is written to *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                 "r"(TMEM_COLS)
                 : "memory");
}

// 32 consecutive accumulator columns of this warp's 32 lanes: thread i gets
// lane (base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    // The registers are valid only after the wait; tying them to it keeps
    // every use below it.
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                   "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// Round to TF32 (10 explicit mantissa bits), nearest with ties away from
// zero; the low 13 bits of the FP32 pattern are cleared.
__device__ __forceinline__ float to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r & 0xFFFFE000u);
}

__device__ __forceinline__ void split_tf32(float x, float &hi, float &lo) {
    hi = to_tf32(x);
    lo = to_tf32(x - hi);  // x - hi is exact in FP32
}

// ---------------------------------------------------------------------------
// Split pass.
// ---------------------------------------------------------------------------

struct SplitJob {
    const float *A;   // M x K, lda (null: A is split inside the MMA kernel)
    long long lda;
    int M, Mp;
    int a_vec4;       // A 16-byte aligned and lda a multiple of 4
    const float *B;   // K x N, ldb
    long long ldb;
    int N, Np;
    int K, Kp;
    float *outA, *outB;
    int a_blocks;     // blocks [0, a_blocks) split A; the rest split B
};

// A -> outA: rows [0, Mp) the hi parts and [Mp, 2 Mp) the lo parts, each row
// Kp floats (a multiple of 32), zero outside A.
__device__ __forceinline__ void split_a(const SplitJob &j, int block, int nblocks) {
    const int q_row = j.Kp / 4;
    const long long total = (long long)j.Mp * q_row;
    for (long long i = block * 256LL + threadIdx.x; i < total; i += nblocks * 256LL) {
        const int r = (int)(i / q_row), c = (int)(i % q_row) * 4;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < j.M) {
            const float *row = j.A + (long long)r * j.lda;
            if (j.a_vec4 && c + 3 < j.K) {
                x = __ldg(reinterpret_cast<const float4 *>(row + c));
            } else {
                if (c < j.K) x.x = __ldg(row + c);
                if (c + 1 < j.K) x.y = __ldg(row + c + 1);
                if (c + 2 < j.K) x.z = __ldg(row + c + 2);
                if (c + 3 < j.K) x.w = __ldg(row + c + 3);
            }
        }
        float4 h, l;
        split_tf32(x.x, h.x, l.x);
        split_tf32(x.y, h.y, l.y);
        split_tf32(x.z, h.z, l.z);
        split_tf32(x.w, h.w, l.w);
        *reinterpret_cast<float4 *>(j.outA + (size_t)r * j.Kp + c) = h;
        *reinterpret_cast<float4 *>(j.outA + ((size_t)j.Mp + r) * j.Kp + c) = l;
    }
}

// B -> outB transposed: row n of the hi part holds column n of B's hi values
// over k; lo rows start at Np.  Rows of Kp floats, zero outside B.  64 x 64
// tiles through shared memory (k fastest over the grid), so that reads run
// along B's rows and writes along the output's.
__device__ __forceinline__ void split_b(const SplitJob &j, int block, int nblocks,
                                        float (*t)[65]) {
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const long long k_tiles = (j.Kp + 63) / 64, tiles = k_tiles * ((j.Np + 63) / 64);
    for (long long b = block; b < tiles; b += nblocks) {
        const int k0 = (int)(b % k_tiles) * 64, n0 = (int)(b / k_tiles) * 64;
#pragma unroll
        for (int r = ty; r < 64; r += 8) {
            const int k = k0 + r;
            const float *row = j.B + (long long)k * j.ldb;
            const bool kin = k < j.K;
            t[r][tx] = (kin && n0 + tx < j.N) ? __ldg(row + n0 + tx) : 0.0f;
            t[r][tx + 32] = (kin && n0 + tx + 32 < j.N) ? __ldg(row + n0 + tx + 32) : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int r = ty; r < 64; r += 8) {
            const int n = n0 + r;
            if (n < j.Np) {
                float *hi = j.outB + (size_t)n * j.Kp, *lo = j.outB + ((size_t)j.Np + n) * j.Kp;
                float h, l;
                if (k0 + tx < j.Kp) {
                    split_tf32(t[tx][r], h, l);
                    hi[k0 + tx] = h;
                    lo[k0 + tx] = l;
                }
                if (k0 + tx + 32 < j.Kp) {
                    split_tf32(t[tx + 32][r], h, l);
                    hi[k0 + tx + 32] = h;
                    lo[k0 + tx + 32] = l;
                }
            }
        }
        __syncthreads();
    }
}

// One launch for both operands: the A blocks and the B blocks run side by
// side.
__global__ void __launch_bounds__(256) x3_split_kernel(const SplitJob j) {
    __shared__ float t[64][65];
    // The MMA kernel may start its set-up now; it waits for this grid's
    // results before its first load.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if ((int)blockIdx.x < j.a_blocks)
        split_a(j, blockIdx.x, j.a_blocks);
    else
        split_b(j, blockIdx.x - j.a_blocks, gridDim.x - j.a_blocks, t);
}

// C = alpha * (sum of the K ranges' raw tiles, in range order) + beta * C.
__global__ void __launch_bounds__(256) x3_reduce_kernel(const float *__restrict__ part,
                                                        int splits, long long stride,
                                                        long long ld_part, int M, int N,
                                                        float alpha, float beta, float *C,
                                                        long long ldc, const Epilogue epi) {
    const long long total = (long long)M * N;
    for (long long i = blockIdx.x * 256LL + threadIdx.x; i < total; i += gridDim.x * 256LL) {
        const int m = (int)(i / N), n = (int)(i % N);
        const float *q = part + (long long)m * ld_part + n;
        float sum = q[0];
        for (int j = 1; j < splits; ++j) sum += q[(long long)j * stride];
        float *c = C + (long long)m * ldc + n;
        float v = alpha * sum;
        if (beta != 0.0f) v = __fmaf_rn(beta, *c, v);
        *c = apply_epilogue(v, epi, n);
    }
}

// ---------------------------------------------------------------------------
// MMA kernel.
// ---------------------------------------------------------------------------
// Makes this thread's shared-memory writes visible to the tensor cores'
// (async proxy) reads that a later barrier orders after them.
__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ARAW: the TMA brings A's FP32 tile into the hi slot and warps 2 and 3 split
// it in place (hi there, lo into the lo slot) before the MMAs of that stage;
// otherwise both parts come from the split pass.
template <int BK, int STAGES, bool ARAW>
__global__ void __launch_bounds__(THREADS, (X3Cfg<BK, STAGES>::kCtasPerSm))
    sgemm_3xtf32_kernel(const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapB,
                        const __grid_constant__ CUtensorMap mapC, const X3Params p) {
    using L = X3Cfg<BK, STAGES>;
    constexpr int S = L::kStages;
    constexpr int kConvThreads = 64;  // warps 2 and 3
    extern __shared__ unsigned char x3_smem_raw[];
    __shared__ uint64_t full[S], empty[S], conv[S], accum_bar, c_bar;
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int s_abort;
    __shared__ int s_issued, s_consumed, s_accum_ok, s_converted, s_c_issued;

    // Stages start on a 1024-byte boundary of the shared window (the
    // swizzle pattern is taken from address bits).
    const uint32_t raw = smem_addr(x3_smem_raw);
    unsigned char *smem = x3_smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Tiles in groups of 16 tile rows, column by column inside a group: a
    // wave of CTAs shares about as many A rows as B columns, so fewer operand
    // bytes fall out of L2 between the CTAs that read them (measured 3-5 %
    // faster than walking whole columns at 4092^3 and above).
    // With a K split, CTA blockIdx takes K range blockIdx / tiles of tile
    // blockIdx % tiles.
    const int n_tiles = p.tiles_m * p.tiles_n;
    const int split = (int)blockIdx.x / n_tiles, tile = (int)blockIdx.x % n_tiles;
    constexpr int kGroupM = 16;
    const int per_group = kGroupM * p.tiles_n;
    const int first_m = (tile / per_group) * kGroupM;
    const int gsz = min(p.tiles_m - first_m, kGroupM);
    const int in_group = tile % per_group;
    const int tm = first_m + in_group % gsz, tn = in_group / gsz;
    const int kt0 = split * p.kt_per_split;
    const int nkt = min(p.kt_total - kt0, p.kt_per_split);  // >= 1
    // Output: C, or (K split) this range's slice of the partial sums, raw.
    float *const out = p.splits > 1 ? p.part + (size_t)split * p.part_stride : p.C;
    const long long ldo = p.splits > 1 ? p.part_ld : p.ldc;
    const int bn = p.bn;
    const int m0 = tm * BM, n0 = tn * bn;

    if (tid == 0) {
        prefetch_tensormap(&mapA);
        prefetch_tensormap(&mapB);
#pragma unroll
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&conv[s], kConvThreads);
        }
        mbar_init(&accum_bar, 1);
        mbar_init(&c_bar, 1);
        s_abort = 0;
        s_issued = 0;
        s_consumed = 0;
        s_accum_ok = 0;
        s_converted = 0;
        s_c_issued = 0;
        fence_barrier_init();
    }
    if (warp == 2) tmem_alloc(&tmem_slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // Producer: the four operand tiles of K slice kt into stage kt % S.
            // The split pass's output is complete and visible after this.
            asm volatile("griddepcontrol.wait;" ::: "memory");
            int kt = 0;
            for (; kt < nkt; ++kt) {
                if (p.skip_loads_from >= 0 && kt >= p.skip_loads_from) break;
                const int s = kt % S;
                if (kt >= S && !mbar_wait_bounded(&empty[s], ((kt / S) - 1) & 1, p.timeout_ns)) {
                    atomicOr(p.err, kErrWaitTimeout);
                    s_abort = 1;
                    break;
                }
                unsigned char *st = smem + (size_t)s * L::kStage;
                mbar_arrive_expect_tx(&full[s],
                                      (ARAW ? 1 : 2) * L::kA + 2 * (uint32_t)bn * BK * 4);
                const int k = (kt0 + kt) * BK;
                tma_load_2d(st, &mapA, &full[s], k, m0);
                if (!ARAW) tma_load_2d(st + L::kA, &mapA, &full[s], k, p.a_lo_row + m0);
                tma_load_2d(st + 2 * L::kA, &mapB, &full[s], k, n0);
                tma_load_2d(st + 2 * L::kA + L::kB, &mapB, &full[s], k, p.b_lo_row + n0);
            }
            s_issued = kt;
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            // MMA issuer: per K step of 8, the two correction products first,
            // then hi*hi; the first product of the tile overwrites D.
            int kt = 0;
            for (; kt < nkt; ++kt) {
                const int s = kt % S;
                if (!mbar_wait_bounded(ARAW ? &conv[s] : &full[s], (kt / S) & 1, p.timeout_ns)) {
                    atomicOr(p.err, kErrWaitTimeout);
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a_hi = sbase + s * L::kStage, a_lo = a_hi + L::kA;
                const uint32_t b_hi = a_hi + 2 * L::kA, b_lo = b_hi + L::kB;
                const uint32_t idesc = make_idesc(bn);
#pragma unroll
                for (int kk = 0; kk < BK / 8; ++kk) {
                    const uint32_t off = kk * 32;  // 8 TF32 values along K
                    mma_tf32(tmem, smem_desc<BK>(a_lo + off), smem_desc<BK>(b_hi + off), idesc,
                             (kt | kk) != 0);
                    mma_tf32(tmem, smem_desc<BK>(a_hi + off), smem_desc<BK>(b_lo + off), idesc, 1);
                    mma_tf32(tmem, smem_desc<BK>(a_hi + off), smem_desc<BK>(b_hi + off), idesc, 1);
                }
                mma_commit(&empty[s]);  // stage s is free once these MMAs are done
            }
            s_consumed = kt;
            mma_commit(&accum_bar);
        }
        __syncwarp();
    } else if (ARAW) {
        // Warps 2 and 3: split each landed A tile in place.  The conversion
        // is elementwise, so the swizzled positions the TMA chose are kept.
        const int c = tid - 64;
        int kt = 0;
        for (; kt < nkt; ++kt) {
            const int s = kt % S;
            if (!mbar_wait_bounded(&full[s], (kt / S) & 1, p.timeout_ns)) {
                atomicOr(p.err, kErrWaitTimeout);
                s_abort = 1;
                break;
            }
            float *a_hi = reinterpret_cast<float *>(smem + (size_t)s * L::kStage);
            float *a_lo = a_hi + L::kA / 4;
#pragma unroll
            for (int i = 0; i < (int)(L::kA / 16) / kConvThreads; ++i) {
                const int off = (i * kConvThreads + c) * 4;
                const float4 x = ld_shared_f4(a_hi + off);
                float4 h, l;
                split_tf32(x.x, h.x, l.x);
                split_tf32(x.y, h.y, l.y);
                split_tf32(x.z, h.z, l.z);
                split_tf32(x.w, h.w, l.w);
                st_shared_f4(a_hi + off, h);
                st_shared_f4(a_lo + off, l);
            }
            fence_proxy_async_shared();
            mbar_arrive(&conv[s]);
        }
        if (lane == 0) atomicMax(&s_converted, kt);
        __syncwarp();
    }
    __syncthreads();

    if (tid == 0) {
        // The accumulator is final (and every MMA finished) once the last
        // commit arrives.
        s_accum_ok = mbar_wait_bounded(&accum_bar, 0, p.timeout_ns) ? 1 : 0;
        if (!s_accum_ok) atomicOr(p.err, kErrDrainTimeout);
        // beta != 0: the stages are idle now; bring this tile's C in with the
        // TMA, 32 x 32 blocks, block (w, c) at floats (w * 8 + c) * 1024.
        if (L::kCTile && s_accum_ok && !s_abort && p.beta != 0.0f && p.c_tma) {
            const int chunks = (bn + 31) / 32;
            mbar_arrive_expect_tx(&c_bar, 4u * chunks * 32 * 32 * 4);
            for (int w = 0; w < 4; ++w)
                for (int c = 0; c < chunks; ++c)
                    tma_load_2d(smem + (size_t)(w * 8 + c) * 4096, &mapC, &c_bar, n0 + c * 32,
                                m0 + w * 32);
            s_c_issued = 1;
        }
    }
    __syncthreads();

    if (!s_abort && s_accum_ok) {
        tc_fence_after();
        // Epilogue: warp w owns accumulator lanes (rows) 32w .. 32w + 31.
        // Each 32-column block goes register -> shared (row per thread) ->
        // global (one row of 32 consecutive floats per warp store).
        // C (beta != 0) comes from shared memory when the TMA brought it,
        // else from global memory, 32 independent loads per thread first.
        const float *c_tile = reinterpret_cast<const float *>(smem);  // 128 KB
        float *stage = reinterpret_cast<float *>(smem + (L::kCTile ? 128 * 1024 : 0)) +
                       warp * (32 * 33);
        const uint32_t t_warp = tmem + ((uint32_t)(warp * 32) << 16);
        const int row0 = m0 + warp * 32;
        bool c_ok = true;
        if (s_c_issued) {
            int ok = 1;
            if (lane == 0) ok = mbar_wait_bounded(&c_bar, 0, p.timeout_ns) ? 1 : 0;
            c_ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
            if (!c_ok && lane == 0) atomicOr(p.err, kErrWaitTimeout);
        }
        for (int c = 0; c_ok && c * 32 < bn; ++c) {
            if (n0 + c * 32 >= p.N) break;  // uniform over the warp
            const int n = n0 + c * 32 + lane;
            const bool col_ok = n < p.N && c * 32 + lane < bn;
            float cv[32];
            if (p.beta != 0.0f) {
                if (s_c_issued) {
                    const float *blk = c_tile + (warp * 8 + c) * 1024;
#pragma unroll
                    for (int i = 0; i < 32; ++i) cv[i] = blk[i * 32 + lane];
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        cv[i] = (col_ok && row0 + i < p.M) ? out[(long long)(row0 + i) * ldo + n]
                                                           : 0.0f;
                }
            }
            uint32_t r[32];
            tmem_ld32(t_warp + c * 32, r);
#pragma unroll
            for (int j = 0; j < 32; ++j) stage[lane * 33 + j] = __uint_as_float(r[j]);
            __syncwarp();
            // The bias / activation test is made once per column block: the
            // plain loops are what calls without an epilogue run.
            const bool has_bias = p.epi.bias != nullptr, relu = p.epi.act == kActRelu;
            if (col_ok && (has_bias || relu)) {
                const float bias_n = has_bias ? __ldg(p.epi.bias + n) : 0.0f;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int m = row0 + i;
                    if (m < p.M) {
                        float v = p.alpha * stage[i * 33 + lane];
                        if (p.beta != 0.0f) v = __fmaf_rn(p.beta, cv[i], v);
                        if (has_bias) v += bias_n;  // as apply_epilogue: no add without a bias
                        if (relu) v = (v < 0.0f) ? 0.0f : v;
                        out[(long long)m * ldo + n] = v;
                    }
                }
            } else if (col_ok && p.beta != 0.0f) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int m = row0 + i;
                    if (m < p.M)
                        out[(long long)m * ldo + n] =
                            __fmaf_rn(p.beta, cv[i], p.alpha * stage[i * 33 + lane]);
                }
            } else if (col_ok) {
#pragma unroll 4
                for (int i = 0; i < 32; ++i) {
                    const int m = row0 + i;
                    if (m >= p.M) break;
                    out[(long long)m * ldo + n] = p.alpha * stage[i * 33 + lane];
                }
            }
            __syncwarp();
        }
    }

    if (tid == 0) {
        // Nothing may land in this CTA's shared memory after it exits: the
        // stage-release arrivals of the last commits, and (after a timeout)
        // loads that were issued but never consumed.
        const int consumed = s_consumed, issued = s_issued;
        // loads whose arrival someone waited for: by the converters (ARAW)
        // or by the MMA issuer
        const int landed = ARAW ? s_converted : consumed;
        for (int s = 0; s < S && s < consumed; ++s) {
            const int uses = (consumed - s + S - 1) / S;  // commits made to empty[s]
            if (!mbar_wait_bounded(&empty[s], (uses - 1) & 1, 1000000000ull)) {
                atomicOr(p.err, kErrDrainTimeout);
                break;
            }
        }
        if (s_c_issued && !mbar_wait_bounded(&c_bar, 0, 1000000000ull))
            atomicOr(p.err, kErrDrainTimeout);
        for (int j = landed; j < issued; ++j) {
            if (!mbar_wait_bounded(&full[j % S], (j / S) & 1, 1000000000ull)) {
                atomicOr(p.err, kErrDrainTimeout);
                break;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem);
    }
}

// ---------------------------------------------------------------------------
// Tensor-pipe rate probe: the TF32 dense peak the 3xTF32 kernel is judged
// against, measured in the same run.  One CTA per SM (its shared memory
// request leaves room for one) allocates 256 tensor-memory columns; one
// thread issues `iters` x 4 tcgen05.mma kind::tf32 of M 128, N 256, K 8 back
// to back into one accumulator, reading a 128 x 32 A tile and a 256 x 32 B
// tile (128-byte-swizzled K-major rows) of scattered values in [-0.5, 0.5)
// (zero operands would draw less power and run at a higher clock than real
// data), commits them to an mbarrier and waits (bounded) for them before the
// tensor memory is freed.
// FLOPs per launch: blocks * iters * 4 * 2 * 128 * 256 * 8.
// ---------------------------------------------------------------------------
constexpr uint32_t kProbeA = BM * 32 * 4, kProbeB = BN * 32 * 4;
constexpr size_t kProbeSmem = 120 * 1024;  // > half the SM: one CTA per SM

__global__ void __launch_bounds__(THREADS, 1)
    x3_mma_probe_kernel(long long iters, int *err, unsigned long long timeout_ns) {
    extern __shared__ unsigned char probe_raw[];
    __shared__ uint64_t done;
    __shared__ uint32_t tmem_slot;
    const uint32_t raw = smem_addr(probe_raw);
    unsigned char *smem = probe_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sbase = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5;
    float *f = reinterpret_cast<float *>(smem);
    for (int i = tid; i < (int)((kProbeA + kProbeB) / 4); i += THREADS) {
        const uint32_t h = (uint32_t)(i + 1) * 2654435761u;  // multiplicative hash
        f[i] = (float)(h >> 9) * (1.0f / 8388608.0f) - 0.5f;
    }
    fence_proxy_async_shared();
    if (tid == 0) {
        mbar_init(&done, 1);
        fence_barrier_init();
    }
    if (warp == 2) tmem_alloc(&tmem_slot);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (tid == 0) {
        const uint32_t idesc = make_idesc(BN);
        for (long long it = 0; it < iters; ++it) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_tf32(tmem, smem_desc<32>(sbase + kk * 32),
                         smem_desc<32>(sbase + kProbeA + kk * 32), idesc, (it | kk) != 0);
        }
        mma_commit(&done);
        if (!mbar_wait_bounded(&done, 0, timeout_ns)) {
            // Let the MMAs drain (bounded) before the columns are freed.
            atomicOr(err, kErrWaitTimeout);
            if (!mbar_wait_bounded(&done, 0, 1000000000ull)) atomicOr(err, kErrDrainTimeout);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem);
    }
}

}  // namespace

cudaError_t tf32_probe_configure() {
    return cudaFuncSetAttribute(x3_mma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)kProbeSmem);
}

cudaError_t launch_tf32_probe(long long iters, int blocks, int *err, unsigned long long timeout_ns,
                              cudaStream_t stream) {
    x3_mma_probe_kernel<<<blocks, THREADS, kProbeSmem, stream>>>(iters, err, timeout_ns);
    return cudaGetLastError();
}

namespace {
template <int BK, int S, bool ARAW>
cudaError_t x3_configure_one() {
    const cudaError_t e = cudaFuncSetAttribute(sgemm_3xtf32_kernel<BK, S, ARAW>,
                                               cudaFuncAttributePreferredSharedMemoryCarveout,
                                               100);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(sgemm_3xtf32_kernel<BK, S, ARAW>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)X3Cfg<BK, S>::kSmem);
}
template <int BK, int S, bool ARAW>
cudaError_t x3_launch_one(const CUtensorMap &mapA, const CUtensorMap &mapB,
                          const CUtensorMap &mapC, const X3Params &p, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.tiles_m * p.tiles_n * p.splits);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = X3Cfg<BK, S>::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sgemm_3xtf32_kernel<BK, S, ARAW>, mapA, mapB, mapC, p);
}
}  // namespace

bool x3_form_valid(int bk, int stages) {
    return (bk == 16 && (stages == 4 || stages == 2)) || (bk == 32 && stages == 2);
}

cudaError_t x3_configure(int bk, int stages, bool a_raw) {
    if (bk == 16 && stages == 4)
        return a_raw ? x3_configure_one<16, 4, true>() : x3_configure_one<16, 4, false>();
    if (bk == 16 && stages == 2)
        return a_raw ? x3_configure_one<16, 2, true>() : x3_configure_one<16, 2, false>();
    if (bk == 32 && stages == 2)
        return a_raw ? x3_configure_one<32, 2, true>() : x3_configure_one<32, 2, false>();
    return cudaErrorInvalidValue;
}

cudaError_t launch_x3(int bk, int stages, bool a_raw, const CUtensorMap &mapA,
                      const CUtensorMap &mapB, const CUtensorMap &mapC, const X3Params &p,
                      cudaStream_t stream) {
    if (bk == 16 && stages == 4)
        return a_raw ? x3_launch_one<16, 4, true>(mapA, mapB, mapC, p, stream)
                     : x3_launch_one<16, 4, false>(mapA, mapB, mapC, p, stream);
    if (bk == 16 && stages == 2)
        return a_raw ? x3_launch_one<16, 2, true>(mapA, mapB, mapC, p, stream)
                     : x3_launch_one<16, 2, false>(mapA, mapB, mapC, p, stream);
    if (bk == 32 && stages == 2)
        return a_raw ? x3_launch_one<32, 2, true>(mapA, mapB, mapC, p, stream)
                     : x3_launch_one<32, 2, false>(mapA, mapB, mapC, p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_x3_reduce(const float *part, int splits, long long stride, long long ld_part,
                             int M, int N, float alpha, float beta, float *C, long long ldc,
                             const Epilogue &epi, int num_sms, cudaStream_t stream) {
    const long long total = (long long)M * N;
    const long long blocks = std::min<long long>((total + 255) / 256, (long long)num_sms * 8);
    x3_reduce_kernel<<<(int)std::max<long long>(blocks, 1), 256, 0, stream>>>(
        part, splits, stride, ld_part, M, N, alpha, beta, C, ldc, epi);
    return cudaGetLastError();
}

cudaError_t launch_x3_split(const float *A, long long lda, int M, const float *B, long long ldb,
                            int N, int K, float *splitA, int Mp, float *splitB, int Np, int Kp,
                            int num_sms, cudaStream_t stream) {
    SplitJob j;
    j.A = A; j.lda = lda; j.M = M; j.Mp = Mp;
    j.a_vec4 = A && !(reinterpret_cast<uintptr_t>(A) & 15u) && !(lda & 3);
    j.B = B; j.ldb = ldb; j.N = N; j.Np = Np; j.K = K; j.Kp = Kp;
    j.outA = splitA; j.outB = splitB;
    // Blocks in proportion to the bytes each side moves (the same per
    // element), 16 per SM in all.
    const long long a_elems = A ? (long long)Mp * Kp : 0, b_elems = (long long)Np * Kp;
    const long long total_blocks = (long long)num_sms * 8;  // all resident at once
    long long a_blocks = A ? std::max<long long>(1, total_blocks * a_elems / (a_elems + b_elems)) : 0;
    a_blocks = std::min<long long>(a_blocks, (a_elems / 4 + 255) / 256);
    const long long b_tiles = (long long)((Kp + 63) / 64) * ((Np + 63) / 64);
    const long long b_blocks = std::max<long long>(1, std::min(total_blocks - a_blocks, b_tiles));
    j.a_blocks = (int)a_blocks;
    x3_split_kernel<<<(int)(a_blocks + b_blocks), 256, 0, stream>>>(j);
    return cudaGetLastError();
}

}  // namespace sgemm
