// Variant selection and work split for one SGEMM call.
//
// Wave quantisation ("Optimizing Matrix Multiply on CUDA, Part 1", section
// "Small and Odd Sizes"): tiles run in waves of one per SM, so a last,
// partly filled wave leaves SMs idle.  Following "Part 2" (sections
// "Selecting Among Three Kernels" and "Distributing the Partially Filled
// Wave"), the planner estimates the work of the busiest SM for each
// candidate split and takes the cheapest:
//   - data-parallel: ceil(T / G) whole tiles per SM;
//   - stream-K: keep d full waves of whole tiles (d = floor(T/G) or one
//     fewer) and share the k-iterations of the other tiles evenly, with an
//     allowance per extra piece for combining partial sums.  Pieces are kept
//     to at most nine per tile (shares of at least an eighth of K), the most
//     the last CTA of a tile combines through its idle TMA ring; beyond that
//     the combination runs from L2 and costs more than it balances ("Part 2"
//     found two to four pieces best on a 48-SM part; measured on GB300,
//     640 x 640 x 8192: 5 pieces 320 us, 9 pieces 180 us, 11 pieces 217 us;
//     768 x 768 x 4096: 5 pieces 172 us, 9 pieces 105 us).
#include "plan.h"

#include <stdio.h>

#include "kernels.h"

namespace sgemm {

static_assert(sizeof(Plan::sk_starts) / sizeof(int) == kSkinnyMaxGrid + 1,
              "Plan::sk_starts holds one start per CTA and the end");

namespace {


// Time model of each kernel on GB300 (2070 MHz), fitted to CUDA-event times
// of single launches after an L2 flush (the planner sweep):
//   t = launch + slices of the busiest CTA x time of one slice at the SM's
//       CTA occupancy + (split tiles) fix-up + per extra piece,
// plus, for the tiled kernel on unaligned operands, the copy to aligned rows.
// launch: a 1 x 1 x 1 product takes 6.1 us from event to event.
struct KernelModel {
    int64_t bm, bn, bk;
    int ctas_per_sm;
    double slice_us[5];  // [c]: one CTA's slice with c CTAs resident per SM
    double fixup_us;     // once, when some tile is split
    double piece_us;     // per extra piece of the most-split tile
    double shared_fixup_us;  // once more when the split CTAs share SMs
    // Whole tiles only (no stream-K tail): slice time x dp_slice_scale and
    // dp_wave_us more per wave of tiles (first copies, the store).
    double dp_slice_scale;
    double dp_wave_us;
};
constexpr double kLaunchUs = 6.1;
// Tiled kernel: 2^20 multiply-adds per 128 x 256 x 32 slice, one CTA per SM;
// split tiles 14 us once plus 2 us per extra piece of the most-split tile
// (fitted over twelve shapes: 1536^3 with 2 pieces 131.5 us, 2048^3 with 3
// 273 us, 1024^3 with 4 60.4 us, 1024 x 1024 x 8192 with 6 283 us, 768 x
// 768 x 4096 with 8 104 us, 640 x 640 x 8192 with 8 178 us).  Whole tiles
// without a tail: 4.56 us a slice and 18 us a wave (one wave: 1000 x 3000 x
// 231 66.5 us, 1024^3 172.3, 2048^3 317.4, 768 x 768 x 4096 608.3, 1024 x
// 1024 x 8192 1190.9; two: 2049^3 635.9).
constexpr KernelModel kTileModel = {kTileBM, kTileBN, kTileBK, 1, {0, 4.7, 0, 0, 0}, 14.0, 2.0, 0.0,
                                    4.56 / 4.7, 18.0};
// Mid-size kernel, 128 x 128 x 16 slices: 1.43 us alone on an SM (512^3,
// 768^3, 100 x 5000 x 3000, 640 x 640 x 8192), 2.58 us per CTA with two per SM
// (2048^3 with 304 CTAs of 108 slices: 305 us; 1280^3, 4096^3); fix-up
// through the ring 4 us plus 2.5 us per
// extra piece (1024 x 1024 x 512 with 2 and 4 pieces: 37.3 and 39.4 us),
// and 5 us more with two CTAs per SM, where a CTA's fix-up runs beside the
// other's main loop (1280^3: 94.9 us, 2048 x 1024 x 1024: 96.7 us, 1400 x
// 1300 x 512: 61 us, each with 4 pieces).
constexpr KernelModel kMidModel = {128, kMidBN, kMidBK, 2, {0, 1.43, 2.58, 0, 0}, 4.0, 2.5, 5.0,
                                   1.0, 0.0};
// 64 x 128 x 16 slices, up to four CTAs per SM; a third or fourth CTA adds
// no throughput (64 x 8192 x 8192: 304 CTAs of 108 slices 170 us, 456 CTAs of
// 72 slices 211 us); 3 us per extra piece (40 x 40 x 4000, one tile in eight
// pieces: 64.3 us).
constexpr KernelModel kMid64Model = {64, kMidBN, kMidBK, 4, {0, 1.0, 1.5, 2.65, 3.5}, 3.0, 3.0, 0.0,
                                     1.0, 0.0};
// B in 4-byte copies (rows off 16 bytes) makes a mid-size slice slower
// (2049^3: 2.93 us per slice against 2.77 at 2048^3) and each unit's first
// copies slower to arrive: 1023 x 1025 x 513 (two units a CTA) took 51.2 us
// with 297 CTAs of 8 slices and with 140 of 17, about 7 us above the aligned
// 1024 x 1024 x 512 model.
constexpr double kMidUnalignedB[5] = {1.06, 1.06, 1.06, 1.06, 1.06};
constexpr double kMidUnalignedUnitUs = 3.5;
// Split-K kernel: one 64 x 128 (or 64 x 64) tile per CTA, one CTA per SM,
// slices of 64 k.  Per wave: a fixed part (first copies, the groups' sums
// added through shared memory, the store) and K / 64 slices plus a quarter
// slice for the rounding of the last one.  64 x 128 tiles: 1024 x 1024 x 512
// 29.3 us, 640^3 34.8, 1024^3 52.0, 768 x 768 x 4096 188 us, 1024 x 1024 x
// 8192 365 us; B in 4-byte copies (rows off 16 bytes) about 1.18x a slice
// (1023^3 60-61 us, 1023 x 1025 x 513 35.3 us).  64 x 64 tiles: 512^3 21.2
// us, 640^3 22.5, 768^3 26.6, 1024^3 (two waves) 60.1, 768 x 768 x 4096
// 112; with B in 4-byte copies 1.15x a slice (511^3 24.6 us, 1025^3 67.6).
constexpr double kKsSliceUs = 2.82;
constexpr double kKsFixedUs = 1.0;
constexpr double kKsUnalignedB = 1.18;
constexpr double kKsSliceUs64 = 1.6;
constexpr double kKsFixedUs64 = 1.5;
constexpr double kKsUnalignedB64 = 1.15;
constexpr double kNoScale[5] = {1, 1, 1, 1, 1};
// 64 x 64 kernel, one tile per CTA and 16-k slices: 0.78 us per slice at up to
// one CTA per SM (128^3: 12.3 us; 512^3: 30.9 us), growing with the CTAs an
// SM holds, first almost in proportion, then less (tiles per SM 1.7: 80 us
// at 1024^3; 3.0: 75.5 us at 1400 x 1300 x 512; 6.7: 478 us at 2048^3;
// 14.5: 163 us at 3000 x 3000 x 300).
constexpr double kGenericSliceUs = 0.78;
static double generic_scale(double tiles_per_sm) {
    if (tiles_per_sm <= 1.0) return 1.0;
    const double a = 0.9 * tiles_per_sm, b = 0.62 * tiles_per_sm + 0.6;
    return a < b ? a : b;
}
// Copy of unaligned operands for the tiled kernel: read and write at about
// 3 TB/s (2047^3: 24 us over 2048^3; 4095^3: 80 us over 4096^3), plus its
// own launch.
constexpr double kPackBytesPerUs = 3.0e6;
constexpr double kPackFixedUs = 4.0;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t gcd64(int64_t a, int64_t b) {
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

bool aligned16(uint64_t addr) { return (addr & 15u) == 0; }

int64_t round_up4(int64_t x) { return (x + 3) / 4 * 4; }

}  // namespace

const char *variant_name(int v) {
    switch (v) {
        case kVarNone: return "none";
        case kVarScale: return "scale";
        case kVarGeneric: return "generic";
        case kVarTile: return "tile";
        case kVarStreamK: return "streamk";
        case kVarSkinny: return "skinny";
        case kVarMid: return "mid";
        case kVarMid64: return "mid64";
        case kVarKsplit: return "ksplit";
        case kVarNarrow: return "narrow";
        case kVarKsplit64: return "ksplit64";
        case kVarSmall: return "small";
        default: return "?";
    }
}

// Time of one CTA slice when `ctas` CTAs share `sms` SMs (at most the
// model's CTAs per SM).
static double slice_us(const KernelModel &m, int64_t ctas, int64_t sms, const double *scale) {
    int64_t c = ceil_div(ctas, sms);
    if (c < 1) c = 1;
    if (c > m.ctas_per_sm) c = m.ctas_per_sm;
    return m.slice_us[c] * scale[c];
}

// Tiles of the model's shape on a persistent grid of at most
// sms * ctas_per_sm CTAs: whole tiles round-robin, or full waves whole and a
// stream-K tail; the candidate with the least estimated time.  `cost` is the
// busiest CTA's slices plus the fix-up allowance in slices; `est_us` the
// model's time (launch included).
static void plan_grid(const PlanInput &in, Plan *pl, bool allow_sk, bool force_sk,
                      const KernelModel &m, const double *slice_scale) {
    const int64_t sms = in.num_sms > 0 ? in.num_sms : 1;
    const int64_t G = sms * m.ctas_per_sm;
    const int64_t tm = ceil_div(in.M, m.bm), tn = ceil_div(in.N, m.bn);
    const int64_t T = tm * tn;
    const int64_t KT = ceil_div(in.K, m.bk);
    pl->tiles_m = (int)tm;
    pl->tiles_n = (int)tn;
    pl->kt_total = (int)KT;
    pl->group_m = (int)(tm < 8 ? tm : 8);
    pl->c_vec4 = (aligned16(in.c_addr) && in.ldc % 4 == 0) ? 1 : 0;

    // Data-parallel candidate.
    Plan best = *pl;
    best.variant = kVarTile;
    best.dp_tiles = (int)T;
    best.sk_tiles = 0;
    best.sk_share = 1;
    best.grid = (int)(T < G ? T : G);
    best.cost = (double)ceil_div(T, G) * (double)KT;
    best.est_us = kLaunchUs +
                  best.cost * slice_us(m, best.grid, sms, slice_scale) * m.dp_slice_scale +
                  (double)ceil_div(T, G) * m.dp_wave_us;
    best.reason = "whole tiles";

    const bool sk_fits = T * KT < (int64_t(1) << 30);
    if (allow_sk && sk_fits && (T % G != 0 || force_sk)) {
        const int64_t full = T / G;
        const double piece_slices =
            m.piece_us / (m.slice_us[m.ctas_per_sm] * slice_scale[m.ctas_per_sm]);
        for (int64_t d = full; d >= 0 && d >= full - 1; --d) {
            const int64_t dp = d * G;
            const int64_t sk_tiles = T - dp;
            if (sk_tiles <= 0) continue;
            const int64_t total = sk_tiles * KT;
            int64_t share = ceil_div(total, G);
            const int64_t min_share = ceil_div(KT, 8);
            // Shares from the smallest the grid and the piece limit allow,
            // upward: a larger share can save a piece or leave the SMs fewer
            // CTAs each.
            int64_t last = share;
            if (in.force_splits > 0) {
                // As close to the requested split as the grid allows.
                const int64_t want = ceil_div(KT, in.force_splits);
                share = want > share ? want : share;
                last = share;
            } else {
                if (share < min_share) share = min_share;
                last = m.ctas_per_sm > 1 ? 2 * share + 2 : share + share / 2 + 2;
                if (last > KT) last = KT > share ? KT : share;
            }
            if (share < 1) share = 1;
            bool taken = false;
            for (int64_t sh = share; sh <= last; ++sh) {
                const int64_t ctas = ceil_div(total, sh);
                if (ctas > G) continue;
                // Most pieces any tile is cut into: tile t starts at offset
                // t KT mod sh of a range, a multiple of gcd(KT, sh), so at
                // most sh - gcd into one.
                const int64_t pieces = ceil_div(KT + sh - gcd64(KT, sh), sh);
                const int64_t max_pieces = pieces < ctas ? pieces : ctas;
                const int64_t extra = max_pieces > 1 ? max_pieces - 1 : 0;
                // A share that splits no tile is the whole-tile plan again.
                if (extra == 0 && !force_sk) continue;
                const int64_t grid = dp > 0 ? G : ctas;
                const double cost = (double)d * KT + (double)sh + piece_slices * (double)extra;
                const double est =
                    kLaunchUs + ((double)d * KT + (double)sh) * slice_us(m, grid, sms, slice_scale) +
                    (extra > 0 ? m.fixup_us + m.piece_us * (double)extra +
                                     (grid > sms ? m.shared_fixup_us : 0.0)
                               : 0.0);
                if (est < best.est_us || (force_sk && !taken)) {
                    best.variant = kVarStreamK;
                    best.dp_tiles = (int)dp;
                    best.sk_tiles = (int)sk_tiles;
                    best.sk_share = (int)sh;
                    best.grid = (int)grid;
                    best.cost = cost;
                    best.est_us = est;
                    best.reason = "stream-K tail";
                    taken = true;
                }
            }
            if (taken && force_sk) break;
        }
    }
    *pl = best;
}

static void plan_tile(const PlanInput &in, Plan *pl, bool allow_sk, int64_t pack_floats) {
    plan_grid(in, pl, allow_sk, in.force_variant == kVarStreamK, kTileModel, kNoScale);
    if (pl->pack_a || pl->pack_b)
        pl->est_us += 2.0 * 4.0 * (double)pack_floats / kPackBytesPerUs + kPackFixedUs;
}

// The mid-size kernel (any alignment): bm x 128 tiles, K slices of 16,
// mid_ctas_per_sm(bm) CTAs per SM.
static void plan_mid(const PlanInput &in, Plan *pl, int bm) {
    const bool b_ok = aligned16(in.b_addr) && in.ldb % 4 == 0;
    plan_grid(in, pl, true, in.force_splits > 0, bm == 64 ? kMid64Model : kMidModel,
              b_ok ? kNoScale : kMidUnalignedB);
    pl->variant = kVarMid;
    pl->mid_bm = bm;
    pl->b_vec = b_ok ? 4 : 1;
    if (!b_ok) {
        // Units of the busiest CTA: a stream-K range shorter than a tile
        // usually ends in the tile after the one it starts in.
        const int64_t units = pl->sk_tiles > 0
                                  ? (pl->sk_share < pl->kt_total
                                         ? 2
                                         : (pl->sk_share + pl->kt_total - 1) / pl->kt_total + 1)
                                  : 1;
        pl->est_us += kMidUnalignedUnitUs * (double)units;
    }
    pl->reason = pl->sk_tiles > 0 ? "mid tiles, stream-K tail" : "mid tiles";
}

// The split-K kernel: one 64 x 128 tile per CTA over the whole K, in waves of
// one CTA per SM.
static void plan_ksplit(const PlanInput &in, Plan *pl, int bn) {
    const int64_t sms = in.num_sms > 0 ? in.num_sms : 1;
    const bool b_ok = aligned16(in.b_addr) && in.ldb % 4 == 0;
    const int64_t tm = ceil_div(in.M, kKsBM), tn = ceil_div(in.N, bn);
    const int64_t T = tm * tn;
    const int64_t KT = ceil_div(in.K, kKsBK);
    pl->variant = kVarKsplit;
    pl->tiles_m = (int)tm;
    pl->tiles_n = (int)tn;
    pl->kt_total = (int)KT;
    pl->group_m = (int)(tm < 8 ? tm : 8);
    pl->dp_tiles = (int)T;
    pl->sk_tiles = 0;
    pl->sk_share = 1;
    pl->grid = (int)T;
    pl->c_vec4 = (aligned16(in.c_addr) && in.ldc % 4 == 0) ? 1 : 0;
    pl->mid_bm = kKsBM;
    pl->ks_bn = bn;
    pl->b_vec = b_ok ? 4 : 1;
    const int64_t waves = ceil_div(T, sms);
    const double slices = (double)in.K / kKsBK + 0.25;
    pl->cost = (double)waves * slices;
    const double slice_us = bn == 64 ? kKsSliceUs64 * (b_ok ? 1.0 : kKsUnalignedB64)
                                     : kKsSliceUs * (b_ok ? 1.0 : kKsUnalignedB);
    pl->est_us = kLaunchUs + (double)waves * ((bn == 64 ? kKsFixedUs64 : kKsFixedUs) +
                                              slices * slice_us);
    pl->reason = "split-K inside the CTA";
}

// Streaming rates of the narrow and skinny kernels (bytes of the streamed
// operand per microsecond; 1 x 8192 x 8192 on the skinny kernel: 49 us) and
// the cost of a kernel queued right behind another one.
constexpr double kStreamBytesPerUs = 5.5e6;
constexpr double kChainedLaunchUs = 2.0;
// The narrow kernel's CTAs per SM and the time of one pass over a chunk of
// its K when the chunk, not the streaming, sets the pace.
constexpr int kNarrowCtasPerSm = 2;
constexpr double kNarrowChunkUs = 0.8;

// The narrow kernel (N <= kNarrowMaxN): contiguous row ranges, one warp per
// row, CTAs of 8 warps, up to kNarrowCtasPerSm per SM.
void narrow_grid(int64_t M, int num_sms, int *grid_out, int *rows_out) {
    const int64_t sms = num_sms > 0 ? num_sms : 1;
    int64_t grid = ceil_div(M, 8);
    if (grid > sms * kNarrowCtasPerSm) grid = sms * kNarrowCtasPerSm;
    if (grid < 1) grid = 1;
    const int64_t rows = ceil_div(M, grid);
    *grid_out = (int)ceil_div(M, rows);
    *rows_out = (int)rows;
}

static void plan_narrow(const PlanInput &in, Plan *pl) {
    int g = 0, r = 0;
    narrow_grid(in.M, in.num_sms, &g, &r);
    const int64_t grid = g, rows = r;
    pl->variant = kVarNarrow;
    pl->grid = (int)grid;
    pl->narrow_rows = (int)rows;
    pl->narrow_nn = in.N <= 1 ? 1 : in.N <= 2 ? 2 : 4;
    pl->a_vec = (aligned16(in.a_addr) && in.lda % 4 == 0) ? 4 : 1;
    pl->tiles_m = (int)grid;
    pl->tiles_n = 1;
    pl->kt_total = (int)ceil_div(in.K, narrow_kch(in.K, pl->narrow_nn));
    const double stream = (double)in.M * (double)in.K * 4.0 / kStreamBytesPerUs;
    const double passes = (double)ceil_div(rows, 8) * (double)pl->kt_total * kNarrowChunkUs;
    pl->cost = (double)ceil_div(rows, 8) * (double)pl->kt_total;
    pl->est_us = kLaunchUs + (stream > passes ? stream : passes);
    pl->reason = "narrow N: stream A once";
}

// The small-product kernel: one 32 x 32 tile per CTA, up to
// kSmallCtasPerSm CTAs per SM; each wave costs K / 64 slices (plus a quarter
// for the rounding of the last) at the time of one slice with that wave's
// CTAs per SM, fitted on GB300: 128^3 8.2 us, 256^3 10.2, 384^3 11.7 (one
// CTA per SM), 512^3 18.4 (two), 640^3 27.0, 600 x 600 x 2000 72.4 (three),
// 768^3 38.9, 128 x 4096 x 1024 49.9 (four), 1024^3 82.4 (four, then three).
constexpr double kSmallFixedUs = 0.3;
constexpr double kSmallSliceUs[kSmallCtasPerSm + 1] = {0, 0.87, 1.5, 2.07, 2.7};
constexpr double kSmallUnalignedB = 1.2;

static void plan_small(const PlanInput &in, Plan *pl) {
    const int64_t sms = in.num_sms > 0 ? in.num_sms : 1;
    const bool b_ok = aligned16(in.b_addr) && in.ldb % 4 == 0;
    const int64_t tm = ceil_div(in.M, kSmallBM), tn = ceil_div(in.N, kSmallBN);
    const int64_t T = tm * tn;
    pl->variant = kVarSmall;
    pl->tiles_m = (int)tm;
    pl->tiles_n = (int)tn;
    pl->kt_total = (int)ceil_div(in.K, kSmallBK);
    pl->group_m = 1;
    pl->dp_tiles = (int)T;
    pl->sk_tiles = 0;
    pl->sk_share = 1;
    pl->grid = (int)T;
    pl->c_vec4 = (aligned16(in.c_addr) && in.ldc % 4 == 0) ? 1 : 0;
    pl->b_vec = b_ok ? 4 : 1;
    const int64_t per_wave = sms * kSmallCtasPerSm;
    const int64_t full = T / per_wave, rem = T % per_wave;
    const double slices = (double)in.K / kSmallBK + 0.25;
    const double scale = b_ok ? 1.0 : kSmallUnalignedB;
    double t = (double)full * (kSmallFixedUs + slices * kSmallSliceUs[kSmallCtasPerSm] * scale);
    if (rem > 0) t += kSmallFixedUs + slices * kSmallSliceUs[ceil_div(rem, sms)] * scale;
    pl->cost = (double)(full + (rem > 0)) * slices;
    pl->est_us = kLaunchUs + t;
    pl->reason = "32 x 32 tiles, split K inside the CTA";
}

// The 64 x 64 kernel: one tile per CTA over the whole K.
static void plan_generic(const PlanInput &in, Plan *pl) {
    const int64_t sms = in.num_sms > 0 ? in.num_sms : 1;
    pl->variant = kVarGeneric;
    pl->tiles_m = (int)ceil_div(in.M, kGenBM);
    pl->tiles_n = (int)ceil_div(in.N, kGenBN);
    pl->kt_total = (int)ceil_div(in.K, kGenBK);
    pl->grid = pl->tiles_m * pl->tiles_n;
    const double scale = generic_scale((double)pl->grid / (double)sms);
    pl->cost = (double)pl->kt_total;
    pl->est_us = kLaunchUs + (double)pl->kt_total * kGenericSliceUs * scale;
}

// Contiguous ranges of the skinny kernel's positions, one per CTA, balanced
// in time rather than in positions: a range pays `unit_end` positions for
// every slab boundary it crosses, and a range that could cross a boundary
// only by paying more than it has left ends on the boundary instead.  Each
// range takes as much as a budget of T allows; returns the number of ranges
// (CTAs), or -1 if they do not fit in max_ctas.
static int64_t skinny_ranges(int64_t total, int64_t KT, int64_t max_ctas, int64_t unit_end,
                             int64_t T, int *starts) {
    int64_t s = 0, c = 0;
    while (s < total) {
        if (c >= max_ctas) return -1;
        if (starts) starts[c] = (int)s;
        int64_t e = s, budget = T;
        while (true) {
            const int64_t b = (e / KT + 1) * KT;  // next slab boundary after e
            if (e + budget <= b) {
                e += budget;
                break;
            }
            budget -= b - e;
            e = b;
            if (e >= total || budget <= unit_end) break;
            budget -= unit_end;
        }
        s = e < total ? e : total;
        ++c;
    }
    if (starts) starts[c] = (int)total;
    return c;
}

int make_plan(const PlanInput &in, Plan *pl) {
    Plan p = {};
    p.variant = kVarGeneric;
    p.sk_share = 1;
    p.group_m = 1;
    p.reason = "";
    if (in.M == 0 || in.N == 0) {
        p.variant = kVarNone;
        p.reason = "empty output";
        *pl = p;
        return 0;
    }
    if (in.K == 0 || in.alpha == 0.0f) {
        p.variant = kVarScale;
        p.reason = "alpha == 0 or K == 0";
        *pl = p;
        return 0;
    }
    if (in.M > INT32_MAX / 2 || in.N > INT32_MAX / 2 || in.K > INT32_MAX / 2) return -1;

    const bool a_ok = aligned16(in.a_addr) && in.lda % 4 == 0 && in.lda < (int64_t(1) << 37);
    const bool b_ok = aligned16(in.b_addr) && in.ldb % 4 == 0 && in.ldb < (int64_t(1) << 37);
    const bool tma_ok = a_ok && b_ok;
    int want = in.force_variant;
    if (want == kVarSkinny && !tma_ok) return -2;
    if (want == kVarSkinny && in.M > kSkinnyMaxM) return -3;

    // M <= 32: every B element feeds at most 32 products, so the product is
    // bound by streaming B (M <= 16) or close to it; a tile of 64 or 128 rows
    // would spend 2-8x the multiply-adds (measured, 32 x 8192 x 8192: see the
    // planner sweep).
    // Below about 2^21 elements of B the skinny kernel's start-up and fix-up
    // outweigh the streaming (32 x 32 x 32: 14.7 us against 6.9 on the
    // small-product kernel; 16 x 1024 x 1024: 21.5 against 20.5), so the time
    // model chooses there.
    const bool big_b = in.N * in.K >= (int64_t(1) << 21);
    if (tma_ok && (want == kVarSkinny || (want < 0 && in.M <= kSkinnyMaxM && big_b))) {
        // Persistent grid: every CTA the SMs hold at once.
        int64_t G = (in.num_sms > 0 ? in.num_sms : 1) * kSkinnyCtasPerSm;
        if (G > kSkinnyMaxGrid) G = kSkinnyMaxGrid;
        const int64_t slabs = ceil_div(in.N, kSkinnyBN);
        const int64_t KT = ceil_div(in.K, kSkinnyBK);
        const int64_t total = slabs * KT;
        if (total < (int64_t(1) << 30)) {
            // Smallest budget whose ranges fit the grid (a forced split
            // count asks for ranges of at least KT / splits positions).
            // (one range over everything pays at most one unit end per slab)
            int64_t lo = ceil_div(total, G), hi = total + kSkinnyUnitEndCost * slabs;
            if (in.force_splits > 0) {
                const int64_t w = ceil_div(KT, in.force_splits);
                if (w > lo) lo = w;
                if (hi < lo) hi = lo;
            }
            while (lo < hi) {
                const int64_t mid = lo + (hi - lo) / 2;
                if (skinny_ranges(total, KT, G, kSkinnyUnitEndCost, mid, nullptr) > 0)
                    hi = mid;
                else
                    lo = mid + 1;
            }
            p.variant = kVarSkinny;
            p.m_tile = in.M <= 8 ? 8 : in.M <= 16 ? 16 : 32;
            p.slabs = (int)slabs;
            p.tiles_n = (int)slabs;
            p.tiles_m = 1;
            p.kt_total = (int)KT;
            p.sk_share = (int)lo;
            p.grid = (int)skinny_ranges(total, KT, G, kSkinnyUnitEndCost, lo, p.sk_starts);
            p.sk_two_units = 0;
            for (int c = 0; c < p.grid; ++c)
                if (p.sk_starts[c] / KT != (p.sk_starts[c + 1] - 1) / KT) ++p.sk_two_units;
            p.c_vec4 = 0;
            p.cost = (double)lo;
            p.reason = "small M: stream B once";
            *pl = p;
            return 0;
        }
    }

    // Forced kernels (tests and the planner sweep).
    if (want == kVarGeneric) {
        plan_generic(in, &p);
        p.reason = "forced";
        *pl = p;
        return 0;
    }
    if (want == kVarMid || want == kVarMid64) {
        plan_mid(in, &p, want == kVarMid64 ? 64 : 128);
        *pl = p;
        return 0;
    }
    if (want == kVarSmall) {
        if (ceil_div(in.M, kSmallBM) * ceil_div(in.N, kSmallBN) > INT32_MAX) return -2;
        plan_small(in, &p);
        *pl = p;
        return 0;
    }
    if (want == kVarNarrow) {
        if (in.N > kNarrowMaxN) return -3;
        plan_narrow(in, &p);
        *pl = p;
        return 0;
    }
    if (want == kVarKsplit || want == kVarKsplit64) {
        const int bn = want == kVarKsplit64 ? 64 : 128;
        if (ceil_div(in.M, kKsBM) * ceil_div(in.N, bn) > INT32_MAX) return -2;
        plan_ksplit(in, &p, bn);
        *pl = p;
        return 0;
    }
    // Operands the TMA cannot map (a pointer or leading dimension off 16
    // bytes) can be copied to 16-byte-aligned rows for the tiled kernel.
    const int64_t pack_floats = (a_ok ? 0 : in.M * round_up4(in.K)) +
                                (b_ok ? 0 : in.K * round_up4(in.N));
    const bool packable = pack_floats < (int64_t(1) << 31);
    auto tile_plan = [&](Plan *t, bool allow_sk) {
        t->pack_a = !a_ok;
        t->pack_b = !b_ok;
        t->lda_packed = t->pack_a ? round_up4(in.K) : in.lda;
        t->ldb_packed = t->pack_b ? round_up4(in.N) : in.ldb;
        plan_tile(in, t, allow_sk, pack_floats);
        if (!tma_ok) t->reason = "operands copied to aligned rows";
    };
    // The tiled kernel on all but a thin last strip of rows (<= 32: the
    // skinny kernel) and of columns (<= kNarrowMaxN: the narrow kernel), so
    // that no tile row or column holds only a few useful elements ("Part 2",
    // section "Selecting Among Three Kernels": at 2049 the last column of
    // 128 x 256 tiles holds one useful column).
    auto tile_edges_plan = [&](Plan *t) -> bool {
        const int64_t em = in.M % kTileBM, en = in.N % kTileBN;
        if (em + en == 0 || em > kSkinnyMaxM || en > kNarrowMaxN) return false;
        const int64_t M0 = in.M - em, N0 = in.N - en;
        if (M0 < kTileBM || N0 < kTileBN) return false;
        PlanInput core = in;
        core.M = M0;
        core.N = N0;
        tile_plan(t, true);  // copies, tile fields of the whole product
        const double pack_us = (t->pack_a || t->pack_b)
                                   ? 2.0 * 4.0 * (double)pack_floats / kPackBytesPerUs + kPackFixedUs
                                   : 0.0;
        plan_grid(core, t, true, false, kTileModel, kNoScale);
        t->est_us += pack_us;
        t->edge_m = (int)em;
        t->edge_n = (int)en;
        if (em > 0)
            t->est_us += kChainedLaunchUs + (double)N0 * (double)in.K * 4.0 / kStreamBytesPerUs;
        if (en > 0)
            t->est_us += kChainedLaunchUs + (double)in.M * (double)in.K * 4.0 / kStreamBytesPerUs;
        t->reason = "tiles, thin edges on the skinny/narrow kernels";
        return true;
    };
    if (want == kVarTile || want == kVarStreamK) {
        if (!tma_ok && !packable) return -2;
        tile_plan(&p, want != kVarTile);
        *pl = p;
        return 0;
    }

    // Automatic ("Part 2", section "Selecting Among Three Kernels"): the
    // least estimated time among the tiled kernel (aligned operands, or
    // copies of them unless M <= 32, where copying B would double the bytes
    // moved), the mid-size kernel with 128-row tiles and, for M <= 64, with
    // 64-row tiles, the split-K kernel and the 64 x 64 kernel.
    Plan cand[9];
    int n = 0;
    cand[n] = p;
    plan_mid(in, &cand[n++], 128);
    if (in.N <= kNarrowMaxN) {
        cand[n] = p;
        plan_narrow(in, &cand[n++]);
    }
    if (ceil_div(in.M, kKsBM) * ceil_div(in.N, 64) <= INT32_MAX) {
        cand[n] = p;
        plan_ksplit(in, &cand[n++], 128);
        cand[n] = p;
        plan_ksplit(in, &cand[n++], 64);
    }
    if (ceil_div(in.M, kSmallBM) * ceil_div(in.N, kSmallBN) <= INT32_MAX) {
        cand[n] = p;
        plan_small(in, &cand[n++]);
    }
    if (in.M <= 64) {
        cand[n] = p;
        plan_mid(in, &cand[n++], 64);
    }
    if (tma_ok || (packable && in.M > kSkinnyMaxM)) {
        cand[n] = p;
        tile_plan(&cand[n++], true);
        cand[n] = p;
        if (tile_edges_plan(&cand[n])) ++n;
    }
    cand[n] = p;
    plan_generic(in, &cand[n]);
    cand[n++].reason = "64 x 64 tiles";
    int bi = 0;
    for (int i = 1; i < n; ++i)
        if (cand[i].est_us < cand[bi].est_us) bi = i;
    double alt = 0;
    for (int i = 0; i < n; ++i)
        if (i != bi && (alt == 0 || cand[i].est_us < alt)) alt = cand[i].est_us;
    cand[bi].alt_us = alt;
    *pl = cand[bi];
    return 0;
}

int describe_plan(const Plan &p, char *buf, size_t len) {
    return snprintf(buf, len,
                    "variant=%s tiles_m=%d tiles_n=%d kt=%d dp_tiles=%d sk_tiles=%d sk_share=%d "
                    "grid=%d group_m=%d c_vec4=%d m_tile=%d two_unit_ctas=%d pack_a=%d pack_b=%d "
                    "bm=%d bvec=%d ks_bn=%d edge_m=%d edge_n=%d narrow_nn=%d narrow_rows=%d avec=%d "
                    "cost=%.2f est_us=%.1f alt_us=%.1f reason=%s",
                    variant_name(p.variant), p.tiles_m, p.tiles_n, p.kt_total, p.dp_tiles,
                    p.sk_tiles, p.sk_share, p.grid, p.group_m, p.c_vec4, p.m_tile,
                    p.variant == kVarSkinny ? p.sk_two_units : 0, p.pack_a ? 1 : 0,
                    p.pack_b ? 1 : 0, p.mid_bm, p.b_vec, p.ks_bn, p.edge_m, p.edge_n, p.narrow_nn,
                    p.narrow_rows, p.a_vec, p.cost, p.est_us, p.alt_us,
                    p.reason ? p.reason : "");
}

}  // namespace sgemm
