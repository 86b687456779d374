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

// Per extra piece of a stream-K tile, in k-iterations of a tile: measured on
// GB300, 1024^3 with 6 pieces per tile (share 7) took 63.5 us against 61.4
// with 5 (share 8), one iteration less work for one piece more.
constexpr double kFixupCost = 1.5;
constexpr int64_t kSmallSlicesPerSm = 4;
// With the copy of an unaligned operand to pay for, the tiled kernel needs
// more work: measured, 1023 x 1025 x 513 (4.5 slices per SM) is faster on the
// 64 x 64 kernel and 1023^3 (6.7) through the copy.
constexpr int64_t kPackSlicesPerSm = 6;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

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
        default: return "?";
    }
}

static void plan_tile(const PlanInput &in, Plan *pl, bool allow_sk) {
    const int64_t G = in.num_sms > 0 ? in.num_sms : 1;
    const int64_t tm = ceil_div(in.M, kTileBM), tn = ceil_div(in.N, kTileBN);
    const int64_t T = tm * tn;
    const int64_t KT = ceil_div(in.K, kTileBK);
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
    best.reason = "whole tiles";

    const bool sk_fits = T * KT < (int64_t(1) << 30);
    if (allow_sk && sk_fits && (T % G != 0 || in.force_variant == kVarStreamK)) {
        const int64_t full = T / G;
        for (int64_t d = full; d >= 0 && d >= full - 1; --d) {
            const int64_t dp = d * G;
            const int64_t sk_tiles = T - dp;
            if (sk_tiles <= 0) continue;
            const int64_t total = sk_tiles * KT;
            int64_t share = ceil_div(total, G);
            const int64_t min_share = ceil_div(KT, 8);
            // Shares from the smallest the grid and the piece limit allow, a
            // little upward: a larger share can save a piece.
            int64_t last = share;
            if (in.force_splits > 0) {
                // As close to the requested split as the grid allows.
                const int64_t want = ceil_div(KT, in.force_splits);
                share = want > share ? want : share;
                last = share;
            } else {
                if (share < min_share) share = min_share;
                last = share + share / 2 + 2;
                if (last > KT) last = KT > share ? KT : share;
            }
            if (share < 1) share = 1;
            bool taken = false;
            for (int64_t sh = share; sh <= last; ++sh) {
                const int64_t ctas = ceil_div(total, sh);
                if (ctas > G) continue;
                // Most pieces any tile is cut into.
                const int64_t pieces = (KT + sh - 2) / sh + 1;
                const int64_t max_pieces = pieces < ctas ? pieces : ctas;
                const double cost = (double)d * KT + (double)sh +
                                    kFixupCost * (double)(max_pieces > 1 ? max_pieces - 1 : 0);
                if (cost < best.cost || (in.force_variant == kVarStreamK && !taken)) {
                    best.variant = kVarStreamK;
                    best.dp_tiles = (int)dp;
                    best.sk_tiles = (int)sk_tiles;
                    best.sk_share = (int)sh;
                    best.grid = (int)(dp > 0 ? G : ctas);
                    best.cost = cost;
                    best.reason = "stream-K tail";
                    taken = true;
                }
            }
            if (taken && in.force_variant == kVarStreamK) break;
        }
    }
    *pl = best;
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

    // M <= 16: every B element feeds at most 16 products, so the product is
    // bound by streaming B; a 128-row tile would spend 8x the multiply-adds.
    if (tma_ok && (want == kVarSkinny || (want < 0 && in.M <= kSkinnyMaxM))) {
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
            p.m_tile = in.M <= 8 ? 8 : 16;
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

    // A product with at most kSmallSlicesPerSm 128 x 256 x 32 tile slices per
    // SM leaves most SMs idle under the tiled kernel, or splits its few tiles
    // into pieces whose combination costs more than they balance; 64 x 64
    // tiles spread it over more SMs.  (Measured on GB300 over square sizes:
    // the 64 x 64 kernel wins up to 768^3, 2.8 slices per SM; the tiled
    // kernel from 1024^3, 6.7.)
    bool small = false, small_unaligned = false;
    if (want < 0) {
        const int64_t G = in.num_sms > 0 ? in.num_sms : 1;
        const int64_t slices = ceil_div(in.M, kTileBM) * ceil_div(in.N, kTileBN) *
                               ceil_div(in.K, kTileBK);
        small = slices <= kSmallSlicesPerSm * G;
        small_unaligned = slices <= kPackSlicesPerSm * G;
    }
    // Operands the TMA cannot map (a pointer or leading dimension off 16
    // bytes) are first copied to 16-byte-aligned rows when the product is
    // large enough for the tiled kernel to repay the copy; smaller products
    // (and the M <= 16 regime, where copying B would double the bytes moved)
    // take the bounds-checked 64 x 64 kernel.
    const int64_t pack_floats = (a_ok ? 0 : in.M * round_up4(in.K)) +
                                (b_ok ? 0 : in.K * round_up4(in.N));
    const bool packable = pack_floats < (int64_t(1) << 31);
    const bool pack = !tma_ok && packable &&
                      (want == kVarTile || want == kVarStreamK ||
                       (want < 0 && !small_unaligned && in.M > kSkinnyMaxM));
    if ((want == kVarTile || want == kVarStreamK) && !tma_ok && !pack) return -2;
    if (want == kVarGeneric || (want < 0 && ((!tma_ok && !pack) || small))) {
        p.variant = kVarGeneric;
        p.tiles_m = (int)ceil_div(in.M, kGenBM);
        p.tiles_n = (int)ceil_div(in.N, kGenBN);
        p.kt_total = (int)ceil_div(in.K, kGenBK);
        p.grid = p.tiles_m * p.tiles_n;
        p.cost = 0;
        p.reason = !tma_ok ? "operands not 16-byte aligned" : small ? "small product" : "forced";
        *pl = p;
        return 0;
    }
    p.pack_a = pack && !a_ok;
    p.pack_b = pack && !b_ok;
    p.lda_packed = p.pack_a ? round_up4(in.K) : in.lda;
    p.ldb_packed = p.pack_b ? round_up4(in.N) : in.ldb;
    plan_tile(in, &p, want != kVarTile);
    if (pack) p.reason = "operands copied to aligned rows";
    *pl = p;
    return 0;
}

int describe_plan(const Plan &p, char *buf, size_t len) {
    return snprintf(buf, len,
                    "variant=%s tiles_m=%d tiles_n=%d kt=%d dp_tiles=%d sk_tiles=%d sk_share=%d "
                    "grid=%d group_m=%d c_vec4=%d m_tile=%d two_unit_ctas=%d pack_a=%d pack_b=%d "
                    "cost=%.2f reason=%s",
                    variant_name(p.variant), p.tiles_m, p.tiles_n, p.kt_total, p.dp_tiles,
                    p.sk_tiles, p.sk_share, p.grid, p.group_m, p.c_vec4, p.m_tile,
                    p.variant == kVarSkinny ? p.sk_two_units : 0, p.pack_a ? 1 : 0,
                    p.pack_b ? 1 : 0, p.cost, p.reason ? p.reason : "");
}

}  // namespace sgemm
