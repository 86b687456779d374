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
//     to at most about five per tile (shares of at least a quarter of K):
//     finer splits cost more than they balance ("Part 2": up to 16 pieces
//     lost to cuBLAS; two to four worked).
#include "plan.h"

#include <stdio.h>

#include "kernels.h"

namespace sgemm {

namespace {

constexpr double kFixupCost = 0.5;  // per extra piece, in k-iterations of a tile

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(uint64_t addr) { return (addr & 15u) == 0; }

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
            const int64_t min_share = ceil_div(KT, 4);
            if (in.force_splits > 0) {
                // As close to the requested split as the grid allows.
                const int64_t want = ceil_div(KT, in.force_splits);
                share = want > share ? want : share;
            } else if (share < min_share) {
                share = min_share;
            }
            if (share < 1) share = 1;
            const int64_t ctas = ceil_div(total, share);
            if (ctas > G) continue;
            // Most pieces any tile is cut into.
            const int64_t pieces = (KT + share - 2) / share + 1;
            const int64_t max_pieces = pieces < ctas ? pieces : ctas;
            const double cost = (double)d * KT + (double)share +
                                kFixupCost * (double)(max_pieces > 1 ? max_pieces - 1 : 0);
            if (cost < best.cost || in.force_variant == kVarStreamK) {
                best.variant = kVarStreamK;
                best.dp_tiles = (int)dp;
                best.sk_tiles = (int)sk_tiles;
                best.sk_share = (int)share;
                best.grid = (int)(dp > 0 ? G : ctas);
                best.cost = cost;
                best.reason = "stream-K tail";
                if (in.force_variant == kVarStreamK) break;
            }
        }
    }
    *pl = best;
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

    const bool tma_ok = aligned16(in.a_addr) && aligned16(in.b_addr) && in.lda % 4 == 0 &&
                        in.ldb % 4 == 0 && in.lda < (int64_t(1) << 37) &&
                        in.ldb < (int64_t(1) << 37);
    int want = in.force_variant;
    if ((want == kVarTile || want == kVarStreamK || want == kVarSkinny) && !tma_ok) return -2;
    if (want == kVarSkinny && in.M > kSkinnyMaxM) return -3;

    // M <= 16: every B element feeds at most 16 products, so the product is
    // bound by streaming B; a 128-row tile would spend 8x the multiply-adds.
    if (tma_ok && (want == kVarSkinny || (want < 0 && in.M <= kSkinnyMaxM))) {
        // Persistent grid: every CTA the SMs hold at once.
        const int64_t G = (in.num_sms > 0 ? in.num_sms : 1) * kSkinnyCtasPerSm;
        const int64_t slabs = ceil_div(in.N, kSkinnyBN);
        const int64_t KT = ceil_div(in.K, kSkinnyBK);
        const int64_t total = slabs * KT;
        if (total < (int64_t(1) << 30)) {
            int64_t share = ceil_div(total, G);
            if (in.force_splits > 0) {
                const int64_t w = ceil_div(KT, in.force_splits);
                share = w > share ? w : share;
            }
            p.variant = kVarSkinny;
            p.m_tile = in.M <= 8 ? 8 : 16;
            p.slabs = (int)slabs;
            p.tiles_n = (int)slabs;
            p.tiles_m = 1;
            p.kt_total = (int)KT;
            p.sk_share = (int)share;
            p.grid = (int)ceil_div(total, share);
            p.c_vec4 = 0;
            p.cost = (double)share;
            p.reason = "small M: stream B once";
            *pl = p;
            return 0;
        }
    }

    // A product with fewer 128 x 256 x 32 tile slices than SMs leaves most
    // SMs idle under the tiled kernel, or splits its few tiles into pieces
    // whose combination costs more than they balance; 64 x 64 tiles spread
    // it over more SMs.
    bool small = false;
    if (want < 0 && tma_ok) {
        const int64_t G = in.num_sms > 0 ? in.num_sms : 1;
        const int64_t slices = ceil_div(in.M, kTileBM) * ceil_div(in.N, kTileBN) *
                               ceil_div(in.K, kTileBK);
        small = slices <= G;
    }
    if (want == kVarGeneric || (want < 0 && (!tma_ok || small))) {
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
    plan_tile(in, &p, want != kVarTile);
    *pl = p;
    return 0;
}

int describe_plan(const Plan &p, char *buf, size_t len) {
    return snprintf(buf, len,
                    "variant=%s tiles_m=%d tiles_n=%d kt=%d dp_tiles=%d sk_tiles=%d sk_share=%d "
                    "grid=%d group_m=%d c_vec4=%d m_tile=%d cost=%.2f reason=%s",
                    variant_name(p.variant), p.tiles_m, p.tiles_n, p.kt_total, p.dp_tiles,
                    p.sk_tiles, p.sk_share, p.grid, p.group_m, p.c_vec4, p.m_tile, p.cost,
                    p.reason ? p.reason : "");
}

}  // namespace sgemm
