// Host-side planner: picks the kernel variant and the work split for one
// SGEMM call.  Pure host code (no CUDA calls), so it can be exercised on a
// machine without a GPU through sgemm_plan_describe().
#pragma once

#include <stddef.h>
#include <stdint.h>

namespace sgemm {

enum Variant : int {
    kVarNone = -2,      // nothing to do (M == 0 or N == 0)
    kVarScale = -3,     // alpha == 0 or K == 0: C = beta * C
    kVarGeneric = 0,
    kVarTile = 1,       // data-parallel only
    kVarStreamK = 2,    // data-parallel waves + stream-K tail
    kVarSkinny = 3,
    kVarMid = 4,        // mid-size kernel, bm x 128 tiles (bm = 128 when forced)
    kVarMid64 = 5,      // forced: the mid-size kernel with 64 x 128 tiles
    kVarKsplit = 6,     // split-K inside the CTA: 64 x 128 tiles, one per CTA
    kVarNarrow = 7,     // N <= kNarrowMaxN: a warp per row of A
    kVarKsplit64 = 8,   // forced: the split-K kernel with 64 x 64 tiles
    kVarSmall = 9,      // 32 x 32 tiles, split K inside the CTA, small products
};

struct PlanInput {
    int64_t M, N, K, lda, ldb, ldc;
    uint64_t a_addr, b_addr, c_addr;
    float alpha, beta;
    int num_sms;
    int force_variant;  // -1 = automatic
    int force_splits;   // 0 = automatic
};

struct Plan {
    int variant;
    // tile / stream-K
    int tiles_m, tiles_n, kt_total;
    int dp_tiles, sk_tiles, sk_share;
    int group_m;
    int grid;
    int c_vec4;
    // skinny: CTA c takes positions [sk_starts[c], sk_starts[c + 1])
    int m_tile, slabs;
    int sk_starts[161];
    int sk_two_units;  // CTAs whose range crosses a slab boundary
    // mid-size and split-K kernels: tile height (128 or 64) and B copy width
    // in floats (4 or 1)
    int mid_bm, b_vec;
    // split-K kernel: tile width (128 or 64)
    int ks_bn;
    // estimated time of the chosen plan (microseconds) and of the best other
    // candidate considered (0 when there was none)
    double est_us, alt_us;
    // tiled kernel: the last edge_m rows (<= 32, the skinny kernel) and the
    // last edge_n columns (<= kNarrowMaxN, the narrow kernel) of C are left
    // to other kernels; the tile counts cover the rest
    int edge_m, edge_n;
    // narrow kernel: columns it is built for (1, 2, 4), rows per CTA, and
    // A's load width in floats (4 or 1)
    int narrow_nn, narrow_rows, a_vec;
    // operands copied to 16-byte-aligned rows first (leading dimensions after the copy)
    bool pack_a, pack_b;
    int64_t lda_packed, ldb_packed;
    double cost;  // estimated busiest-SM work, in k-iterations of one tile
    const char *reason;
};

// Returns 0 and fills `out`, or a negative value for arguments no variant
// can take (the caller has validated sizes already).
int make_plan(const PlanInput &in, Plan *out);

// The narrow kernel's grid over M rows: CTAs and the rows each owns.
void narrow_grid(int64_t M, int num_sms, int *grid, int *rows);

// Writes a one-line key=value description of `plan`.
int describe_plan(const Plan &plan, char *buf, size_t len);

const char *variant_name(int variant);

}  // namespace sgemm
