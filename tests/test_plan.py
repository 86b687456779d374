"""Host-side planner checks (no GPU): variant choice, wave arithmetic and the
stream-K split, on a GPU described by its SM count (152 on GB300)."""
import math

import numpy as np
import pytest

import dense_fp32_sgemm_gb300 as sg

SMS = 152


@pytest.fixture(scope="module", autouse=True)
def built():
    sg.build()
    sg.set_plan_override(-1, 0)
    yield
    sg.set_plan_override(-1, 0)


def ceil4(x):
    return (x + 3) // 4 * 4


def plan(M, N, K, aligned_ld=True, **kw):
    if aligned_ld:
        kw.setdefault("lda", ceil4(max(K, 1)))
        kw.setdefault("ldb", ceil4(max(N, 1)))
        kw.setdefault("ldc", ceil4(max(N, 1)))
    kw.setdefault("a_addr", 1 << 20)
    kw.setdefault("b_addr", 2 << 20)
    kw.setdefault("c_addr", 3 << 20)
    kw.setdefault("num_sms", SMS)
    return sg.plan_describe(M, N, K, **kw)


def ints(p, *keys):
    return [int(p[k]) for k in keys]


def test_quick_returns():
    assert plan(0, 5, 7)["variant"] == "none"
    assert plan(5, 0, 7)["variant"] == "none"
    assert plan(5, 6, 0)["variant"] == "scale"


def test_misaligned_operands():
    # Unaligned rows (lda = ldb = 1023): the mid-size kernel reads them with
    # 4-byte copies, so no copy pass is planned ...
    p = plan(1023, 1023, 1023, aligned_ld=False)
    assert p["variant"] in ("mid", "ksplit") and ints(p, "bvec", "pack_a", "pack_b") == [1, 0, 0]
    # (one wave of 64 x 128 tiles: the split-K kernel; measured 37.9 us against
    # 45.5 on the 64 x 64 kernel and 49.9 on the mid-size one)
    p = plan(1023, 1025, 513, aligned_ld=False)
    assert p["variant"] == "ksplit" and ints(p, "bvec", "pack_a", "pack_b") == [1, 0, 0]
    # ... B aligned keeps its 16-byte copies
    p = plan(1023, 1024, 1023, lda=1023)
    assert p["variant"] in ("mid", "ksplit") and p["bvec"] == "4"
    # M <= 16 with an unaligned operand: not the skinny kernel (TMA), and the
    # tiled kernel's copy of B is never considered
    p = plan(16, 8192, 8191, aligned_ld=False)
    assert p["variant"] == "mid" and ints(p, "pack_a", "pack_b") == [0, 0]
    # forcing the tiled kernel on unaligned operands copies only the
    # unaligned one to aligned rows
    sg.set_plan_override(sg.VARIANT_TILE, 0)
    try:
        p = plan(300, 400, 500, b_addr=(2 << 20) + 8)
        assert p["variant"] == "tile" and ints(p, "pack_a", "pack_b") == [0, 1]
        p = plan(2048, 2048, 2048, a_addr=(1 << 20) + 4)
        assert ints(p, "pack_a", "pack_b") == [1, 0]
    finally:
        sg.set_plan_override(-1, 0)


def test_2048_cube_uses_stream_k_over_all_sms():
    # 128 tiles of 128 x 256 would fill 128 of 152 SMs (one partial wave);
    # stream-K shares their 128 * 64 k-iterations evenly.
    p = plan(2048, 2048, 2048)
    assert p["variant"] == "streamk"
    tm, tn, kt, dp, sk, share, grid = ints(p, "tiles_m", "tiles_n", "kt", "dp_tiles",
                                           "sk_tiles", "sk_share", "grid")
    assert (tm, tn, kt) == (16, 8, 64)
    assert dp == 0 and sk == 128
    assert share == math.ceil(128 * 64 / SMS)
    assert grid == SMS
    assert float(p["cost"]) < 64  # beats one whole tile per SM


def test_4092_cube_keeps_full_waves_whole():
    p = plan(4092, 4092, 4092, beta=2.0)
    tm, tn, kt, dp, sk = ints(p, "tiles_m", "tiles_n", "kt", "dp_tiles", "sk_tiles")
    assert (tm, tn, kt) == (32, 16, 128)
    assert p["variant"] == "streamk"
    assert dp % SMS == 0 and dp + sk == tm * tn
    assert float(p["cost"]) < math.ceil(tm * tn / SMS) * kt


def test_exact_waves_stay_data_parallel():
    # 152 * 2 tiles: two full waves, nothing to balance.  (K long enough that
    # the tiled kernel is the fastest: at K = 512 the mid-size kernel's time
    # model wins.)
    p = plan(128 * 19, 256 * 16, 2048)
    assert p["variant"] == "tile"
    assert ints(p, "dp_tiles", "grid") == [304, SMS]


def tile_invariants(p, M, N, K, forced_sk=False):
    tm, tn, kt, dp, sk, share, grid = ints(p, "tiles_m", "tiles_n", "kt", "dp_tiles",
                                           "sk_tiles", "sk_share", "grid")
    T = tm * tn
    em, en = ints(p, "edge_m", "edge_n")  # rows and columns left to other kernels
    assert 0 <= em <= 32 and 0 <= en <= 4
    assert tm == math.ceil((M - em) / 128) and tn == math.ceil((N - en) / 256)
    assert kt == math.ceil(K / 32)
    assert dp + sk == T
    assert 1 <= grid <= SMS
    if sk:
        assert dp % SMS == 0
        # every stream-K iteration is owned by some CTA of the grid
        assert share * grid >= sk * kt
        # pieces per tile stay within what the idle ring combines (nine)
        assert share >= math.ceil(kt / 8)
        assert (kt + share - 2) // share + 1 <= 9
        # an automatic stream-K tail splits some tile: a share of whole tiles
        # is the whole-tile plan, which carries its own cost per wave
        if not forced_sk:
            assert share % kt != 0
    # the chosen cost never exceeds the data-parallel cost (a forced stream-K
    # split takes the first candidate)
    if not forced_sk:
        assert float(p["cost"]) <= math.ceil(T / SMS) * kt + 1e-9


def small_invariants(p, M, N, K):
    # one 32 x 32 tile per CTA over the whole K in 64-k slices
    tm, tn, kt, dp, sk, grid = ints(p, "tiles_m", "tiles_n", "kt", "dp_tiles", "sk_tiles", "grid")
    assert tm == math.ceil(M / 32) and tn == math.ceil(N / 32) and kt == math.ceil(K / 64)
    assert dp == tm * tn == grid and sk == 0 and p["bvec"] in ("1", "4")


def narrow_invariants(p, M, N, K):
    # N <= 4; contiguous row ranges covering M once, at most two CTAs per SM
    grid, rows, nn = ints(p, "grid", "narrow_rows", "narrow_nn")
    assert N <= 4 and nn == (1 if N == 1 else 2 if N == 2 else 4)
    assert 1 <= grid <= 2 * SMS
    assert rows * grid >= M and rows * (grid - 1) < M


def ksplit_invariants(p, M, N, K):
    # one 64 x bn tile per CTA (bn 128 or 64) over the whole K in 64-k slices
    tm, tn, kt, dp, sk, grid, bn = ints(p, "tiles_m", "tiles_n", "kt", "dp_tiles", "sk_tiles",
                                        "grid", "ks_bn")
    assert p["bm"] == "64" and p["bvec"] in ("1", "4") and bn in (128, 64)
    assert tm == math.ceil(M / 64) and tn == math.ceil(N / bn) and kt == math.ceil(K / 64)
    assert dp == tm * tn == grid and sk == 0


def mid_invariants(p, M, N, K):
    bm = int(p["bm"])
    assert bm in (128, 64)
    cps = 2 if bm == 128 else 4
    tm, tn, kt, dp, sk, share, grid = ints(p, "tiles_m", "tiles_n", "kt", "dp_tiles",
                                           "sk_tiles", "sk_share", "grid")
    T = tm * tn
    assert tm == math.ceil(M / bm) and tn == math.ceil(N / 128) and kt == math.ceil(K / 16)
    assert dp + sk == T
    assert 1 <= grid <= SMS * cps
    if sk:
        assert dp % (SMS * cps) == 0
        assert share * grid >= sk * kt
        assert (kt + share - 2) // share + 1 <= 9


@pytest.mark.parametrize("M,N,K", [(128, 128, 32 * 700), (1000, 3000, 231), (8192, 6144, 2048),
                                   (17, 8192, 8192), (4000, 300, 20000), (129, 257, 32 * 160),
                                   (40, 1, 100000), (5000, 5000, 1)])
def test_plan_invariants(M, N, K):
    # The tiled kernel forced whole, forced stream-K, and the mid-size kernel
    # forced with either tile height each cover the work; the automatic plan
    # is one of them or the 64 x 64 kernel.
    for variant in (sg.VARIANT_TILE, sg.VARIANT_STREAMK):
        sg.set_plan_override(variant, 0)
        try:
            tile_invariants(plan(M, N, K), M, N, K, forced_sk=variant == sg.VARIANT_STREAMK)
        finally:
            sg.set_plan_override(-1, 0)
    for variant in (sg.VARIANT_MID, sg.VARIANT_MID64):
        sg.set_plan_override(variant, 0)
        try:
            mid_invariants(plan(M, N, K), M, N, K)
        finally:
            sg.set_plan_override(-1, 0)
    for variant in (sg.VARIANT_KSPLIT, sg.VARIANT_KSPLIT64):
        sg.set_plan_override(variant, 0)
        try:
            ksplit_invariants(plan(M, N, K), M, N, K)
        finally:
            sg.set_plan_override(-1, 0)
    sg.set_plan_override(sg.VARIANT_SMALL, 0)
    try:
        small_invariants(plan(M, N, K), M, N, K)
    finally:
        sg.set_plan_override(-1, 0)
    p = plan(M, N, K)
    if p["variant"] in ("tile", "streamk"):
        tile_invariants(p, M, N, K)
    elif p["variant"] == "mid":
        mid_invariants(p, M, N, K)
    elif p["variant"] == "ksplit":
        ksplit_invariants(p, M, N, K)
    elif p["variant"] == "skinny":
        assert M <= 32
    elif p["variant"] == "narrow":
        narrow_invariants(p, M, N, K)
    elif p["variant"] == "small":
        small_invariants(p, M, N, K)
    else:
        assert p["variant"] == "generic"


@pytest.mark.parametrize("M,N,K", [(64, 64, 64), (129, 257, 33), (300, 520, 64), (128, 128, 128),
                                   (256, 256, 256), (512, 512, 512), (32, 32, 32)])
def test_small_products_take_the_32x32_kernel(M, N, K):
    # Measured on GB300: 32 x 32 tiles spread small products over the most
    # SMs, four CTAs to an SM (128^3: 8.2 us against 12.3 on 64 x 64 split-K
    # tiles and 12.6 on the 64 x 64 kernel; 512^3: 18.4 against 22.5).
    p = plan(M, N, K)
    assert p["variant"] == "small"
    small_invariants(p, M, N, K)


@pytest.mark.parametrize("M,N,K", [(640, 640, 640), (768, 768, 768), (128, 4096, 1024)])
def test_small_products_take_64x64_split_k_tiles(M, N, K):
    # From about four 32 x 32 tiles per SM, 64 x 64 tiles with eight warps
    # splitting K (768^3: 28.7 us against 38.9 on 32 x 32 tiles and 34.8 on
    # the mid-size kernel).
    p = plan(M, N, K)
    assert p["variant"] == "ksplit" and p["ks_bn"] == "64"
    ksplit_invariants(p, M, N, K)


@pytest.mark.parametrize("M,N,K", [(896, 896, 896), (100, 5000, 3000), (1400, 1300, 512)])
def test_mid_size_products_take_the_mid_kernel(M, N, K):
    # 128 x 128 tiles with a stream-K tail, where 64 x 64 tiles would take two
    # waves (896^3: 47.1 us against 49.1 on the 64 x 128 split-K kernel).
    p = plan(M, N, K)
    assert p["variant"] == "mid" and p["bm"] == "128"


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 512), (1024, 1152, 512), (1024, 1024, 1024)])
def test_one_wave_of_64x128_tiles_takes_the_split_k_kernel(M, N, K):
    # 128-144 tiles of 64 x 128 fill the SMs in one wave with no partial sums
    # in global memory (1024^3: 54.8 us against 59.4 on the mid-size kernel,
    # 60.4 on the tiled kernel with a stream-K tail).
    p = plan(M, N, K)
    assert p["variant"] == "ksplit" and p["ks_bn"] == "128"
    ksplit_invariants(p, M, N, K)


@pytest.mark.parametrize("M", [33, 48, 64])
def test_short_products_take_64_row_tiles(M):
    # 33 <= M <= 64: 64-row tiles waste at most 31 rows a tile (64 x 8192 x
    # 8192: 173.5 us against 283 on the 128 x 256 tiled kernel).
    p = plan(M, 8192, 8192)
    assert p["variant"] == "mid" and p["bm"] == "64"


@pytest.mark.parametrize("M", [17, 24, 32])
def test_up_to_32_rows_stream_b_once(M):
    # 17 <= M <= 32 with aligned operands: the skinny kernel with a 32-row A
    # tile (two groups of warps each summing 16 rows); unaligned operands
    # take 64-row mid-size tiles.
    p = plan(M, 8192, 8192)
    assert p["variant"] == "skinny" and p["m_tile"] == "32"
    p = plan(M, 8192, 8191, aligned_ld=False)
    assert p["variant"] == "mid" and p["bm"] == "64"


@pytest.mark.parametrize("M,N,K", [(2048, 2048, 2048), (4092, 4092, 4092), (8192, 6144, 2048),
                                   (3072, 3072, 3072), (8192, 256, 8192)])
def test_large_aligned_products_take_the_tiled_kernel(M, N, K):
    p = plan(M, N, K)
    assert p["variant"] in ("tile", "streamk")


def test_estimates_are_reported_and_ordered():
    # The plan reports its estimate and the best other candidate's.
    p = plan(2048, 2048, 2048)
    est, alt = float(p["est_us"]), float(p["alt_us"])
    assert 200 < est < 350 and alt >= est


def test_forced_split_count():
    sg.set_plan_override(sg.VARIANT_STREAMK, 3)
    try:
        p = plan(256, 512, 960)
        assert p["variant"] == "streamk"
        kt, share = ints(p, "kt", "sk_share")
        assert share == math.ceil(kt / 3)
        # A split too fine for the grid is coarsened until every CTA has one range.
        sg.set_plan_override(sg.VARIANT_STREAMK, 16)
        p = plan(4096, 4096, 4096)
        tm, tn, kt, dp, sk, share, grid = ints(p, "tiles_m", "tiles_n", "kt", "dp_tiles",
                                               "sk_tiles", "sk_share", "grid")
        assert p["variant"] == "streamk" and share * grid >= sk * kt
    finally:
        sg.set_plan_override(-1, 0)


def test_forced_generic():
    sg.set_plan_override(sg.VARIANT_GENERIC, 0)
    try:
        assert plan(512, 512, 512)["variant"] == "generic"
    finally:
        sg.set_plan_override(-1, 0)


UNIT_END = 6  # positions a range pays for each slab boundary it crosses


@pytest.mark.parametrize("M,N,K", [(16, 8192, 8192), (1, 4096, 4096), (9, 3000, 720),
                                   (8, 100000, 64), (16, 10240, 320), (32, 8192, 8192),
                                   (20, 3000, 800)])
def test_skinny_plan(M, N, K):
    # M <= 16: the streaming kernel over 256-column slabs and 32-row positions,
    # the (slab, k) plane cut into contiguous ranges, one per CTA of a
    # one-CTA-per-SM grid, balanced in time: the budget is the smallest that
    # fits the grid, at most one unit end above the even share.
    p = plan(M, N, K)
    assert p["variant"] == "skinny"
    slabs, kt, budget, grid, m_tile, two = ints(p, "tiles_n", "kt", "sk_share", "grid", "m_tile",
                                                "two_unit_ctas")
    total = slabs * kt
    assert slabs == math.ceil(N / 256) and kt == math.ceil(K / 32)
    assert m_tile == (8 if M <= 8 else 16 if M <= 16 else 32)
    assert 1 <= grid <= SMS
    assert budget >= math.ceil(total / SMS)
    if kt >= 32:
        # long slabs: a range crosses at most one boundary, so the budget is
        # at most one unit end above the even share
        assert budget <= math.ceil(total / SMS) + UNIT_END + 1
        assert 0 <= two <= min(grid, slabs - 1)


def test_skinny_16x8192x8192_split():
    # 32 slabs x 256 positions over 152 CTAs: budget 55; the 24 ranges that
    # cross a slab boundary hold 49 positions and pay for one more unit end.
    p = plan(16, 8192, 8192)
    assert ints(p, "tiles_n", "kt", "sk_share", "grid", "two_unit_ctas") == [32, 256, 55, 152, 24]


@pytest.mark.parametrize("M,N,K,share,grid", [(768, 768, 4096, 16, 144), (640, 640, 8192, 32, 120)])
def test_deep_products_with_few_tiles_split_finer(M, N, K, share, grid):
    # The tiled kernel on 18 and 15 tiles: shares of an eighth of K keep most
    # SMs busy while each tile stays within nine pieces.
    sg.set_plan_override(sg.VARIANT_STREAMK, 0)
    try:
        p = plan(M, N, K)
    finally:
        sg.set_plan_override(-1, 0)
    assert p["variant"] == "streamk"
    assert ints(p, "sk_share", "grid") == [share, grid]


# ----- the 3xTF32 entry point's choices (sgemm_plan_describe_3xtf32) --------

def x3(M, N, K, **kw):
    kw.setdefault("lda", K)
    kw.setdefault("a_addr", 1 << 20)
    kw.setdefault("num_sms", SMS)
    return sg.plan_describe_3xtf32(M, N, K, **kw)


@pytest.mark.parametrize("M,N,K", [(16, 8192, 8192), (1000, 1000, 63), (1, 5, 7)])
def test_3xtf32_short_or_skinny_products_take_the_ffma_kernels(M, N, K):
    assert x3(M, N, K) == {"path": "ffma"}


@pytest.mark.parametrize("M,N,K,tile_n,splits,cps,a_in", [
    # one wave of 240-wide tiles (144 CTAs), one CTA per SM
    (2048, 2048, 2048, 240, 1, 1, 0),
    # 608 tiles of 224: exactly four waves; two CTAs per SM
    (4092, 4092, 4092, 224, 1, 2, 0),
    # large output with A rows on 128-byte lines: A split in the kernel
    (8192, 8192, 8192, 256, 1, 2, 1),
    # deep products with few tiles: cut into K ranges
    (768, 768, 4096, 128, 4, 1, 0),
    (1024, 1024, 8192, 176, 3, 1, 0),
])
def test_3xtf32_plans(M, N, K, tile_n, splits, cps, a_in):
    p = x3(M, N, K)
    assert p["path"] == "tensor"
    assert [int(p[k]) for k in ("tile_n", "splits", "ctas_per_sm", "a_in_kernel")] == \
        [tile_n, splits, cps, a_in]
    tiles = math.ceil(M / 128) * math.ceil(N / tile_n)
    assert int(p["ctas"]) == tiles * splits
    # at least 16 K slices per range
    assert math.ceil(int(p["kt"]) / splits) >= 16 or splits == 1


@pytest.mark.parametrize("M,N", [(300, 520), (2048, 2048), (4092, 4092), (777, 6000), (130, 100)])
def test_3xtf32_tile_width_costs_no_more_waves_than_the_widest(M, N):
    # The chosen width never needs more waves x (width + 32) than 256.
    p = x3(M, N, 1024)
    bn = int(p["tile_n"])
    assert 64 <= bn <= 256 and bn % 16 == 0
    def cost(w):
        return math.ceil(math.ceil(M / 128) * math.ceil(N / w) / SMS) * (w + 32)
    assert cost(bn) <= cost(256)


def test_3xtf32_a_split_needs_aligned_rows():
    assert x3(8192, 8192, 8192, a_addr=(1 << 20) + 64)["a_in_kernel"] == "0"
    assert x3(8192, 8192, 8190, lda=8190)["a_in_kernel"] == "0"


def test_3xtf32_config_forces_forms():
    sg.set_3xtf32_config(32, True, 4, 0)
    try:
        p = x3(2048, 2048, 4096)
        assert (p["bk"], p["stages"], p["ctas_per_sm"], p["a_in_kernel"], p["splits"]) == \
            ("32", "2", "1", "1", "4")
    finally:
        sg.set_3xtf32_config(16, None)


def _random_shapes(seed, count):
    rng = np.random.default_rng(seed)
    return [(int(rng.integers(1, 20000)), int(rng.integers(1, 20000)), int(rng.integers(1, 40000)))
            for _ in range(count)]


def test_random_plans_cover_the_work():
    # Over many seeded shapes the FFMA plan covers every k-iteration of every
    # tile exactly, keeps stream-K tiles within nine pieces, and never costs
    # more than whole tiles; skinny ranges cover every (slab, k) position.
    for M, N, K in _random_shapes(11, 300):
        p = plan(M, N, K)
        v = p["variant"]
        assert v in ("tile", "streamk", "mid", "ksplit", "narrow", "small", "generic", "skinny",
                     "scale", "none"), (M, N, K, v)
        if v in ("tile", "streamk"):
            tile_invariants(p, M, N, K)
        elif v == "mid":
            mid_invariants(p, M, N, K)
        elif v == "ksplit":
            ksplit_invariants(p, M, N, K)
        elif v == "narrow":
            narrow_invariants(p, M, N, K)
        elif v == "small":
            small_invariants(p, M, N, K)
        elif v == "skinny":
            assert M <= 32
            slabs, kt, grid = ints(p, "tiles_n", "kt", "grid")
            assert 1 <= grid <= SMS and slabs == math.ceil(N / 256)


def test_random_3xtf32_plans():
    # The tensor-core plan: widths in [64, 256] in steps of 16, K ranges of at
    # least 16 slices, CTA count = tiles x ranges, two CTAs per SM only past
    # one wave.
    for M, N, K in _random_shapes(12, 300):
        p = x3(M, N, K)
        if K < 64 or M <= 16:
            assert p == {"path": "ffma"}
            continue
        bn, splits, kt, ctas, cps = (int(p[k]) for k in ("tile_n", "splits", "kt", "ctas",
                                                         "ctas_per_sm"))
        assert 64 <= bn <= 256 and bn % 16 == 0
        assert 1 <= splits <= 8
        if splits > 1:
            kps = math.ceil(kt / splits)
            assert kps >= 16 and (splits - 1) * kps < kt
        assert ctas == math.ceil(M / 128) * math.ceil(N / bn) * splits
        assert cps == (2 if ctas > SMS else 1)


# ----- narrow N and thin edges -------------------------------------------------

@pytest.mark.parametrize("M,N,K", [(8192, 1, 8192), (8192, 4, 8192), (100000, 1, 1000),
                                   (2049, 3, 2049), (40, 2, 100)])
def test_narrow_products_stream_a_once(M, N, K):
    # N <= 4 (and M above the skinny kernel's 32 rows): a warp per row of A.
    p = plan(M, N, K)
    assert p["variant"] == "narrow"
    narrow_invariants(p, M, N, K)


@pytest.mark.parametrize("M,N,K,em,en", [(2049, 2049, 2049, 1, 1), (4097, 4097, 4097, 1, 1),
                                         (2050, 2052, 1000, 2, 4), (4096, 4097, 4096, 0, 1),
                                         (2080, 4096, 4096, 32, 0)])
def test_thin_edges_leave_the_tiles_whole(M, N, K, em, en):
    # A last tile row of at most 32 rows goes to the skinny kernel and a last
    # tile column of at most 4 columns to the narrow one; the tiled kernel
    # covers the rest with whole 128 x 256 tiles.
    p = plan(M, N, K)
    assert p["variant"] in ("tile", "streamk")
    assert ints(p, "edge_m", "edge_n") == [em, en]
    tm, tn = ints(p, "tiles_m", "tiles_n")
    assert tm * 128 == M - em and tn * 256 == N - en


def test_forced_tiles_keep_their_edges():
    # The forced tiled variants cover the whole product themselves.
    sg.set_plan_override(sg.VARIANT_STREAMK, 0)
    try:
        p = plan(2049, 2049, 2049)
    finally:
        sg.set_plan_override(-1, 0)
    assert ints(p, "edge_m", "edge_n", "tiles_m", "tiles_n") == [0, 0, 17, 9]
