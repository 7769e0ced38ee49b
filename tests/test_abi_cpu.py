"""CPU-side checks of the C ABI and the host logic the kernels share: the
library builds and exports every entry point declared in include/*.h, the
configuration choice and its argument checks, the grouped raster scheduler,
the 128-byte swizzle map, and the stage byte count -- each against values the
pages print (tests/golden/) or against properties that must hold.
"""
import glob
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def b():
    from tma_pipelined_tensor_fp16_gb300 import build, binding
    build.build()
    return binding


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"^TMAGEMM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, re.M)
    return sorted(set(names))


def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split("=", 1)
            vals[k.strip()] = v.strip()
    return vals


def test_library_exports_every_declared_symbol(b):
    declared = _declared_functions()
    assert len(declared) >= 13
    out = subprocess.run(["nm", "-D", "--defined-only", b.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (\w+)$", out, re.M))
    missing = [n for n in declared if n not in exported]
    assert not missing, missing
    lib = b.lib()
    for n in declared:
        assert getattr(lib, n) is not None


def test_create_plan_without_device_reports_no_device(b):
    assert not b.gemm_create_plan(256, 256, 256, b.GEMM_OUT_F32)
    assert b.gemm_last_status() == b.GEMM_ERR_NO_DEVICE
    assert "device" in b.last_error()


@pytest.mark.parametrize("args,status", [
    ((0, 8, 8, 0), 1), ((8, -1, 8, 0), 1), ((8, 8, 8, 7), 1),
    ((8, 8, 12, 0), 2),        # K not a multiple of 8 (16-byte TMA stride)
    ((8, 6, 8, 0), 2),         # N*4 bytes not a multiple of 16
    ((8, 12, 8, 1), 2),        # N*2 bytes not a multiple of 16
    ((8, 12, 8, 0), 0),        # N*4 = 48 bytes: fine for fp32 output
    # the largest sizes the ABI takes (each below 2^31), and one past them
    ((2 ** 31 - 1, 8, 8, 0), 0), ((2 ** 31, 8, 8, 0), 1),
    ((8, 2 ** 31 - 8, 8, 0), 0), ((8, 2 ** 31 + 8, 8, 0), 1),
    ((8, 8, 2 ** 31 - 8, 0), 0), ((8, 8, 2 ** 31 + 8, 0), 1),
    # legal sizes whose tile count does not fit the schedule's 31-bit indices
    ((2 ** 31 - 8, 2 ** 31 - 8, 8, 1), 2),
])
def test_argument_checks(b, args, status):
    st, _ = b.gemm_select_config(*args)
    assert st == status, b.last_error()
    # plan creation reports shape errors before looking for a device
    if status:
        assert not b.gemm_create_plan(*args)
        assert b.gemm_last_status() == status


def test_depth_that_does_not_fit_is_rejected(b):
    st, _ = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(
        variant="persistent", pipe_depth=5, block_n=256))
    assert st == b.GEMM_ERR_UNSUPPORTED and "does not fit" in b.last_error()
    st, c = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(
        variant="persistent", pipe_depth=4, block_n=256))
    assert st == 0 and c.smem_bytes <= 232448


def test_headline_configuration(b):
    st, c = b.gemm_select_config(8192, 8192, 8192, 1)
    assert st == 0
    assert c.variant == b.GEMM_VAR_DYNAMIC_2CTA
    assert (c.block_m, c.block_n, c.block_k) == (256, 256, 128)
    assert c.pipe_depth == 3 and c.grid == 2048 and c.threads == 192
    assert c.num_tiles == 1024 and c.k_blocks == 128 and c.tmem_cols == 512
    assert (c.dp_tiles, c.sk_tiles, c.workspace_bytes) == (1024, 0, 0)
    # both CTAs' A and half-B tiles, two 64-wide K blocks each
    assert c.tx_bytes == 2 * 2 * (128 * 64 + 128 * 64) * 2
    # an explicit ring depth keeps stages of one 64-wide block
    st, c = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(pipe_depth=6))
    assert st == 0 and (c.block_k, c.pipe_depth) == (64, 6)
    # a grid size or stream-K keeps the static pair schedule
    for o in ({"grid": 152}, {"stream_k": "on"}):
        st, c = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(**o))
        assert st == 0 and c.variant == b.GEMM_VAR_PERSISTENT_2CTA and c.grid == 152
    st, c = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(variant="persistent"))
    assert st == 0 and (c.block_m, c.block_n, c.pipe_depth, c.num_tiles) == (128, 256, 4, 2048)


@pytest.mark.parametrize("M,N,K,dt,variant,bn", [(256, 256, 256, 0, 5, 64),
                                                 (4096, 4096, 4096, 1, 8, 224),
                                                 (8192, 8192, 8192, 1, 8, 256),
                                                 (4000, 3000, 5000, 0, 8, 224),
                                                 (4000, 3000, 4992, 0, 8, 224),
                                                 (8192, 8192, 8200, 1, 8, 256),
                                                 (64, 16384, 16384, 1, 5, 128),
                                                 (128, 65536, 64, 1, 5, 256)])
def test_auto_variant_choice(b, M, N, K, dt, variant, bn):
    st, c = b.gemm_select_config(M, N, K, dt)
    assert st == 0 and c.variant == variant and c.block_n == bn


def test_pair_variant_constraints(b):
    for bn, dt, ok in [(128, 1, True), (160, 1, True), (192, 1, True), (224, 1, True),
                       (160, 0, True), (224, 0, True), (100, 0, False), (64, 0, False)]:
        st, c = b.gemm_select_config(1024, 1024, 64, dt, b.make_options(variant="persistent_2cta",
                                                                         block_n=bn))
        assert (st == 0) == ok, (bn, dt)
        if ok:
            assert c.block_n == bn and c.block_m == 256
            ks = c.block_k // 64  # K blocks of 64 per stage (auto: 2)
            assert c.tx_bytes == 2 * ks * (128 * 64 + (bn // 2) * 64) * 2
            assert c.tmem_cols >= 2 * bn and c.tmem_cols & (c.tmem_cols - 1) == 0
    st, c = b.gemm_select_config(1024, 1024, 64, 1, b.make_options(variant="persistent_2cta",
                                                                    grid=7))
    assert st == 0 and c.grid == 6  # whole clusters of two
    st, _ = b.gemm_select_config(1024, 1024, 64, 1, b.make_options(variant="persistent_2cta",
                                                                    block_n=256, pipe_depth=7))
    assert st == b.GEMM_ERR_UNSUPPORTED
    st, c = b.gemm_select_config(1024, 1024, 64, 1, b.make_options(variant="persistent_2cta",
                                                                    block_n=128, pipe_depth=8))
    assert st == 0  # 24 KB stages: eight fit


def test_dynamic_pair_configuration(b):
    # One cluster per pair tile; the clusters that run cancel the others
    # ("GEMM II -- pipelining with TMA", Step 6: cluster launch control).
    st, c = b.gemm_select_config(8192, 8192, 8192, 1,
                                 b.make_options(variant="dynamic_2cta", stream_k="off"))
    assert st == 0, b.last_error()
    assert c.variant == b.GEMM_VAR_DYNAMIC_2CTA
    assert (c.block_m, c.block_n, c.pipe_depth, c.threads, c.tmem_cols) == (256, 256, 3, 192, 512)
    assert c.grid == 2 * c.num_tiles == 2048
    assert (c.dp_tiles, c.sk_tiles, c.workspace_bytes) == (1024, 0, 0)
    assert c.smem_bytes <= 232448
    st, c = b.gemm_select_config(4000, 3000, 5000, 0, b.make_options(variant="dynamic_2cta"))
    assert st == 0 and c.block_n == 224 and c.grid == 2 * c.num_tiles
    st, _ = b.gemm_select_config(8192, 8192, 8192, 1,
                                 b.make_options(variant="dynamic_2cta", grid=152))
    assert st == b.GEMM_ERR_INVALID_ARG and "grid" in b.last_error()
    st, c = b.gemm_select_config(8192, 8192, 8192, 1,
                                 b.make_options(variant="dynamic_2cta", stream_k="on"))
    assert st == 0 and (c.dp_tiles, c.sk_tiles, c.sk_max_contrib) == (988, 36, 2)
    st, _ = b.gemm_select_config(8192, 8192, 8192, 1,
                                 b.make_options(variant="dynamic_2cta", block_n=64))
    assert st == b.GEMM_ERR_INVALID_ARG
    # the schedule query reports each cluster's own tile; the rest is decided
    # while the kernel runs
    st, c = b.gemm_select_config(1000, 1000, 520, 1,
                                 b.make_options(variant="dynamic_2cta", stream_k="off"))
    assert st == 0
    for w in range(c.grid // 2):
        assert b.gemm_worker_units(c, w) == [(w, 0, c.k_blocks, 0, 1)]


def test_dynamic_split_tail(b):
    # With stream_k = 2 the dynamic schedule splits the tiles of a partial last
    # wave into S equal K ranges, S = clusters // leftover tiles (at most 4, at
    # least 4 stages each); none when the waves are whole or S would be 1.
    def cfg(M, N, K, **o):
        o.setdefault("stream_k", "on")
        st, c = b.gemm_select_config(M, N, K, 1, b.make_options(variant="dynamic_2cta", **o))
        assert st == 0, b.last_error()
        return c
    c = cfg(8192, 8192, 8192)
    assert (c.dp_tiles, c.sk_tiles, c.sk_max_contrib, c.grid) == (988, 36, 2, 2 * 1060)
    c = cfg(1024, 1024, 4096, block_n=256)   # 16 tiles < 76 clusters: 4 ranges each
    assert (c.num_tiles, c.dp_tiles, c.sk_tiles, c.sk_max_contrib) == (16, 0, 16, 4)
    assert c.grid == 2 * 64
    c = cfg(1024, 1024, 256, block_n=256)    # 2 stages: too short to split
    assert c.sk_tiles == 0 and c.grid == 2 * 16
    c = cfg(1024, 1024, 1024, block_n=256)   # 8 stages: two ranges of 4
    assert (c.sk_tiles, c.sk_max_contrib) == (16, 2)
    c = cfg(4096, 4096, 4096, block_n=224)   # 304 tiles = 4 whole waves
    assert c.sk_tiles == 0 and c.grid == 608
    c = cfg(8192, 8192, 8192, stream_k="off")
    assert c.sk_tiles == 0 and c.grid == 2048
    # the schedule query follows the split: each cluster's own unit
    c = cfg(1024, 1024, 4096, block_n=256)
    ks = c.block_k // 64
    stages = (c.k_blocks + ks - 1) // ks
    for w in range(c.grid // 2):
        tile, part = divmod(w, 4)
        kb0, kb1 = part * stages // 4 * ks, min((part + 1) * stages // 4 * ks, c.k_blocks)
        assert b.gemm_worker_units(c, w) == [(tile, kb0, kb1, part, 4)]


def test_narrow_tiles_for_a_single_partial_wave(b):
    # all tiles within half the clusters: each 256 x 256 tile runs as two
    # 256 x 128 tiles on two clusters
    st, c = b.gemm_select_config(1024, 1024, 4096, 1,
                                 b.make_options(variant="dynamic_2cta", block_n=256))
    assert st == 0 and (c.num_tiles, c.tail_halves, c.grid) == (16, 16, 64)
    for w in range(c.grid // 2):
        assert b.gemm_worker_units(c, w) == [(w // 2, 0, c.k_blocks, 0, 1)]
    for M, N, K, opts in [(8192, 8192, 8192, {}),                      # many waves
                          (1024, 1024, 4096, {"stream_k": "off"}),
                          (1024, 1024, 4096, {"block_k": 64}),         # K = 64 stages
                          (2560, 2560, 4096, {"block_n": 256}),        # 100 tiles
                          (1024, 1024, 4096, {"block_n": 192})]:
        st, c = b.gemm_select_config(M, N, K, 1, b.make_options(variant="dynamic_2cta", **opts))
        assert st == 0 and c.tail_halves == 0, (M, N, K, opts)


def test_block_k_128_stages(b):
    # a stage of K = 128 as two 128-byte swizzle groups of 64 fp16 ("05 Async
    # Data Movement - TMA", Using 3D TMA to Move Multiple Swizzle Atoms): twice
    # the bytes per barrier phase, half as many stages fit
    for v in ("persistent_2cta", "dynamic_2cta"):
        st, c = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(variant=v, block_k=128))
        assert st == 0, b.last_error()
        assert (c.block_k, c.pipe_depth, c.k_blocks) == (128, 3, 128)
        assert c.tx_bytes == 2 * 2 * (128 * 64 + 128 * 64) * 2
        assert c.smem_bytes <= 232448
    st, _ = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(
        variant="persistent_2cta", block_k=128, pipe_depth=4))
    assert st == b.GEMM_ERR_UNSUPPORTED and "does not fit" in b.last_error()
    # the lock-step ladder has single-block stages only; K = 256 stages are
    # built for the single-CTA warp-specialised kernel only
    for v, bk in (("pipelined", 128), ("persistent_lockstep", 128), ("tma_serial", 128),
                  ("persistent_2cta", 256), ("dynamic_2cta", 256), ("pipelined", 256)):
        st, _ = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(variant=v, block_k=bk))
        assert st == b.GEMM_ERR_INVALID_ARG, (v, bk)
    st, _ = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(block_k=96))
    assert st == b.GEMM_ERR_INVALID_ARG
    # stream-K (static pair schedule) splits K in 128-wide stages: the 36-tile
    # partial last wave over 76 pairs, 64 stages per tile
    st, c = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(
        variant="persistent_2cta", block_k=128, stream_k="on"))
    assert st == 0 and c.block_k == 128 and c.sk_tiles == 1024 % 76
    assert c.sk_kb_per_worker == -(-(c.sk_tiles * 64) // 76)
    st, c = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(
        variant="dynamic_2cta", block_k=128, stream_k="on"))
    assert st == 0 and (c.block_k, c.sk_tiles, c.sk_max_contrib) == (128, 36, 2)  # split tail
    st, c = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(block_k=64))
    assert st == 0 and c.block_k == 64 and c.pipe_depth == 6
    # automatic: 128-wide stages only over 128-byte aligned rows (K % 64 == 0)
    for K, bk in [(4992, 128), (5056, 128), (5000, 64), (5064, 64)]:
        st, c = b.gemm_select_config(4000, 3000, K, 0)
        assert st == 0 and c.block_k == bk, K


def test_stage_byte_count_matches_page_formula(b):
    # byte_count = (BLK_M*BLK_K + BLK_N*BLK_K) * 2 for fp16 tiles
    g = _golden("p1_step4_byte_count.txt")
    for bn in (64, 128, 256):
        st, c = b.gemm_select_config(1024, 1024, 1024, 1, b.make_options(block_n=bn))
        assert st == 0
        assert c.tx_bytes == (c.block_m * c.block_k + c.block_n * c.block_k) * int(g["F16_SIZE"])
    # the 2048 + 2048 = 4096 worked example: two 2048-byte tiles on one barrier
    assert int(g["example_tile_bytes"]) * 2 == int(g["example_expect_tx"])


def test_tile_arithmetic_of_the_persistent_step(b):
    g = _golden("p1_step6_tile_arithmetic.txt")
    n = int(g["matrix"])
    st, c = b.gemm_select_config(n, n, n, 1, b.make_options(block_n=int(g["tile"]), grid=int(
        g["sm_count"]), variant="persistent"), sm_count=int(g["sm_count"]))
    assert st == 0
    assert c.num_tiles == int(g["tiles"])
    assert round(c.num_tiles / c.grid) == int(g["tiles_per_cta"])


@pytest.mark.parametrize("M,N,group", [(4096, 4096, 8), (4000, 3000, 8), (64, 16384, 8),
                                       (1000, 72, 3), (128 * 13, 256 * 5, 4)])
def test_raster_covers_every_tile_once_in_group_order(b, M, N, group):
    st, c = b.gemm_select_config(M, N, 64, 1, b.make_options(group_m=group, block_n=256))
    assert st == 0
    seen = np.zeros((c.tiles_m, c.tiles_n), dtype=np.int64)
    prev = None
    for t in range(c.num_tiles):
        st, m, n = b.gemm_schedule_tile(c, t)
        assert st == 0
        seen[m, n] += 1
        # consecutive tiles stay inside one group of `group` M-tiles
        g0 = (m // group)
        if prev is not None:
            assert g0 >= prev[0]
            if g0 == prev[0]:
                assert n >= prev[2]
        prev = (g0, m, n)
    assert (seen == 1).all()
    st, _, _ = b.gemm_schedule_tile(c, c.num_tiles)
    assert st == b.GEMM_ERR_INVALID_ARG


def test_raster_is_the_grouped_order_of_the_persistent_step(b):
    # "GEMM II" Step 6 (l2_group_size): tiles run down a group of G tile rows
    # before moving one tile column right; the last group may be shorter
    rng = np.random.default_rng(3)
    for _ in range(200):
        M, N = int(rng.integers(1, 6000)), int(rng.integers(1, 6000)) // 8 * 8 + 8
        G = int(rng.integers(1, 17))
        st, c = b.gemm_select_config(M, N, 64, 1, b.make_options(group_m=G, block_n=256,
                                                                  variant="persistent"))
        assert st == 0
        for t in range(c.num_tiles):
            first_row = G * (t // (G * c.tiles_n))
            rows = min(c.tiles_m - first_row, G)
            r = t % (G * c.tiles_n)
            assert b.gemm_schedule_tile(c, t) == (0, first_row + r % rows, r // rows), (M, N, G, t)


def test_persistent_ctas_partition_the_tiles(b):
    st, c = b.gemm_select_config(4000, 3000, 5000, 0)
    assert st == 0
    owner = {}
    for cta in range(c.grid):
        for t in range(cta, c.num_tiles, c.grid):
            assert t not in owner
            owner[t] = cta
    assert len(owner) == c.num_tiles


def test_swizzle_map_matches_page_rule_and_bank_analysis(b):
    g = _golden("p2_swizzle_128b.txt")
    # physical 16-byte sector = logical sector XOR (row mod 8), inside an
    # 8-row x 128-byte atom; bytes inside a sector keep their order
    for row in range(16):
        for byte in range(128):
            off = b.gemm_sw128_offset(row, byte)
            assert off // 128 == row
            assert (off % 128) // 16 == (byte // 16) ^ (row % 8)
            assert off % 16 == byte % 16
    # eight consecutive rows reading one logical sector column hit eight
    # distinct 4-bank sectors (no conflict) in the 128-byte-grouped layout
    for col in range(8):
        sectors = {(b.gemm_sw128_offset(r, col * 16) // 16) % 8 for r in range(8)}
        assert len(sectors) == int(g["grouped_distinct_bank_sectors"])
    # the page's ungrouped 256-byte-row comparison: XOR term advances by two
    # per row, leaving only four distinct sectors (a 2-way conflict)
    for col in range(16):
        sectors = {((col % 8) ^ ((2 * r + col // 8) % 8)) for r in range(8)}
        assert len(sectors) == int(g["ungrouped_distinct_bank_sectors"])
    assert b.gemm_sw128_offset(0, 128) == -1


@pytest.mark.parametrize("M,N,K,opts", [
    (8192, 8192, 8192, {"stream_k": "on"}),                   # pair, 36-tile tail
    (4096, 4096, 4096, {"stream_k": "on"}),
    (4000, 3000, 5000, {"stream_k": "on"}),                   # ragged K blocks
    (64, 16384, 16384, {"stream_k": "on"}),                   # every tile shared
    (1000, 1000, 520, {"variant": "persistent", "grid": 7, "stream_k": "on"}),
    (1000, 1000, 520, {"variant": "persistent_2cta", "grid": 10, "stream_k": "on"}),
    (1000, 1000, 520, {"variant": "dynamic_2cta"}),           # own whole tile per cluster
    (1000, 1000, 520, {"variant": "dynamic_2cta", "stream_k": "on"}),  # 28 tiles split in 2
    (8192, 8192, 8192, {"variant": "dynamic_2cta", "stream_k": "on"}),  # 36-tile split tail
    (1024, 1024, 4096, {"variant": "dynamic_2cta", "block_n": 256, "stream_k": "on"}),
    (300, 520, 64, {"variant": "persistent", "stream_k": "on"}),   # one K block per tile
])
def test_work_units_cover_every_k_block_once(b, M, N, K, opts):
    st, c = b.gemm_select_config(M, N, K, 1, b.make_options(**opts))
    assert st == 0, b.last_error()
    _assert_units_cover(b, c)


def test_work_units_cover_every_k_block_once_random_shapes(b):
    rng = np.random.default_rng(2025)
    for _ in range(150):
        M, N = int(rng.integers(1, 3000)), int(rng.integers(1, 3000)) // 8 * 8 + 8
        K = int(rng.integers(1, 3000)) // 8 * 8 + 8
        for opts in ({"variant": "persistent", "stream_k": "on"},
                     {"variant": "persistent_2cta", "stream_k": "on"},
                     {"variant": "dynamic_2cta", "stream_k": "on"},
                     {"variant": "dynamic_2cta"},
                     {"variant": "persistent", "grid": int(rng.integers(1, 152))}):
            st, c = b.gemm_select_config(M, N, K, 1, b.make_options(**opts))
            assert st == 0, (M, N, K, opts, b.last_error())
            _assert_units_cover(b, c)


def _assert_units_cover(b, c):
    pair = c.variant in (b.GEMM_VAR_PERSISTENT_2CTA, b.GEMM_VAR_DYNAMIC_2CTA)
    workers = c.grid // 2 if pair else c.grid
    cover = np.zeros((c.num_tiles, c.k_blocks), dtype=np.int64)
    contribs = {}
    work = []
    for w in range(workers):
        units = b.gemm_worker_units(c, w)
        work.append(sum(kb1 - kb0 for _, kb0, kb1, _, _ in units))
        for tile, kb0, kb1, j, nc in units:
            assert 0 <= kb0 < kb1 <= c.k_blocks
            cover[tile, kb0:kb1] += 1
            if nc > 1:
                assert tile >= c.dp_tiles and nc <= c.sk_max_contrib
                contribs.setdefault(tile, []).append((j, kb0, kb1, nc))
            else:
                assert (kb0, kb1) == (0, c.k_blocks) or tile >= c.dp_tiles
    assert (cover == 1).all()
    for tile, lst in contribs.items():
        lst.sort()
        assert [j for j, _, _, _ in lst] == list(range(lst[0][3]))  # ranks 0..n-1, once each
        assert all(a[2] == b_[1] for a, b_ in zip(lst, lst[1:]))     # ranks follow K order
    if c.sk_tiles and c.variant == b.GEMM_VAR_DYNAMIC_2CTA:
        # a split tile's ranges differ by at most one stage
        for lst in contribs.values():
            sizes = [kb1 - kb0 for _, kb0, kb1, _ in lst]
            assert max(sizes) - min(sizes) <= c.block_k // 64
    elif c.sk_tiles:
        # equal shares: every worker's K-block count within one range of the others
        # shares are counted in pipeline stages of block_k / 64 K blocks
        assert max(work) - min(work) <= c.sk_kb_per_worker * (c.block_k // 64)


def test_stream_k_choice(b):
    on = b.make_options(stream_k="on")
    st, c = b.gemm_select_config(8192, 8192, 8192, 1, on)
    # the static pair schedule with 128-wide stages: 36 tail tiles x 64 stages
    # over 76 pairs
    assert c.variant == b.GEMM_VAR_PERSISTENT_2CTA and c.block_k == 128
    assert (c.dp_tiles, c.sk_tiles, c.sk_kb_per_worker) == (988, 36, 31)
    assert c.dp_tiles % (c.grid // 2) == 0
    st, c = b.gemm_select_config(8192, 8192, 8192, 1, b.make_options(stream_k="on", block_k=64))
    assert (c.dp_tiles, c.sk_tiles, c.sk_kb_per_worker) == (988, 36, 61)
    for opts in (None, b.make_options(stream_k="off")):  # auto = off
        st, c = b.gemm_select_config(8192, 8192, 8192, 1, opts)
        assert (c.dp_tiles, c.sk_tiles, c.workspace_bytes) == (1024, 0, 0)
    st, c = b.gemm_select_config(64, 16384, 16384, 1, on)
    assert c.grid == 152 and c.sk_tiles == c.num_tiles == 128 and c.dp_tiles == 0
    st, c = b.gemm_select_config(64, 16384, 16384, 1)
    assert c.grid == 128 and c.sk_tiles == 0


def test_half_height_a_slots_for_at_most_64_rows(b):
    st, c = b.gemm_select_config(64, 16384, 16384, 1)
    assert st == 0 and c.a_rows == 64 and c.pipe_depth == 8
    assert c.tx_bytes == (64 * 64 + c.block_n * 64) * 2
    st, c = b.gemm_select_config(65, 16384, 16384, 1, b.make_options(variant="persistent"))
    assert c.a_rows == 128
    st, c = b.gemm_select_config(64, 1024, 1024, 1, b.make_options(variant="pipelined"))
    assert c.a_rows == 128  # lock-step kernels keep full-height slots


def test_missing_library_fails_loudly(b, monkeypatch, tmp_path):
    # no fallback path: without the built library every entry point raises
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "libtmagemm.so"))
    with pytest.raises(RuntimeError, match="is missing: build it first"):
        b.Plan(256, 256, 256, out="f32")
    with pytest.raises(RuntimeError, match="is missing"):
        b.gemm_select_config(256, 256, 256, 0)


def _random_shapes(n, seed):
    rng = np.random.default_rng(seed)
    edges = [1, 2, 63, 64, 65, 127, 128, 129, 255, 256, 257, 511, 513]
    for _ in range(n):
        M = int(rng.choice(edges)) if rng.random() < 0.3 else int(rng.integers(1, 20000))
        dt = int(rng.integers(0, 2))
        step = 8 if dt == 1 else 4  # N * sizeof(C element) a multiple of 16 bytes
        N = max(step, int(rng.integers(1, 20000)) // step * step)
        K = max(8, int(rng.integers(1, 20000)) // 8 * 8)
        yield M, N, K, dt


def test_plan_invariants_over_random_shapes(b):
    # Every valid shape gets a plan from every variant, and each plan is
    # self-consistent: tile counts cover M and N, shared memory and TMEM fit,
    # two accumulators for the persistent kernels, and the byte budget is
    # the bytes the stage's copies deliver (both CTAs' with a pair).
    import math
    for M, N, K, dt in _random_shapes(1500, 2024):
        for v in range(0, 9):
            st, c = b.gemm_select_config(M, N, K, dt, b.make_options(variant=v))
            where = (M, N, K, dt, v)
            assert st == 0, (where, b.last_error())
            var, bm, bn = c.variant, c.block_m, c.block_n
            pair = var in (7, 8)
            assert var == v or v == 0, where
            assert bm == (256 if pair else 128), where
            assert c.tiles_m == math.ceil(M / bm) and c.tiles_n == math.ceil(N / bn), where
            assert c.num_tiles == c.tiles_m * c.tiles_n, where
            assert c.k_blocks == math.ceil(K / 64), where
            assert 1 <= c.pipe_depth <= 8 and 0 < c.smem_bytes <= 232448, where
            t = c.tmem_cols
            assert t == 0 or (32 <= t <= 512 and t & (t - 1) == 0), where
            if var in (5, 7, 8):
                assert t >= 2 * bn, where
            if var in (4, 5, 7, 8):
                per_cta = (c.a_rows * 64 + (bn // 2 if pair else bn) * 64) * 2 * (c.block_k // 64)
                assert c.tx_bytes == (2 * per_cta if pair else per_cta), where
            assert c.a_rows == 128 or (c.a_rows == 64 and M <= 64 and not pair), where
            if var in (5, 7):
                assert c.grid <= 152, where


def test_single_cta_multi_block_stages(b):
    # The single-CTA warp-specialised kernel takes stages of 2 or 4 K blocks of
    # 64: ksub sub-slots per stage, the byte budget ksub times one block's,
    # and as many stages as fit.
    for v in ("persistent", "ws_pipelined"):
        for bk, ks in ((64, 1), (128, 2), (256, 4)):
            st, c = b.gemm_select_config(1000, 1000, 1000, 1,
                                         b.make_options(variant=v, block_k=bk, block_n=128))
            assert st == 0, b.last_error()
            per_block = (128 * 64 + 128 * 64) * 2
            assert (c.block_k, c.tx_bytes, c.k_blocks) == (bk, ks * per_block, 16)
            assert c.pipe_depth == {1: 6, 2: 3, 4: 1}[ks], (v, bk, c.pipe_depth)
            assert c.smem_bytes <= 232448
    # at most 64 rows: 64-row A slots, so twice as many stages of 4 blocks fit
    st, c = b.gemm_select_config(64, 16384, 16384, 1, b.make_options(variant="persistent",
                                                                     block_k=256))
    assert st == 0 and (c.a_rows, c.block_k, c.pipe_depth) == (64, 256, 2)
    assert c.tx_bytes == 4 * (64 * 64 + 128 * 64) * 2
    # an explicit depth must fit in stages of the asked K extent
    st, _ = b.gemm_select_config(64, 16384, 16384, 1, b.make_options(
        variant="persistent", block_k=256, pipe_depth=3))
    assert st == b.GEMM_ERR_UNSUPPORTED and "does not fit" in b.last_error()


def test_single_cta_stream_k_in_multi_block_stages(b):
    # the units of a stream-K split are stages of the plan's K extent; the
    # automatic skinny plan keeps single-block stages
    st, c = b.gemm_select_config(64, 16384, 16384, 1)
    assert st == 0 and (c.variant, c.block_n, c.block_k, c.pipe_depth) == (5, 128, 64, 8)
    st, c = b.gemm_select_config(64, 16384, 16384, 1, b.make_options(
        variant="persistent", block_k=256, stream_k="on", grid=152))
    assert st == 0 and c.block_k == 256 and c.sk_tiles > 0
    _assert_units_cover(b, c)
