"""GPU parity of the CTA-pair variant (persistent_2cta: clusters of two CTAs,
tcgen05.mma.cta_group::2, 256 x 256 pair tiles) against the CPU oracle.

Covers pair tiles whose second CTA is partly or wholly past the last row,
ragged N and K, every depth 1..6 against short K loops, many tiles per pair,
integer inputs bit-exact and the five workload shapes at full size; and
stages of K = 128 (block_k = 128, two 64-wide swizzle groups per stage) under
both tile schedules.
"""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_fp16_gb300 import inputs

from gpu_util import assert_close, assert_exact, full_reference, record_error, run

pytestmark = pytest.mark.gpu
V = "persistent_2cta"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("bk", [0, 64])
@pytest.mark.parametrize("out", ["f32", "f16"])
@pytest.mark.parametrize("shape", [(1, 8, 8), (100, 256, 64), (129, 136, 200), (256, 256, 256),
                                   (300, 520, 328), (640, 776, 456)],
                         ids=lambda s: "x".join(map(str, s)))
def test_pair_small_shapes(out, shape, bk):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "uniform", 300 + M + N + K)
    got, guard, desc = run(A, B, out, guard_rows=3, variant=V, block_k=bk)
    assert_close(got, oracle.gemm(A, B), K, out, desc)
    assert np.isnan(guard.astype(np.float32)).all(), "wrote past the end of C"


@pytest.mark.parametrize("depth", [1, 2, 3, 4, 5, 6])
def test_pair_depths_short_k(depth):
    for kt in sorted({1, max(depth - 1, 1), depth, depth + 1, 2 * depth + 1}):
        M, N, K = 384, 512, 64 * kt - 8 * (kt % 2)
        A, B = inputs.make_operands(M, N, K, "normal", 2000 + depth * 16 + kt)
        got, _, desc = run(A, B, "f32", variant=V, pipe_depth=depth)
        assert_close(got, oracle.gemm(A, B), K, "f32", "K tiles=%d %s" % (kt, desc))


@pytest.mark.parametrize("grid", [2, 6, 0])
def test_pair_many_tiles_per_cluster(grid):
    M, N, K = 1280, 1024, 320
    A, B = inputs.make_operands(M, N, K, "uniform", 77)
    got, _, desc = run(A, B, "f16", variant=V, grid=grid, group_m=3)
    assert_close(got, oracle.gemm(A, B), K, "f16", desc)


@pytest.mark.parametrize("bk", [64, 128])
@pytest.mark.parametrize("out,bn", [("f32", 128), ("f32", 160), ("f32", 192), ("f32", 224),
                                    ("f32", 256), ("f16", 128), ("f16", 160), ("f16", 192),
                                    ("f16", 224), ("f16", 256)])
def test_pair_tile_widths(out, bn, bk):
    # ragged in every dimension, several tiles per pair and a second CTA whose
    # rows run past M in the last tile row
    M, N, K = 700, 1000, 456
    A, B = inputs.make_operands(M, N, K, "normal", 900 + bn)
    got, guard, desc = run(A, B, out, guard_rows=2, variant=V, block_n=bn, grid=8, block_k=bk)
    assert "x%dx%d" % (bn, bk) in desc, desc
    assert_close(got, oracle.gemm(A, B), K, out, desc)
    assert np.isnan(guard.astype(np.float32)).all()
    Ai, Bi = inputs.make_operands(M, N, K, "int", 5)
    goti, _, _ = run(Ai, Bi, out, variant=V, block_n=bn, grid=8, block_k=bk)
    assert_exact(goti, oracle.gemm(Ai, Bi), out, desc)


@pytest.mark.parametrize("out", ["f32", "f16"])
def test_pair_integer_bit_exact(out):
    M, N, K = 520, 392, 1000
    A, B = inputs.make_operands(M, N, K, "int", 8)
    got, _, desc = run(A, B, out, variant=V)
    assert_exact(got, oracle.gemm(A, B), out, desc)


@pytest.mark.parametrize("cfg", inputs.CONFIGS, ids=[c["name"] for c in inputs.CONFIGS])
def test_pair_workloads_every_entry(cfg):
    M, N, K, out = cfg["M"], cfg["N"], cfg["K"], cfg["out"]
    A, B, ref = full_reference(cfg)
    got, _, desc = run(A, B, out, variant=V)
    assert np.isfinite(got.astype(np.float32)).all(), desc
    record_error("%s (%s)" % (cfg["name"], V), got, ref, K, out)
    assert_close(got, ref, K, out, desc)
    Ai, Bi, refi = full_reference(cfg, "int", 60 + cfg["seed"])
    goti, _, _ = run(Ai, Bi, out, variant=V)
    assert_exact(goti, refi, out, desc)


def test_pair_watchdog_timeout():
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    from tma_pipelined_tensor_fp16_gb300 import binding
    M, N, K = 512, 512, 256
    A, B = inputs.make_operands(M, N, K, "uniform", 3)
    dA = torch.from_numpy(A.view(np.float16)).cuda()
    dB = torch.from_numpy(B.view(np.float16)).cuda()
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    plan = pkg.Plan(M, N, K, out="f32", variant=V, debug_stall=1, wait_budget_ms=100)
    plan(dA, dB, C)
    torch.cuda.synchronize()
    assert plan.device_status() == binding.GEMM_ERR_TIMEOUT
    plan.close()
    got, _, desc = run(A, B, "f32", variant=V)
    assert_close(got, oracle.gemm(A, B), K, "f32", "after timeout: " + desc)


@pytest.mark.parametrize("variant", ["persistent_2cta", "dynamic_2cta"])
@pytest.mark.parametrize("out", ["f32", "f16"])
@pytest.mark.parametrize("K", [8, 136, 520, 1032])
def test_pair_block_k_128(variant, out, K):
    # stages of K = 128 as two 64-wide swizzle groups; an odd number of 64-wide
    # K blocks leaves the second group of the last stage past K (zero-filled,
    # its MMAs skipped)
    M, N = 1100, 1000
    A, B = inputs.make_operands(M, N, K, "normal", 4100 + K)
    for depth in (0, 1, 2):
        got, guard, desc = run(A, B, out, guard_rows=2, variant=variant, block_k=128,
                               pipe_depth=depth)
        assert desc.split("tile=")[1].split()[0].endswith("x128"), desc
        assert_close(got, oracle.gemm(A, B), K, out, desc)
        assert np.isnan(guard.astype(np.float32)).all()
    Ai, Bi = inputs.make_operands(M, N, K, "int", 41)
    goti, _, desc = run(Ai, Bi, out, variant=variant, block_k=128)
    assert_exact(goti, oracle.gemm(Ai, Bi), out, desc)


@pytest.mark.parametrize("cfg", [c for c in inputs.CONFIGS if c["M"] > 128],
                         ids=[c["name"] for c in inputs.CONFIGS if c["M"] > 128])
def test_pair_block_k_128_workloads(cfg):
    M, N, K, out = cfg["M"], cfg["N"], cfg["K"], cfg["out"]
    A, B, ref = full_reference(cfg)
    # whole tiles on the dynamic schedule (no split tail): the same sums in the
    # same order as the static schedule, bit for bit
    got, _, desc = run(A, B, out, variant="dynamic_2cta", block_k=128, stream_k="off")
    stat, _, _ = run(A, B, out, variant="persistent_2cta", block_k=128)
    assert np.array_equal(got.view(np.uint8), stat.view(np.uint8)), desc
    record_error("%s (dynamic_2cta, block_k 128)" % cfg["name"], got, ref, K, out)
    assert_close(got, ref, K, out, desc)
