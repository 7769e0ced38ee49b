"""GPU parity of the single-CTA warp-specialised kernel with stages of 2 or 4
K blocks (block_k = 128 / 256) against the CPU oracle.

A stage holds ksub 64-wide K blocks, each in a sub-slot of its own, behind
one barrier round trip ("05 Async Data Movement - TMA", Using 3D TMA to Move
Multiple Swizzle Atoms, loaded as ksub 2-D boxes).  Covered: both variants,
both output types, ragged M, N and K (the last stage then holds blocks past K,
which arrive zero-filled and are not multiplied), at most 64 rows (64-row A
slots), every ring depth that fits against short K loops (K stages in {1,
D-1, D, D+1, 2D+1}), many tiles per CTA with the K snake, stream-K splits in
units of stages, integer inputs bit for bit, and the NaN guard band past C.
"""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_fp16_gb300 import inputs

from gpu_util import assert_close, assert_exact, run

pytestmark = pytest.mark.gpu

SHAPES = [
    (1, 8, 8),         # one element row, one K chunk
    (64, 520, 1000),   # 64-row A slots; K = 15 blocks + 40 columns
    (129, 136, 200),   # ragged everywhere, 4 K blocks (the last 8 columns)
    (300, 520, 328),   # several tiles each way
    (390, 776, 456),   # 8 K blocks, the last ragged
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("variant", ["persistent", "ws_pipelined"])
@pytest.mark.parametrize("block_k", [128, 256])
@pytest.mark.parametrize("out", ["f32", "f16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_multi_block_stages_match_oracle(variant, block_k, out, shape):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "uniform", 500 + M + N + K + block_k)
    got, guard, desc = run(A, B, out, guard_rows=3, variant=variant, block_k=block_k)
    assert "x%d pipe" % block_k in desc, desc
    assert_close(got, oracle.gemm(A, B), K, out, "%s %s" % (out, desc))
    assert np.isnan(guard.astype(np.float32)).all(), "wrote past the end of C"


@pytest.mark.parametrize("variant", ["persistent", "ws_pipelined"])
@pytest.mark.parametrize("block_k", [128, 256])
@pytest.mark.parametrize("out", ["f32", "f16"])
def test_multi_block_stages_integer_bit_exact(variant, block_k, out):
    for M, N, K in ((257, 200, 520), (64, 392, 1000)):
        A, B = inputs.make_operands(M, N, K, "int", 17 + M)
        got, _, desc = run(A, B, out, variant=variant, block_k=block_k)
        assert_exact(got, oracle.gemm(A, B), out, desc)


@pytest.mark.parametrize("block_k,depths", [(128, [1, 2, 3, 4]), (256, [1, 2])])
@pytest.mark.parametrize("M", [160, 48])
def test_multi_block_depth_sweep_short_k(block_k, depths, M):
    # block_n = 64 leaves the most room for stages; K is counted in stages of
    # block_k, the odd counts ending ragged (inside the last stage's first
    # block, so the others lie wholly past K)
    ks = block_k // 64
    for depth in depths:
        for st in sorted({1, max(depth - 1, 1), depth, depth + 1, 2 * depth + 1}):
            K = block_k * st - (block_k - 56) * (st % 2)
            A, B = inputs.make_operands(M, 192, K, "normal", 2000 + depth * 16 + st + ks)
            for variant in ("persistent", "ws_pipelined"):
                got, _, desc = run(A, B, "f32", variant=variant, pipe_depth=depth, block_n=64,
                                   block_k=block_k)
                assert_close(got, oracle.gemm(A, B), K, "f32",
                             "%s stages=%d %s" % (variant, st, desc))


@pytest.mark.parametrize("block_k", [128, 256])
@pytest.mark.parametrize("grid", [1, 7])
def test_multi_block_many_tiles_per_cta(block_k, grid):
    # many tiles per CTA: the ring position and both accumulators run on
    # across tiles, and every other tile walks its stages downwards (K snake)
    M, N, K = 700, 640, 1480
    A, B = inputs.make_operands(M, N, K, "uniform", 55 + block_k)
    for k_order in ("snake", "up"):
        got, _, desc = run(A, B, "f16", variant="persistent", grid=grid, block_n=64,
                           block_k=block_k, k_order=k_order)
        assert_close(got, oracle.gemm(A, B), K, "f16", "%s %s" % (k_order, desc))


@pytest.mark.parametrize("block_k", [128, 256])
@pytest.mark.parametrize("out", ["f32", "f16"])
def test_multi_block_stream_k_integer_bit_exact(block_k, out):
    # partial sums of K-stage ranges added in a fixed order: exact on
    # integer inputs, and the same bits on every run
    M, N, K = 64, 8192, 2056
    A, B = inputs.make_operands(M, N, K, "int", 93)
    got, _, desc = run(A, B, out, variant="persistent", block_k=block_k, stream_k="on", grid=152)
    assert "stream_k=0/" not in desc, desc
    assert_exact(got, oracle.gemm(A, B), out, desc)
    again, _, _ = run(A, B, out, variant="persistent", block_k=block_k, stream_k="on", grid=152)
    assert np.array_equal(got.view(np.uint8), again.view(np.uint8)), "run-to-run difference"


@pytest.mark.parametrize("block_k", [128, 256])
def test_multi_block_stream_k(block_k):
    # stream-K over 152 CTAs splits the tiles of the partial last wave in
    # ranges of stages; partial sums meet in the workspace
    for M, N, K in ((64, 16384, 2056), (520, 1000, 1000)):
        A, B = inputs.make_operands(M, N, K, "normal", 91 + M)
        got, _, desc = run(A, B, "f32", variant="persistent", block_k=block_k, stream_k="on",
                           grid=152)
        assert "stream_k=0/" not in desc or M == 520, desc
        assert_close(got, oracle.gemm(A, B), K, "f32", desc)


def test_skinny_shape_with_four_block_stages():
    # 64 rows (64-row A slots), stages of 4 K blocks: 512 contiguous bytes of
    # every row of B per stage
    M, N, K = 64, 16384, 4096
    A, B = inputs.make_operands(M, N, K, "uniform", 4)
    got, _, desc = run(A, B, "f16", variant="persistent", block_k=256)
    assert "variant=persistent tile=128x128x256 pipe_depth=2" in desc, desc
    assert_close(got, oracle.gemm(A, B), K, "f16", desc)
