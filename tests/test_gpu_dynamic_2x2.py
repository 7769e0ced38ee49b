"""GPU parity of the two-pairs-per-cluster variant (dynamic_2x2) against the
CPU oracle.

A cluster of four CTAs computes two side-by-side 256-row pair tiles.  The
CTAs of equal rank in the two pairs need the same 128 rows of A: each loads
one 64-row half with a multicast TMA copy into both ("05 Async Data Movement
- TMA": a tile read once from global memory feeds several CTAs of a
cluster), and each pair's MMA leader frees a stage in all four CTAs.  The
schedule is the dynamic one (cluster launch control) over such units.

Covers shapes with an odd number of tile columns (the last unit's second
tile lies past N and must not be stored), one unit, units above the number
of resident clusters, some 114 units per resident cluster (the response
ring wrapping many times), the three tile widths and both stage widths,
integer inputs bit-exact, identity with the one-pair kernel when both walk K in the
same order, the workload shapes, repeated launches, the unit sequence seen
by the device timeline, and the watchdog.
"""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_fp16_gb300 import inputs

from gpu_util import assert_close, assert_exact, run, run_repeated

pytestmark = pytest.mark.gpu
V = "dynamic_2x2"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _sample(M, N, count, seed):
    rng = np.random.default_rng(seed)
    rows = np.concatenate([rng.integers(0, M, count), [0, M - 1, min(255, M - 1)]])
    cols = np.concatenate([rng.integers(0, N, count), [N - 1, 0, min(255, N - 1)]])
    return rows.astype(np.int64), cols.astype(np.int64)


@pytest.mark.parametrize("out", ["f32", "f16"])
@pytest.mark.parametrize("shape", [(1, 8, 8), (100, 256, 64), (300, 520, 328), (640, 776, 456),
                                   (1280, 1024, 320), (2304, 2560, 192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_2x2_small_shapes(out, shape):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "uniform", 700 + M + N + K)
    got, guard, desc = run(A, B, out, guard_rows=3, variant=V)
    assert_close(got, oracle.gemm(A, B), K, out, desc)
    assert np.isnan(guard.astype(np.float32)).all(), "wrote past the end of C"


@pytest.mark.parametrize("bk", [64, 128])
@pytest.mark.parametrize("out,bn", [("f32", 192), ("f32", 224), ("f32", 256),
                                    ("f16", 192), ("f16", 224), ("f16", 256)])
def test_2x2_tile_widths(out, bn, bk):
    # 20 x 5..6 tile columns: units above the 36 clusters that fit at once,
    # an odd column count for two of the widths, ragged in every dimension
    M, N, K = 5000, 1000, 136
    A, B = inputs.make_operands(M, N, K, "normal", 2900 + bn)
    got, guard, desc = run(A, B, out, guard_rows=2, variant=V, block_n=bn, block_k=bk)
    assert "x%dx%d" % (bn, bk) in desc, desc
    assert_close(got, oracle.gemm(A, B), K, out, desc)
    assert np.isnan(guard.astype(np.float32)).all()
    Ai, Bi = inputs.make_operands(M, N, K, "int", 16)
    goti, _, _ = run(Ai, Bi, out, variant=V, block_n=bn, block_k=bk)
    assert_exact(goti, oracle.gemm(Ai, Bi), out, desc)


@pytest.mark.parametrize("depth", [1, 3, 6])
def test_2x2_depths_short_k(depth):
    for kt in sorted({1, depth, depth + 1}):
        M, N, K = 2560, 2048, 64 * kt - 8 * (kt % 2)
        A, B = inputs.make_operands(M, N, K, "normal", 3100 + depth * 16 + kt)
        got, _, desc = run(A, B, "f32", variant=V, pipe_depth=depth)
        assert_close(got, oracle.gemm(A, B), K, "f32", "K tiles=%d %s" % (kt, desc))


@pytest.mark.parametrize("bk", [64, 128])
def test_2x2_equals_one_pair_kernel(bk):
    # With K walked upwards by every tile, each output is the same fp32 sum in
    # the same order as in the one-pair kernel: identical bit for bit.
    M, N, K = 3000, 2600, 1032
    A, B = inputs.make_operands(M, N, K, "uniform", 88)
    got, _, desc = run(A, B, "f16", variant=V, block_n=224, block_k=bk, k_order="up")
    ref, _, desc1 = run(A, B, "f16", variant="dynamic_2cta", block_n=224, block_k=bk,
                        k_order="up")
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), (desc, desc1)
    rows, cols = _sample(M, N, 2000, 88)
    assert_close(got[rows, cols], oracle.gemm_entries(A, B, rows, cols), K, "f16", desc)


def test_2x2_many_units_per_cluster():
    # 4096 units (two 256-wide pair tiles each) over 36 resident clusters of
    # four: about 114 cancellations per cluster, the four-slot response ring
    # wrapping some 28 times.  The host model of that ring shows a reader
    # miscount only after about 85 units per cluster with two pairs, so
    # shorter runs could not catch one; a short K keeps this quick.
    M, N, K = 65536, 8192, 128
    A, B = inputs.make_operands(M, N, K, "uniform", 79)
    got, guard, desc = run(A, B, "f16", guard_rows=2, variant=V, block_n=256, k_order="up")
    assert np.isnan(guard.astype(np.float32)).all()
    assert not np.isnan(got.astype(np.float32)).any(), desc
    ref, _, desc1 = run(A, B, "f16", variant="dynamic_2cta", block_n=256, k_order="up")
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), (desc, desc1)
    rows, cols = _sample(M, N, 4000, 79)
    assert_close(got[rows, cols], oracle.gemm_entries(A, B, rows, cols), K, "f16", desc)


@pytest.mark.parametrize("cfg", [c for c in inputs.CONFIGS if c["M"] > 128],
                         ids=[c["name"] for c in inputs.CONFIGS if c["M"] > 128])
def test_2x2_workloads_sampled(cfg):
    M, N, K, out = cfg["M"], cfg["N"], cfg["K"], cfg["out"]
    A, B = inputs.make_operands(M, N, K, cfg["dist"], cfg["seed"])
    got, _, desc = run(A, B, out, variant=V)
    assert not np.isnan(got.astype(np.float32)).any(), desc
    rows, cols = _sample(M, N, 2000, cfg["seed"])
    assert_close(got[rows, cols], oracle.gemm_entries(A, B, rows, cols), K, out, desc)


def test_2x2_same_plan_launched_repeatedly():
    M, N, K = 3072, 4096, 1024
    A, B = inputs.make_operands(M, N, K, "uniform", 67)
    outs = run_repeated(A, B, "f16", 5, variant=V)
    ref = outs[0]
    assert not np.isnan(ref.astype(np.float32)).any()
    rows, cols = _sample(M, N, 2000, 67)
    assert_close(ref[rows, cols], oracle.gemm_entries(A, B, rows, cols), K, "f16", V)
    for i, o in enumerate(outs[1:], 1):
        assert np.array_equal(o.view(np.uint16), ref.view(np.uint16)), "launch %d differs" % i


def test_2x2_visits_every_unit_once():
    from tma_pipelined_tensor_fp16_gb300 import timeline
    M = N = K = 4096
    tr, cfg = timeline.record(M, N, K, "f16", "uniform", 1, warmup=2, units=64, variant=V)
    live = timeline.ran(tr)
    assert len(live) % 4 == 0 and len(live) < cfg["grid"]  # most clusters were cancelled
    units = cfg["tiles_m"] * ((cfg["tiles_n"] + 1) // 2)
    seen = []
    for b in live:
        n = int(tr[b, 0, timeline.H_UNITS])
        assert 0 < n <= 64
        seq = [int(tr[b, 1 + i, timeline.U_TILE]) >> 32 for i in range(n)]
        if b % 4 == 0:
            seen.extend(seq)
        else:  # all four CTAs of a cluster walk the same sequence
            first = b - b % 4
            assert seq == [int(tr[first, 1 + i, timeline.U_TILE]) >> 32 for i in range(n)]
    assert sorted(seen) == list(range(units))


def test_2x2_watchdog_timeout():
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    from tma_pipelined_tensor_fp16_gb300 import binding
    M, N, K = 2048, 2048, 256
    A, B = inputs.make_operands(M, N, K, "uniform", 4)
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
