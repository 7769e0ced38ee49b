"""GPU parity of the dynamic CTA-pair schedule (dynamic_2cta) against the CPU
oracle.  The grid holds one cluster per pair tile; a running cluster cancels
clusters that have not started (cluster launch control) and computes their
tiles ("GEMM II -- pipelining with TMA", Step 6: hardware work-stealing in
place of the precomputed tile assignment).

Covers one tile (the first request finds nothing to cancel), tile counts below
and above the number of resident clusters, every pair width, integer inputs
bit-exact, the five workload shapes at full size, that the tile sequence
visits every tile exactly once (from the device timeline), that results are
identical bit for bit to the static schedule's and from run to run, and the
watchdog.
"""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_fp16_gb300 import inputs

from gpu_util import assert_close, assert_exact, full_reference, record_error, run, run_repeated

pytestmark = pytest.mark.gpu
V = "dynamic_2cta"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("out", ["f32", "f16"])
@pytest.mark.parametrize("shape", [(1, 8, 8), (100, 256, 64), (300, 520, 328), (640, 776, 456),
                                   (1280, 1024, 320), (2304, 2560, 192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_dynamic_small_shapes(out, shape):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "uniform", 500 + M + N + K)
    got, guard, desc = run(A, B, out, guard_rows=3, variant=V)
    assert_close(got, oracle.gemm(A, B), K, out, desc)
    assert np.isnan(guard.astype(np.float32)).all(), "wrote past the end of C"


@pytest.mark.parametrize("bk", [64, 128])
@pytest.mark.parametrize("out,bn", [("f32", 128), ("f32", 160), ("f32", 192), ("f32", 224),
                                    ("f32", 256), ("f16", 128), ("f16", 160), ("f16", 192),
                                    ("f16", 224), ("f16", 256)])
def test_dynamic_tile_widths(out, bn, bk):
    # 80 to 160 tiles: more than the 76 clusters that fit at once, so most
    # tiles are taken over by cancellation; ragged in every dimension
    M, N, K = 5000, 1000, 136
    A, B = inputs.make_operands(M, N, K, "normal", 1900 + bn)
    got, guard, desc = run(A, B, out, guard_rows=2, variant=V, block_n=bn, block_k=bk)
    assert "x%dx%d" % (bn, bk) in desc, desc
    assert_close(got, oracle.gemm(A, B), K, out, desc)
    assert np.isnan(guard.astype(np.float32)).all()
    Ai, Bi = inputs.make_operands(M, N, K, "int", 15)
    goti, _, _ = run(Ai, Bi, out, variant=V, block_n=bn, block_k=bk)
    assert_exact(goti, oracle.gemm(Ai, Bi), out, desc)


@pytest.mark.parametrize("depth", [1, 3, 6])
def test_dynamic_depths_short_k(depth):
    for kt in sorted({1, depth, depth + 1}):
        M, N, K = 2560, 2048, 64 * kt - 8 * (kt % 2)
        A, B = inputs.make_operands(M, N, K, "normal", 3000 + depth * 16 + kt)
        got, _, desc = run(A, B, "f32", variant=V, pipe_depth=depth)
        assert_close(got, oracle.gemm(A, B), K, "f32", "K tiles=%d %s" % (kt, desc))


@pytest.mark.parametrize("cfg", inputs.CONFIGS, ids=[c["name"] for c in inputs.CONFIGS])
def test_dynamic_workloads_match_static_schedule(cfg):
    # Every tile walks K in the same direction under both schedules, so the
    # fp32 sums are formed in the same order and the outputs agree bit for bit
    # (with whole tiles: the split tail, on by default, sums K ranges apart).
    M, N, K, out = cfg["M"], cfg["N"], cfg["K"], cfg["out"]
    A, B, _ = full_reference(cfg)
    whole, _, desc_w = run(A, B, out, variant=V, stream_k="off")
    ref_static, _, desc_s = run(A, B, out, variant="persistent_2cta")
    assert np.array_equal(whole.view(np.uint8), ref_static.view(np.uint8)), (desc_w, desc_s)
    got, _, desc = run(A, B, out, variant=V)
    _, _, ref = full_reference(cfg)
    record_error("%s (%s)" % (cfg["name"], V), got, ref, K, out)
    assert_close(got, ref, K, out, desc)
    again, _, _ = run(A, B, out, variant=V)
    assert np.array_equal(got.view(np.uint8), again.view(np.uint8)), "run-to-run difference"


def test_dynamic_visits_every_tile_once():
    from tma_pipelined_tensor_fp16_gb300 import timeline
    M = N = K = 4096
    tr, cfg = timeline.record(M, N, K, "f16", "uniform", 1, warmup=2, units=64, variant=V)
    live = timeline.ran(tr)
    assert len(live) % 2 == 0 and len(live) < cfg["grid"]  # most clusters were cancelled
    seen = []
    for b in live:
        n = int(tr[b, 0, timeline.H_UNITS])
        assert 0 < n <= 64
        tiles = [int(tr[b, 1 + i, timeline.U_TILE]) >> 32 for i in range(n)]
        if b % 2 == 0:
            seen.extend(tiles)
        else:  # both CTAs of a cluster walk the same sequence
            assert tiles == [int(tr[b - 1, 1 + i, timeline.U_TILE]) >> 32 for i in range(n)]
    assert sorted(seen) == list(range(cfg["num_tiles"]))


def test_dynamic_watchdog_timeout():
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    from tma_pipelined_tensor_fp16_gb300 import binding
    M, N, K = 2048, 2048, 256
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


@pytest.mark.parametrize("opts", [{"variant": "dynamic_2cta", "block_k": 64},
                                  {"variant": "dynamic_2cta", "block_k": 128},
                                  {"variant": "persistent_2cta", "block_k": 128},
                                  {"variant": "persistent_2cta", "stream_k": "on"},
                                  {"variant": "persistent"}],
                         ids=["dyn64", "dyn128", "static128", "static_streamk", "single"])
def test_same_plan_launched_repeatedly(opts):
    # one plan, five launches on one stream (as the benchmark runs it): every
    # launch writes every output and all five agree bit for bit; several waves
    # of tiles, so most clusters of the dynamic grid are cancelled each time
    M, N, K = 3072, 4096, 1024
    A, B = inputs.make_operands(M, N, K, "uniform", 66)
    outs = run_repeated(A, B, "f16", 5, **opts)
    variant = opts["variant"]
    ref = outs[0]
    assert not np.isnan(ref.astype(np.float32)).any()
    assert_close(ref, oracle.gemm(A, B), K, "f16", variant)
    for i, o in enumerate(outs[1:], 1):
        assert np.array_equal(o.view(np.uint16), ref.view(np.uint16)), "launch %d differs" % i


@pytest.mark.parametrize("bk", [64, 128])
def test_dynamic_many_tiles_per_cluster(bk):
    # 4096 pair tiles over 76 resident clusters: about 54 cancellations per
    # cluster, the response ring wrapping many times; a short K keeps it quick
    M, N, K = 32768, 8192, 128
    A, B = inputs.make_operands(M, N, K, "uniform", 77)
    got, guard, desc = run(A, B, "f16", guard_rows=2, variant=V, block_k=bk)
    assert np.isnan(guard.astype(np.float32)).all()
    assert not np.isnan(got.astype(np.float32)).any(), desc
    ref, _, _ = run(A, B, "f16", variant="persistent_2cta", block_k=bk)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), desc
    assert_close(got, oracle.gemm(A, B), K, "f16", desc)
