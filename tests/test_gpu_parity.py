"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Tolerances are those stated in gpu_util.

Covers every ladder variant, both output dtypes, ragged shapes spanning
several tiles, the pipeline-depth sweep against short K loops (K tiles in
{1, D-1, D, D+1, 2D+1}), every tile width, the NaN guard band past the end of
C, non-default streams, the host-buffer entry point, and the five workload
shapes at full size in the configuration the benchmark times, every entry of
C against the oracle: random inputs within the tolerance, integer inputs bit
for bit, and the closed forms.
"""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_fp16_gb300 import inputs

from gpu_util import (assert_close, assert_exact, full_reference, record_error, run,
                      run_repeated)

pytestmark = pytest.mark.gpu

VARIANTS = ["sync_tiled", "tma_serial", "pipelined", "ws_pipelined", "persistent",
            "persistent_lockstep"]

SMALL_SHAPES = [
    (1, 8, 8),          # one element row, one K chunk
    (128, 128, 64),     # exactly one tile, one K block
    (129, 136, 200),    # ragged in every dimension
    (300, 520, 328),    # several tiles each way, ragged
    (256, 256, 256),    # the 256^3 workload shape
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("out", ["f32", "f16"])
@pytest.mark.parametrize("shape", SMALL_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_small_shapes_match_oracle(variant, out, shape):
    M, N, K = shape
    A, B = inputs.make_operands(M, N, K, "uniform", 100 + M + N + K)
    got, guard, desc = run(A, B, out, guard_rows=3, variant=variant)
    assert_close(got, oracle.gemm(A, B), K, out, "%s %s %s" % (variant, out, desc))
    assert np.isnan(guard.astype(np.float32)).all(), "wrote past the end of C"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("out", ["f32", "f16"])
def test_integer_inputs_bit_exact(variant, out):
    M, N, K = 257, 200, 520
    A, B = inputs.make_operands(M, N, K, "int", 7)
    got, _, desc = run(A, B, out, variant=variant)
    assert_exact(got, oracle.gemm(A, B), out, "%s %s %s" % (variant, out, desc))


@pytest.mark.parametrize("variant", ["pipelined", "ws_pipelined", "persistent",
                                     "persistent_lockstep"])
@pytest.mark.parametrize("depth", [1, 2, 3, 4, 5, 6, 7, 8])
def test_depth_sweep_short_k(variant, depth):
    # block_n = 64 lets every depth 1..8 fit in shared memory.
    for kt in sorted({1, max(depth - 1, 1), depth, depth + 1, 2 * depth + 1}):
        M, N, K = 160, 192, 64 * kt - 8 * (kt % 2)  # odd K-tile counts end ragged
        A, B = inputs.make_operands(M, N, K, "normal", 1000 + depth * 16 + kt)
        got, _, desc = run(A, B, "f32", variant=variant, pipe_depth=depth, block_n=64)
        assert_close(got, oracle.gemm(A, B), K, "f32", "%s K tiles=%d %s" % (variant, kt, desc))


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("block_n", [64, 128, 256])
@pytest.mark.parametrize("out", ["f32", "f16"])
def test_every_tile_width(variant, block_n, out):
    M, N, K = 390, 776, 456
    A, B = inputs.make_operands(M, N, K, "uniform", block_n)
    got, _, desc = run(A, B, out, variant=variant, block_n=block_n)
    assert_close(got, oracle.gemm(A, B), K, out, desc)


@pytest.mark.parametrize("variant", ["persistent", "ws_pipelined"])
@pytest.mark.parametrize("M", [1, 17, 64])
@pytest.mark.parametrize("depth", [1, 4, 8])
def test_at_most_64_rows_use_half_height_a_slots(variant, M, depth):
    # 64-row A stages: the MMA's rows 64..127 read whatever follows the slot
    # and must never reach C (the NaN guard band would show it)
    for out in ("f32", "f16"):
        for N, K in ((8, 8), (520, 1000)):
            A, B = inputs.make_operands(M, N, K, "normal", 70 + M + depth)
            got, guard, desc = run(A, B, out, guard_rows=80, variant=variant, pipe_depth=depth,
                                   block_n=128)
            assert_close(got, oracle.gemm(A, B), K, out, desc)
            assert np.isnan(guard.astype(np.float32)).all(), "wrote past row M"


@pytest.mark.parametrize("group_m", [1, 3, 8])
@pytest.mark.parametrize("grid", [1, 7, 0])
def test_persistent_schedules(group_m, grid):
    # Many tiles per CTA (grid 1 and 7) exercise the continuous ring phase and
    # both TMEM accumulators over long tile sequences.
    M, N, K = 700, 640, 200
    A, B = inputs.make_operands(M, N, K, "uniform", 55)
    for variant in ("persistent", "persistent_lockstep"):
        got, _, desc = run(A, B, "f16", variant=variant, group_m=group_m, grid=grid,
                           block_n=64, pipe_depth=3)
        assert_close(got, oracle.gemm(A, B), K, "f16", desc)


def test_non_default_stream():
    import torch
    M, N, K = 384, 256, 512
    A, B = inputs.make_operands(M, N, K, "uniform", 9)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        got, _, _ = run(A, B, "f32", stream=s)
    assert_close(got, oracle.gemm(A, B), K, "f32", "side stream")


def test_run_host_entry_point():
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    M, N, K = 300, 248, 264
    A, B = inputs.make_operands(M, N, K, "normal", 12)
    hA = torch.from_numpy(A.view(np.float16)).pin_memory()
    hB = torch.from_numpy(B.view(np.float16)).pin_memory()
    hC = torch.empty((M, N), dtype=torch.float32).pin_memory()
    plan = pkg.Plan(M, N, K, out="f32")
    for _ in range(2):  # the second call reuses the plan's device buffers
        plan.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(),
                      torch.cuda.current_stream().cuda_stream)
        assert_close(hC.numpy(), oracle.gemm(A, B), K, "f32", "run_host")
    plan.close()


@pytest.mark.parametrize("out", ["f32", "f16"])
@pytest.mark.parametrize("variant", ["auto", "persistent"])
def test_run_host_banded_pipeline(out, variant):
    # M >= 2048 with page-locked buffers: B, then A band by band, band GEMMs
    # as rows arrive, C bands copied back while later bands compute; the last
    # band is shorter than the others
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    M, N, K = 2304, 520, 264
    A, B = inputs.make_operands(M, N, K, "uniform", 14)
    hA = torch.from_numpy(A.view(np.float16)).pin_memory()
    hB = torch.from_numpy(B.view(np.float16)).pin_memory()
    dt = torch.float16 if out == "f16" else torch.float32
    hC = torch.full((M, N), float("nan"), dtype=dt).pin_memory()
    plan = pkg.Plan(M, N, K, out=out, variant=variant)
    ref = oracle.gemm(A, B)
    s = torch.cuda.Stream()
    for _ in range(2):
        plan.run_host(hA.data_ptr(), hB.data_ptr(), hC.data_ptr(), s.cuda_stream)
        got = hC.numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert_close(got, ref, K, out, "banded run_host")
        hC.fill_(float("nan"))
    plan.close()


def test_run_host_pageable_buffers():
    import tma_pipelined_tensor_fp16_gb300 as pkg
    M, N, K = 2304, 264, 128
    A, B = inputs.make_operands(M, N, K, "normal", 15)
    C = np.zeros((M, N), dtype=np.float32)
    plan = pkg.Plan(M, N, K, out="f32")
    plan.run_host(A.ctypes.data, B.ctypes.data, C.ctypes.data, 0)
    assert_close(C, oracle.gemm(A, B), K, "f32", "pageable run_host")
    plan.close()


def test_argument_errors_are_reported():
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    from tma_pipelined_tensor_fp16_gb300 import binding
    plan = pkg.Plan(128, 128, 64, out="f16")
    a = torch.zeros(128 * 64 + 8, dtype=torch.float16, device="cuda")
    c = torch.zeros(128 * 128, dtype=torch.float16, device="cuda")
    st = binding.gemm_run(plan.handle, a.data_ptr() + 2, a.data_ptr(), c.data_ptr(), None)
    assert st == binding.GEMM_ERR_UNSUPPORTED
    st = binding.gemm_run(plan.handle, None, a.data_ptr(), c.data_ptr(), None)
    assert st == binding.GEMM_ERR_INVALID_ARG
    plan.close()
    with pytest.raises(binding.GemmError) as e:
        pkg.Plan(256, 256, 256, out="f16", block_n=256, pipe_depth=8)
    assert e.value.status == binding.GEMM_ERR_UNSUPPORTED


# ------------------------------------------------- the five workloads, full size

@pytest.mark.parametrize("cfg", inputs.CONFIGS, ids=[c["name"] for c in inputs.CONFIGS])
def test_workload_random_inputs_every_entry(cfg):
    # The automatic plan bench.py times, launched twice back to back on one
    # stream as the benchmark does; every entry of C against the oracle under
    # the stated tolerance, and the two launches bit-identical.
    M, N, K, out = cfg["M"], cfg["N"], cfg["K"], cfg["out"]
    A, B, ref = full_reference(cfg)
    first, got = run_repeated(A, B, out, 2)
    desc = "%s (automatic plan)" % cfg["name"]
    assert np.isfinite(got.astype(np.float32)).all(), desc
    record_error(desc, got, ref, K, out)
    assert_close(got, ref, K, out, desc)
    assert np.array_equal(first.view(np.uint8), got.view(np.uint8)), "run-to-run difference"


@pytest.mark.parametrize("cfg", inputs.CONFIGS, ids=[c["name"] for c in inputs.CONFIGS])
def test_workload_integer_inputs_bit_exact_every_entry(cfg):
    M, N, K, out = cfg["M"], cfg["N"], cfg["K"], cfg["out"]
    A, B, ref = full_reference(cfg, "int", 40 + cfg["seed"])
    got, _, desc = run(A, B, out)
    assert_exact(got, ref, out, "%s %s" % (cfg["name"], desc))


@pytest.mark.parametrize("cfg", inputs.CONFIGS, ids=[c["name"] for c in inputs.CONFIGS])
def test_workload_all_ones_every_entry(cfg):
    M, N, K, out = cfg["M"], cfg["N"], cfg["K"], cfg["out"]
    if out == "f16" and K > 2048 and (K & (K - 1)):
        pytest.skip("K not exactly representable in fp16")
    A, B = inputs.make_operands(M, N, K, "ones", 0)
    got, _, desc = run(A, B, out)
    assert (got.astype(np.float64) == float(K)).all(), desc


@pytest.mark.parametrize("cfg", inputs.CONFIGS[:3], ids=[c["name"] for c in inputs.CONFIGS[:3]])
def test_workload_permutation_b_every_entry(cfg):
    M, K, out = cfg["M"], cfg["K"], cfg["out"]
    A, _ = inputs.make_operands(M, 1, K, "uniform", cfg["seed"])
    Bp, perm = inputs.permutation_b(K, 5)
    got, _, desc = run(A, Bp, out)
    want = A.view(np.float16)[:, perm]
    if out == "f16":
        assert np.array_equal(got.view(np.uint16), want.view(np.uint16)), desc
    else:
        assert np.array_equal(got, want.astype(np.float32)), desc
