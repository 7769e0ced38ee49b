"""GPU parity of the stream-K tail (partial last wave split into K-block
ranges across all persistent workers, partial tiles summed through the plan's
workspace in contributor order) for the single-CTA and the CTA-pair kernels.

Small grids force many contributors per tile and many units per worker;
integer inputs must stay bit-exact; repeated runs of one plan (whose ticket
words carry over from run to run) must give identical bits.
"""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_fp16_gb300 import inputs

from gpu_util import assert_close, assert_exact, full_reference, record_error, run, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


CASES = [
    # variant, M, N, K, grid, block_n
    ("persistent", 390, 776, 456, 5, 128),
    ("persistent", 129, 136, 1000, 4, 64),
    ("persistent", 64, 2048, 4096, 0, 128),      # every tile shared by the full grid
    ("persistent_2cta", 700, 1000, 520, 10, 256),
    ("persistent_2cta", 300, 264, 2048, 6, 256),
    ("persistent_2cta", 1280, 1024, 320, 14, 256),
    ("persistent_2cta", 700, 1000, 520, 10, 128),
    ("persistent_2cta", 520, 1000, 776, 8, 224),     # fp16: 32-column remainder stored directly
]

# the CTA-pair kernel with stages of K = 128: stream-K ranges are counted in
# such stages, and an odd block count leaves the last stage half past K
CASES_K128 = [
    ("persistent_2cta", 700, 1000, 520, 10, 256),
    ("persistent_2cta", 1280, 1024, 328, 14, 224),
    ("persistent_2cta", 300, 264, 2048, 6, 256),     # 4 tiles over 3 pairs
]


@pytest.mark.parametrize("variant,M,N,K,grid,bn", CASES)
@pytest.mark.parametrize("out", ["f32", "f16"])
def test_stream_k_matches_oracle(variant, M, N, K, grid, bn, out):
    A, B = inputs.make_operands(M, N, K, "normal", 500 + M + K)
    got, guard, desc = run(A, B, out, guard_rows=2, variant=variant, grid=grid, block_n=bn,
                           stream_k="on")
    assert "stream_k=0/" not in desc, desc
    assert_close(got, oracle.gemm(A, B), K, out, desc)
    assert np.isnan(guard.astype(np.float32)).all()


@pytest.mark.parametrize("variant,M,N,K,grid,bn", CASES_K128)
@pytest.mark.parametrize("out", ["f32", "f16"])
def test_stream_k_with_128_wide_stages(variant, M, N, K, grid, bn, out):
    A, B = inputs.make_operands(M, N, K, "normal", 700 + M + K)
    got, guard, desc = run(A, B, out, guard_rows=2, variant=variant, grid=grid, block_n=bn,
                           stream_k="on", block_k=128)
    assert "stream_k=0/" not in desc and "x128 " in desc, desc
    assert_close(got, oracle.gemm(A, B), K, out, desc)
    assert np.isnan(guard.astype(np.float32)).all()
    Ai, Bi = inputs.make_operands(M, N, K, "int", 19)
    goti, _, _ = run(Ai, Bi, out, variant=variant, grid=grid, block_n=bn, stream_k="on",
                     block_k=128)
    assert_exact(goti, oracle.gemm(Ai, Bi), out, desc)


@pytest.mark.parametrize("variant,M,N,K,grid,bn", CASES[:2] + CASES[3:5])
def test_stream_k_integer_bit_exact(variant, M, N, K, grid, bn):
    A, B = inputs.make_operands(M, N, K, "int", 9)
    for out in ("f32", "f16"):
        got, _, desc = run(A, B, out, variant=variant, grid=grid, block_n=bn, stream_k="on")
        assert_exact(got, oracle.gemm(A, B), out, desc)


@pytest.mark.parametrize("variant", ["persistent", "persistent_2cta"])
def test_stream_k_runs_are_bit_identical(variant):
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    M, N, K = 520, 768, 2000
    A, B = inputs.make_operands(M, N, K, "uniform", 31)
    dA, dB = to_device(A), to_device(B)
    grid = 7 if variant == "persistent" else 4
    plan = pkg.Plan(M, N, K, out="f32", variant=variant, grid=grid, block_n=128 if
                    variant == "persistent" else 256, stream_k="on")
    assert plan.config()["sk_tiles"] > 0
    outs = []
    for _ in range(4):
        C = torch.empty((M, N), dtype=torch.float32, device="cuda")
        plan(dA, dB, C)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        outs.append(C.cpu().numpy())
    plan.close()
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))
    assert_close(outs[0], oracle.gemm(A, B), K, "f32", variant)


def test_stream_k_off_and_on_agree_within_tolerance():
    M, N, K = 4000, 3000, 5000
    A, B = inputs.make_operands(M, N, K, "normal", 3)
    # 256-wide pair tiles leave a partial last wave (192 tiles over 76 pairs)
    on, _, d_on = run(A, B, "f32", stream_k="on", block_n=256)
    off, _, d_off = run(A, B, "f32", block_n=256)
    assert "stream_k=0/" in d_off and "stream_k=0/" not in d_on
    assert np.max(np.abs(on.astype(np.float64) - off)) <= 1e-3 * np.sqrt(K)


@pytest.mark.parametrize("cfg", [c for c in inputs.CONFIGS if c["M"] >= 64 and c["K"] >= 4096],
                         ids=lambda c: c["name"])
def test_stream_k_workloads_every_entry(cfg):
    # the full-size workloads with the stream-K tail switched on
    M, N, K, out = cfg["M"], cfg["N"], cfg["K"], cfg["out"]
    A, B, ref = full_reference(cfg)
    got, _, desc = run(A, B, out, stream_k="on", block_n=256 if M > 128 else 0)
    assert "stream_k=0/" not in desc, desc
    record_error("%s (stream-K tail)" % cfg["name"], got, ref, K, out)
    assert_close(got, ref, K, out, desc)
