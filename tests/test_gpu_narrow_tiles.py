"""GPU parity of the dynamic pair schedule's narrow tiles.

When all 256 x 256 tiles fit in at most half the resident clusters, each tile
is computed as two 256 x 128 tiles on two clusters (B through a second tensor
map whose box is half as high).  A half walks the same K blocks in the same
order as the whole tile, so every output is the same fp32 sum: the result is
identical bit for bit to the whole-tile plan's.

Covers one tile, ragged M and N (a right half partly or wholly past N), both
output types against the oracle, integer inputs bit-exact, identity with whole
tiles, repeated launches, graph capture and the watchdog.
"""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_fp16_gb300 import inputs

from gpu_util import assert_close, assert_exact, run, run_repeated

pytestmark = pytest.mark.gpu
NARROW = {"variant": "dynamic_2cta", "block_n": 256}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _halves(M, N, K, out):
    from tma_pipelined_tensor_fp16_gb300 import binding
    st, c = binding.gemm_select_config(M, N, K, 1 if out == "f16" else 0,
                                       binding.make_options(**NARROW))
    assert st == 0, binding.last_error()
    return c.tail_halves


@pytest.mark.parametrize("out", ["f32", "f16"])
@pytest.mark.parametrize("shape", [(256, 256, 128), (1024, 1024, 4096), (1024, 1000, 4096),
                                   (700, 2000, 1024), (300, 800, 2112)],
                         ids=lambda s: "x".join(map(str, s)))
def test_narrow_tiles_match_oracle_and_whole_tiles(out, shape):
    M, N, K = shape
    assert _halves(M, N, K, out) > 0
    A, B = inputs.make_operands(M, N, K, "normal", 60 + M + N)
    got, guard, desc = run(A, B, out, guard_rows=2, **NARROW)
    assert "tail_halves=" in desc and "tail_halves=0" not in desc, desc
    assert_close(got, oracle.gemm(A, B), K, out, desc)
    assert np.isnan(guard.astype(np.float32)).all(), "wrote past the end of C"
    whole, _, desc_w = run(A, B, out, stream_k="off", **NARROW)
    assert "tail_halves=0" in desc_w
    assert np.array_equal(got.view(np.uint8), whole.view(np.uint8)), (desc, desc_w)
    Ai, Bi = inputs.make_operands(M, N, K, "int", 61)
    goti, _, _ = run(Ai, Bi, out, **NARROW)
    assert_exact(goti, oracle.gemm(Ai, Bi), out, desc)


def test_narrow_plan_launched_repeatedly():
    M, N, K = 1024, 1024, 4096
    A, B = inputs.make_operands(M, N, K, "uniform", 62)
    outs = run_repeated(A, B, "f16", 5, **NARROW)
    assert_close(outs[0], oracle.gemm(A, B), K, "f16", "narrow, repeated")
    for i, o in enumerate(outs[1:], 1):
        assert np.array_equal(o.view(np.uint16), outs[0].view(np.uint16)), "launch %d" % i


def test_narrow_plan_captured_in_a_graph():
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    from gpu_util import to_device
    M, N, K = 768, 1024, 2048
    A, B = inputs.make_operands(M, N, K, "uniform", 63)
    dA, dB = to_device(A), to_device(B)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    plan = pkg.Plan(M, N, K, out="f32", **NARROW)
    assert plan.config()["tail_halves"] == 12
    st = torch.cuda.Stream()
    plan(dA, dB, C, stream=st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for _ in range(2):
            plan(dA, dB, C, stream=st)
    ref = oracle.gemm(A, B)
    for _ in range(2):
        with torch.cuda.stream(st):
            C.fill_(float("nan"))
        g.replay()
        st.synchronize()
        assert plan.device_status() == 0, pkg.gemm_last_error()
        assert_close(C.cpu().numpy(), ref, K, "f32", "graph replay, narrow tiles")
    plan.close()


def test_narrow_plan_watchdog_timeout():
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    from tma_pipelined_tensor_fp16_gb300 import binding
    M, N, K = 1024, 1024, 4096
    A, B = inputs.make_operands(M, N, K, "uniform", 64)
    dA = torch.from_numpy(A.view(np.float16)).cuda()
    dB = torch.from_numpy(B.view(np.float16)).cuda()
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    plan = pkg.Plan(M, N, K, out="f32", debug_stall=1, wait_budget_ms=100, **NARROW)
    assert plan.config()["tail_halves"] == 16
    plan(dA, dB, C)
    torch.cuda.synchronize()
    assert plan.device_status() == binding.GEMM_ERR_TIMEOUT
    plan.close()
    got, _, desc = run(A, B, "f32", **NARROW)
    assert_close(got, oracle.gemm(A, B), K, "f32", "after timeout: " + desc)
