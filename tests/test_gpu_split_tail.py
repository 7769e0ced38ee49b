"""GPU parity of the dynamic pair schedule's split tail (stream_k = 2).

When the tiles do not fill whole waves of clusters, the tiles of the partial
last wave (all tiles, when there are fewer tiles than clusters) are each cut
into S equal K ranges run as separate units; the S partial tiles meet in the
workspace and the last to arrive sums them in K order and stores the tile.

Covers S = 2 and S = 4, a ragged K whose ranges differ by one stage, both
output types against the full oracle, integer inputs bit-exact (the partial
sums are exact), the 8192^3 workload sampled, identical results run to run
and from launch to launch of one plan, agreement with whole tiles within the
tolerance, a captured CUDA graph (which runs every tile whole), and the
watchdog with a split plan.
"""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_fp16_gb300 import inputs

from gpu_util import assert_close, assert_exact, full_reference, record_error, run, run_repeated

pytestmark = pytest.mark.gpu
V = "dynamic_2cta"
ON = {"variant": V, "stream_k": "on"}


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _split(M, N, K, out, **opts):
    from tma_pipelined_tensor_fp16_gb300 import binding
    opts.setdefault("stream_k", "on")
    st, c = binding.gemm_select_config(M, N, K, 1 if out == "f16" else 0,
                                       binding.make_options(variant=V, **opts))
    assert st == 0, binding.last_error()
    return c


@pytest.mark.parametrize("out", ["f32", "f16"])
@pytest.mark.parametrize("M,N,K,bn,splits", [(1024, 1024, 4096, 256, 4),   # 16 tiles, 64 units
                                             (1024, 1024, 1024, 256, 2),   # 8 stages: 2 x 4
                                             (1000, 1000, 520, 0, 2),      # 9 stages: 4 + 5
                                             (1500, 1000, 2056, 192, 2)])  # ragged everywhere
def test_split_tiles_match_oracle(out, M, N, K, bn, splits):
    c = _split(M, N, K, out, block_n=bn)
    assert c.sk_tiles > 0 and c.sk_max_contrib == splits, (c.sk_tiles, c.sk_max_contrib)
    A, B = inputs.make_operands(M, N, K, "normal", 40 + K)
    got, guard, desc = run(A, B, out, guard_rows=2, block_n=bn, **ON)
    assert_close(got, oracle.gemm(A, B), K, out, desc)
    assert np.isnan(guard.astype(np.float32)).all(), "wrote past the end of C"
    Ai, Bi = inputs.make_operands(M, N, K, "int", 41)
    goti, _, _ = run(Ai, Bi, out, block_n=bn, **ON)
    assert_exact(goti, oracle.gemm(Ai, Bi), out, desc)


def test_split_tail_of_the_8192_workload():
    cfg = next(c for c in inputs.CONFIGS if c["M"] == 8192)
    M, N, K, out = cfg["M"], cfg["N"], cfg["K"], cfg["out"]
    c = _split(M, N, K, out)
    assert (c.dp_tiles, c.sk_tiles, c.sk_max_contrib) == (988, 36, 2)
    A, B, ref = full_reference(cfg)
    got, _, desc = run(A, B, out, **ON)
    assert not np.isnan(got.astype(np.float32)).any(), desc
    record_error("%s (dynamic split tail)" % cfg["name"], got, ref, K, out)
    assert_close(got, ref, K, out, desc)
    again, _, _ = run(A, B, out, **ON)
    assert np.array_equal(got.view(np.uint16), again.view(np.uint16)), "run-to-run difference"
    whole, _, _ = run(A, B, out, variant=V)
    assert_close(got.astype(np.float64), whole.astype(np.float64), K, out, "split vs whole")


def test_split_plan_launched_repeatedly():
    M, N, K = 1024, 1024, 4096
    A, B = inputs.make_operands(M, N, K, "uniform", 42)
    outs = run_repeated(A, B, "f16", 5, block_n=256, **ON)
    ref = outs[0]
    assert_close(ref, oracle.gemm(A, B), K, "f16", "split, repeated")
    for i, o in enumerate(outs[1:], 1):
        assert np.array_equal(o.view(np.uint16), ref.view(np.uint16)), "launch %d differs" % i


def test_split_plan_captured_in_a_graph_runs_whole_tiles():
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    from gpu_util import to_device
    M, N, K = 1024, 1024, 4096
    A, B = inputs.make_operands(M, N, K, "uniform", 43)
    dA, dB = to_device(A), to_device(B)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    plan = pkg.Plan(M, N, K, out="f32", block_n=256, **ON)
    assert plan.config()["sk_tiles"] == 16
    st = torch.cuda.Stream()
    plan(dA, dB, C, stream=st)  # first launch outside the capture
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for _ in range(2):
            plan(dA, dB, C, stream=st)
    ref = oracle.gemm(A, B)
    for _ in range(3):
        with torch.cuda.stream(st):
            C.fill_(float("nan"))
        g.replay()
        st.synchronize()
        assert plan.device_status() == 0, pkg.gemm_last_error()
        assert_close(C.cpu().numpy(), ref, K, "f32", "graph replay of a split plan")
    plan.close()


def test_split_plan_watchdog_timeout():
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    from tma_pipelined_tensor_fp16_gb300 import binding
    M, N, K = 1024, 1024, 4096
    A, B = inputs.make_operands(M, N, K, "uniform", 44)
    dA = torch.from_numpy(A.view(np.float16)).cuda()
    dB = torch.from_numpy(B.view(np.float16)).cuda()
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    plan = pkg.Plan(M, N, K, out="f32", block_n=256, debug_stall=1, wait_budget_ms=100,
                    **ON)
    assert plan.config()["sk_tiles"] == 16
    plan(dA, dB, C)
    torch.cuda.synchronize()
    assert plan.device_status() == binding.GEMM_ERR_TIMEOUT
    plan.close()
    got, _, desc = run(A, B, "f32", block_n=256, **ON)
    assert_close(got, oracle.gemm(A, B), K, "f32", "after timeout: " + desc)
