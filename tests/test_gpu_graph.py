"""gemm_run captured into a CUDA graph and replayed.

A plan's launches are captured once (after one ordinary launch, which sets
the kernel's shared-memory limit outside the capture) and replayed; every
replay must write the same, correct C as a direct launch.  Covers the dynamic
CTA-pair kernel (a grid whose clusters cancel one another through cluster
launch control) and the single-CTA persistent kernel; and that a plan with
stream-K tiles refuses to be captured (its fix-up tickets are keyed by the
run counter, which a replay repeats).
"""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_fp16_gb300 import inputs

from gpu_util import assert_close, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("M,N,K,variant", [(2304, 2560, 320, "dynamic_2cta"),
                                           (256, 256, 256, "persistent")])
def test_launches_captured_in_a_graph(M, N, K, variant):
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    A, B = inputs.make_operands(M, N, K, "uniform", 91)
    dA, dB = to_device(A), to_device(B)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    plan = pkg.Plan(M, N, K, out="f32", variant=variant)
    st = torch.cuda.Stream()
    plan(dA, dB, C, stream=st)  # first launch outside the capture
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for _ in range(3):
            plan(dA, dB, C, stream=st)
    ref = oracle.gemm(A, B)
    for _ in range(2):
        with torch.cuda.stream(st):
            C.fill_(float("nan"))
        g.replay()
        st.synchronize()
        assert plan.device_status() == 0, pkg.gemm_last_error()
        got = C.cpu().numpy()
        assert_close(got, ref, K, "f32", "graph replay, %s" % plan.describe())
    plan.close()


def test_stream_k_plan_refuses_capture():
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    from tma_pipelined_tensor_fp16_gb300 import binding
    M, N, K = 1000, 1000, 520
    A, B = inputs.make_operands(M, N, K, "uniform", 92)
    dA, dB = to_device(A), to_device(B)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    plan = pkg.Plan(M, N, K, out="f32", variant="persistent_2cta", grid=10, stream_k="on")
    assert plan.config()["sk_tiles"] > 0
    st = torch.cuda.Stream()
    plan(dA, dB, C, stream=st)
    st.synchronize()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(binding.GemmError) as e:
        with torch.cuda.graph(g, stream=st):
            plan(dA, dB, C, stream=st)
    assert e.value.status == binding.GEMM_ERR_UNSUPPORTED
    plan.close()
