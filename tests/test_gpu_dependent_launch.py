"""Ordering of the programmatic dependent launch.

The warp-specialised kernels are launched as programmatic dependents of the
work before them on the stream: their CTAs may start (barriers, TMEM) while the
previous kernel drains, and wait for it to complete (griddepcontrol.wait)
before touching global memory.  These tests put a producer of a GEMM's
operand immediately before the GEMM on the same stream, after poisoning that
operand with NaN, so any read that raced ahead of the producer would carry
NaN into C:

* a torch kernel that writes A (an exact negation);
* a GEMM whose fp16 output is the next GEMM's A operand (chained GEMMs), for
  the CTA-pair kernel feeding the single-CTA kernel, the two-pairs-per-cluster
  kernel, and the other way round.
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


@pytest.mark.parametrize("variant", ["dynamic_2cta", "persistent", "persistent_2cta"])
def test_operand_written_by_the_previous_kernel(variant):
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    M, N, K = 1536, 1280, 1024
    A, B = inputs.make_operands(M, N, K, "uniform", 131)
    neg_src = -to_device(A)  # exact in fp16
    dB = to_device(B)
    dA = torch.empty_like(neg_src)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    plan = pkg.Plan(M, N, K, out="f32", variant=variant)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for _ in range(4):
            dA.fill_(float("nan"))
            C.fill_(float("nan"))
            torch.neg(neg_src, out=dA)  # the kernel the GEMM depends on
            plan(dA, dB, C, stream=st)
    st.synchronize()
    assert plan.device_status() == 0, pkg.gemm_last_error()
    assert_close(C.cpu().numpy(), oracle.gemm(A, B), K, "f32",
                 "A written just before, %s" % plan.describe())
    plan.close()


@pytest.mark.parametrize("first,second", [("dynamic_2cta", "persistent"),
                                          ("persistent", "dynamic_2cta"),
                                          ("persistent_2cta", "dynamic_2cta"),
                                          ("dynamic_2cta", "persistent_2cta")])
def test_chained_gemms(first, second):
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    M, N, K, N2 = 1024, 768, 512, 640
    A, B = inputs.make_operands(M, N, K, "uniform", 132)
    _, B2 = inputs.make_operands(8, N2, N, "uniform", 133)
    dA, dB, dB2 = to_device(A), to_device(B), to_device(B2)
    C1 = torch.empty((M, N), dtype=torch.float16, device="cuda")
    C2 = torch.empty((M, N2), dtype=torch.float32, device="cuda")
    p1 = pkg.Plan(M, N, K, out="f16", variant=first)
    p2 = pkg.Plan(M, N2, N, out="f32", variant=second)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        for _ in range(4):
            C1.fill_(float("nan"))
            C2.fill_(float("nan"))
            p1(dA, dB, C1, stream=st)
            p2(C1, dB2, C2, stream=st)  # reads what p1 has just written
    st.synchronize()
    assert p1.device_status() == 0 and p2.device_status() == 0, pkg.gemm_last_error()
    c1_bits = C1.cpu().numpy().view(np.uint16)
    assert_close(oracle.f16_to_f64(c1_bits), oracle.gemm(A, B), K, "f16",
                 "first GEMM, %s" % p1.describe())
    assert_close(C2.cpu().numpy(), oracle.gemm(c1_bits, B2), N, "f32",
                 "second GEMM on the first one's output, %s" % p2.describe())
    p1.close()
    p2.close()
