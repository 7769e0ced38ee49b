"""The in-kernel watchdog: every mbarrier wait is bounded.  A plan built with
``debug_stall`` makes the TMA producer first wait on a barrier that nothing
ever completes (no fault, no trap, no endless loop: a flag nobody sets).  The
wait must run out after ``wait_budget_ms``, the other roles and CTAs must see
the abort and give up, TMEM must be freed, and the host must read
GEMM_ERR_TIMEOUT from the status record -- after which the context is still
usable and a normal run on the same device is correct.
"""
import numpy as np
import pytest

import oracle
from tma_pipelined_tensor_fp16_gb300 import inputs

from gpu_util import assert_close, run

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("variant,block_k", [("persistent", 64), ("ws_pipelined", 64),
                                             ("persistent", 256), ("ws_pipelined", 128)])
def test_stalled_wait_times_out_and_context_survives(variant, block_k):
    import time

    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    from tma_pipelined_tensor_fp16_gb300 import binding
    M, N, K = 512, 512, 256
    A, B = inputs.make_operands(M, N, K, "uniform", 3)
    dA = torch.from_numpy(A.view(np.float16)).cuda()
    dB = torch.from_numpy(B.view(np.float16)).cuda()
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    plan = pkg.Plan(M, N, K, out="f32", variant=variant, debug_stall=1, wait_budget_ms=100,
                    block_k=block_k)
    t0 = time.time()
    plan(dA, dB, C)
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert plan.device_status() == binding.GEMM_ERR_TIMEOUT
    assert "timed out" in pkg.gemm_last_error()
    assert elapsed < 10.0
    # read-and-clear: the record is clean afterwards
    assert plan.device_status() == binding.GEMM_OK
    plan.close()
    # the context is intact: a normal run right after is correct
    got, _, desc = run(A, B, "f32", variant=variant, block_k=block_k)
    assert_close(got, oracle.gemm(A, B), K, "f32", "after timeout: " + desc)
