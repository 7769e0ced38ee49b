"""The allocation-free entry point gemm_run_noalloc, through the C ABI.

It exists for callers that cannot call cudaMalloc (device memory owned by a
framework allocator or a pre-reserved arena; loops that cannot pay the device
synchronisation of an allocation).  Its output must match gemm_run's -- the
existing entry point with a plan -- within the parity tolerance, on two calls
in a row (the second call reuses the shared static scratch array the first
one left behind).  The file is named to be collected last.
"""
import numpy as np
import pytest

from tma_pipelined_tensor_fp16_gb300 import inputs

from gpu_util import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def _with_plan(A, B, out):
    import torch

    import tma_pipelined_tensor_fp16_gb300 as pkg
    M, K = A.shape
    N = B.shape[0]
    dA = torch.from_numpy(A.view(np.float16)).cuda()
    dB = torch.from_numpy(B.view(np.float16)).cuda()
    C = torch.empty((M, N), dtype=torch.float16 if out == "f16" else torch.float32, device="cuda")
    plan = pkg.Plan(M, N, K, out=out)
    plan(dA, dB, C)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    plan.close()
    return C.cpu().numpy().astype(np.float64)


def _no_alloc(A, B, out, synchronous):
    import torch

    from tma_pipelined_tensor_fp16_gb300 import binding
    M, K = A.shape
    N = B.shape[0]
    dA = torch.from_numpy(A.view(np.float16)).cuda()
    dB = torch.from_numpy(B.view(np.float16)).cuda()
    C = torch.full((M, N), float("nan"),
                   dtype=torch.float16 if out == "f16" else torch.float32, device="cuda")
    torch.cuda.synchronize()
    dt = binding.GEMM_OUT_F16 if out == "f16" else binding.GEMM_OUT_F32
    s = torch.cuda.current_stream()
    st, ds = binding.gemm_run_noalloc(M, N, K, dt, dA.data_ptr(), dB.data_ptr(), C.data_ptr(),
                                      s.cuda_stream, want_status=synchronous)
    assert st == binding.GEMM_OK, binding.last_error()
    if synchronous:
        assert ds == binding.GEMM_OK
    torch.cuda.synchronize()
    return C.cpu().numpy().astype(np.float64)


def test_no_alloc_matches_gemm_run_on_two_calls_in_a_row():
    # small shapes take the single-CTA kernel; the last two have enough pair
    # tiles for the dynamic CTA-pair kernel (stages of K = 64 and of K = 128)
    cases = [((300, 264, 328), "f32", "uniform", 21, False),
             ((520, 392, 1000), "f16", "normal", 22, True),
             ((2560, 1024, 1000), "f16", "normal", 23, True),
             ((2560, 1040, 512), "f32", "uniform", 24, False)]
    for (M, N, K), out, dist, seed, sync in cases:
        A, B = inputs.make_operands(M, N, K, dist, seed)
        want = _with_plan(A, B, out)
        got = _no_alloc(A, B, out, sync)
        assert np.isfinite(got).all()
        assert_close(got, want, K, out, "gemm_run_noalloc vs gemm_run %dx%dx%d %s" % (M, N, K, out))


def test_no_alloc_rejects_bad_arguments():
    import torch

    from tma_pipelined_tensor_fp16_gb300 import binding
    a = torch.zeros(4096, dtype=torch.float16, device="cuda")
    st, _ = binding.gemm_run_noalloc(64, 64, 60, binding.GEMM_OUT_F16, a.data_ptr(),
                                     a.data_ptr(), a.data_ptr(), None, want_status=False)
    assert st == binding.GEMM_ERR_UNSUPPORTED  # K not a multiple of 8
    st, _ = binding.gemm_run_noalloc(64, 64, 64, binding.GEMM_OUT_F16, a.data_ptr() + 2,
                                     a.data_ptr(), a.data_ptr(), None, want_status=False)
    assert st == binding.GEMM_ERR_UNSUPPORTED  # misaligned A
