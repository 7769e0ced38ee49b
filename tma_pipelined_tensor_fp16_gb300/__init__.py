"""GB300-native (sm_103a) TMA-pipelined fp16 GEMM  C = A . B^T.

The GEMM is the C-ABI library ``libtmagemm.so`` (declared in
``include/tmagemm.h``, built by ``build.py`` from ``csrc/``); ``binding``
exposes its entry points under the same names.  ``inputs`` generates the
seeded synthetic operands used by the tests and the benchmark.
"""
from .binding import (  # noqa: F401
    GEMM_OUT_F16, GEMM_OUT_F32, GemmError, Plan, VARIANTS, gemm_create_plan,
    gemm_create_plan_ex, gemm_destroy, gemm_get_device_status, gemm_last_error,
    gemm_last_status, gemm_plan_config, gemm_plan_describe, gemm_run, gemm_run_host,
    gemm_schedule_tile, gemm_select_config, gemm_sw128_offset, make_options)
