"""Q4_0 weight-only matmul for one NVIDIA GB300 (sm_103a).

The compute lives in libq4_0.so (hand-written CUDA: a decode GEMV, a tcgen05
tensor-core GEMM and a quantizer); this package is its thin Python binding.
Build it with ``q4_weight_only_gb300.build.build()``.
"""
from ._lib import (ERR_CUDA, ERR_DEVICE_TIMEOUT, ERR_INVALID_ARG, ERR_UNSUPPORTED,
                   ERR_WORKSPACE, OK, Y_BF16, Y_F32, Q4Error, device_error, gemm, gemm_plan, gemv, gemv_alloc, lib, matmul,
                   matmul_alloc, matmul_grouped, grouped_launches, matmul_host, host_workspace_bytes, quantize, selftest_wait_timeout, status_string, version,
                   weight_bytes)

__all__ = ["quantize", "matmul", "matmul_alloc", "matmul_grouped", "grouped_launches", "matmul_host", "host_workspace_bytes", "gemv", "gemv_alloc", "gemm", "gemm_plan", "weight_bytes", "device_error",
           "version", "status_string", "lib", "selftest_wait_timeout", "Q4Error", "OK", "ERR_INVALID_ARG",
           "ERR_UNSUPPORTED", "ERR_CUDA", "ERR_DEVICE_TIMEOUT", "ERR_WORKSPACE", "Y_F32", "Y_BF16"]
