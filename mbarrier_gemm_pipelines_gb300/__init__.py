"""Warp-specialized TMA/mbarrier pipelines for GB300 (sm_103a).

Operators (C ABI in ``include/gbr.h``; this package is a thin ctypes binding):

* ``gemm_bias_relu``          C = ReLU(A @ B + bias); bf16 / TF32 on tcgen05
                              tensor cores, strict fp32 on CUDA cores (FFMA).
* ``gemm_bias_relu_grouped``  the same per expert segment in one launch.
* ``staged_copy``             TMA gmem -> smem -> gmem through an S-slot ring.
"""
from ._binding import (BF16, F32_FFMA, F32_TF32, OP_COPY, OP_GEMM, GbrError, check, check_device,
                       copy_tuning, device_status, ffma_tuning, gemm_dynamic_schedule, gemm_split_tail,
                       gemm_thin_tail, gemm_tuning, gemm_bias_relu, gemm_bias_relu_grouped,
                       gemm_bias_relu_host, launch_overlap,
                       last_error, launch_count, lib, library_path, max_stages,
                       gemm_bias_relu_tf32_noalloc, selftest_copy_skip_load, selftest_gemm_skip_load,
                       selftest_noalloc_skip_load, selftest_wait_timeout,
                       set_wait_timeout_ns, sm_count, staged_copy)
from ._build import build

__all__ = [
    "BF16", "F32_FFMA", "F32_TF32", "OP_COPY", "OP_GEMM", "GbrError", "build", "check",
    "check_device", "copy_tuning", "device_status", "ffma_tuning", "gemm_dynamic_schedule", "gemm_split_tail", "gemm_thin_tail", "gemm_tuning", "gemm_bias_relu", "gemm_bias_relu_grouped", "gemm_bias_relu_host",
    "last_error", "launch_count", "launch_overlap", "lib", "library_path", "max_stages", "selftest_copy_skip_load",
    "selftest_gemm_skip_load", "selftest_wait_timeout", "gemm_bias_relu_tf32_noalloc",
    "selftest_noalloc_skip_load",
    "set_wait_timeout_ns", "sm_count", "staged_copy",
]
