"""gemm_bias_relu_tf32_noalloc -- the TF32 GEMM + bias + ReLU for callers that
cannot allocate device memory (serving loops that must stay out of allocators,
plug-ins whose host framework owns device allocation, processes whose device
memory is reserved by another allocator).  Its scratch is a fixed device array
inside the library, so its output must match the regular entry point's,
call after call, although every call reuses the same array.

Collected last (file name) so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process,
where its first call is the library's first call on the device."""
import ctypes

import numpy as np
import pytest
import torch

from mbarrier_gemm_pipelines_gb300 import inputs
from gpu_helpers import TOL, load_library, rel_frobenius, require_gpu, to_host_f64

pytestmark = pytest.mark.gpu


def _noalloc(lib, A, B, bias, C, stages):
    M, K = A.shape
    N = B.shape[1]
    return lib.gemm_bias_relu_tf32_noalloc(A.data_ptr(), B.data_ptr(), bias.data_ptr(),
                                           C.data_ptr(), M, N, K, stages,
                                           torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_regular_entry_point_twice():
    require_gpu()
    gbr = load_library()
    from mbarrier_gemm_pipelines_gb300 import _binding as b
    lib = b.lib()
    # Two calls in a row with different shapes: the second reuses the scratch
    # array the first one left behind.
    for M, N, K, seed in [(300, 520, 200, 21), (640, 1024, 2048, 22)]:
        A, B, bias = inputs.gemm_normal(M, N, K, seed=seed)
        dA, dB, dbias = A.cuda(), B.cuda(), bias.cuda()
        C = torch.full((M, N), float("nan"), device="cuda")
        assert _noalloc(lib, dA, dB, dbias, C, 3) == b.OK, b.last_error()
        gbr.check_device()
        ref = gbr.gemm_bias_relu(dA, dB, dbias, dtype="tf32", stages=3)
        gbr.check_device()
        got, want = to_host_f64(C), to_host_f64(ref)
        assert np.isfinite(got).all()
        assert rel_frobenius(got, want) <= TOL["tf32"]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    require_gpu()
    load_library()
    from mbarrier_gemm_pipelines_gb300 import _binding as b
    lib = b.lib()
    M, N, K = 128, 2048, 2052          # K * N > 4194304
    A = torch.zeros((M, K), device="cuda")
    B = torch.zeros((K, N), device="cuda")
    bias = torch.zeros(N, device="cuda")
    C = torch.zeros((M, N), device="cuda")
    before = lib.gbr_launch_count()
    assert _noalloc(lib, A, B, bias, C, 3) == b.ERR_INVALID
    assert "16 MiB" in b.last_error()
    assert lib.gbr_launch_count() == before
