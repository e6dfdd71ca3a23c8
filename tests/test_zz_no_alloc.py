"""gemm_bias_relu_tf32_noalloc -- the TF32 GEMM + bias + ReLU for callers that
cannot allocate device memory (serving loops that must stay out of allocators,
plug-ins whose host framework owns device allocation, processes whose device
memory is reserved by another allocator).  Its status words sit in a fixed
device array inside the library that every call on the device reuses, so its
output is checked against the binary64 oracle call after call, at the TF32 bar.

Collected last (file name) so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process,
where its first call is the library's first call on the device."""
import numpy as np
import pytest
import torch

import oracle
from mbarrier_gemm_pipelines_gb300 import inputs
from gpu_helpers import TOL, load_library, rel_frobenius, require_gpu, to_host_f64

pytestmark = pytest.mark.gpu


def _noalloc(lib, A, B, bias, C, stages):
    """The raw C-ABI call, with the sizes taken from A and B."""
    M, K = A.shape
    N = B.shape[1]
    return lib.gemm_bias_relu_tf32_noalloc(A.data_ptr(), B.data_ptr(), bias.data_ptr(),
                                           C.data_ptr(), M, N, K, stages,
                                           torch.cuda.current_stream().cuda_stream)


def _check_oracle(C, A, B, bias):
    got = to_host_f64(C)
    ref = oracle.gemm_bias_relu(A, B, bias)
    assert np.isfinite(got).all()
    assert rel_frobenius(got, ref) <= TOL["tf32"]
    assert np.abs(got - ref).max() <= 20 * TOL["tf32"] * (np.abs(ref).max() + 1e-30)


def test_noalloc_matches_oracle_twice():
    require_gpu()
    gbr = load_library()
    from mbarrier_gemm_pipelines_gb300 import _binding as b
    lib = b.lib()
    # Two calls in a row with different shapes: the second reuses the status
    # words the first one left behind.
    for M, N, K, seed in [(640, 1024, 2048, 22), (300, 520, 200, 21)]:
        A, B, bias = inputs.gemm_normal(M, N, K, seed=seed)
        C = torch.full((M, N), float("nan"), device="cuda")
        assert _noalloc(lib, A.cuda(), B.cuda(), bias.cuda(), C, 3) == b.OK, b.last_error()
        gbr.check_device()
        _check_oracle(C, A, B, bias)


def test_noalloc_large_b_and_index_limit():
    """B of 2052 x 2048 fp32 (16.0 MiB, read in place: no copy of it is made),
    against the oracle; sizes of 2^31 or more are rejected with nothing
    launched."""
    require_gpu()
    gbr = load_library()
    from mbarrier_gemm_pipelines_gb300 import _binding as b
    lib = b.lib()
    M, N, K = 136, 2048, 2052
    A, B, bias = inputs.gemm_normal(M, N, K, seed=25)
    C = torch.full((M, N), float("nan"), device="cuda")
    assert _noalloc(lib, A.cuda(), B.cuda(), bias.cuda(), C, 4) == b.OK, b.last_error()
    gbr.check_device()
    _check_oracle(C, A, B, bias)
    before = lib.gbr_launch_count()
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.gemm_bias_relu_tf32_noalloc(C.data_ptr(), C.data_ptr(), C.data_ptr(), C.data_ptr(),
                                           1 << 31, 4, 4, 3, stream) == b.ERR_INVALID
    assert "2^31" in b.last_error()
    assert lib.gbr_launch_count() == before


def test_noalloc_rejects_overlap_and_deep_rings():
    require_gpu()
    gbr = load_library()
    from mbarrier_gemm_pipelines_gb300 import _binding as b
    lib = b.lib()
    A, B, bias = inputs.gemm_normal(256, 256, 256, seed=23)
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    C = torch.empty((256, 256), device="cuda")
    before = lib.gbr_launch_count()
    assert _noalloc(lib, dA, dB, db, dA, 3) == b.ERR_INVALID      # C is A
    assert "overlap" in b.last_error()
    assert _noalloc(lib, dA, dB, db, dB, 3) == b.ERR_INVALID      # C is B
    # One CTA per tile: 4 stages at most, although the pair kernel holds more.
    assert gbr.max_stages(gbr.OP_GEMM, gbr.F32_TF32) > 4
    assert _noalloc(lib, dA, dB, db, C, 5) == b.ERR_SMEM
    assert "[1, 4]" in b.last_error()
    assert _noalloc(lib, dA, dB, db, C, 0) == b.ERR_SMEM
    assert lib.gbr_launch_count() == before
    assert _noalloc(lib, dA, dB, db, C, 4) == b.OK
    gbr.check_device()
    _check_oracle(C, A, B, bias)


def test_noalloc_python_wrapper_checks_shapes():
    require_gpu()
    gbr = load_library()
    A = torch.zeros((64, 32), device="cuda")
    B = torch.zeros((32, 96), device="cuda")
    bias = torch.zeros(96, device="cuda")
    before = gbr.launch_count()
    for args in ((A, B, bias, torch.zeros((64, 64), device="cuda")),       # C too narrow
                 (A, torch.zeros((40, 96), device="cuda"), bias,           # K mismatch
                  torch.zeros((64, 96), device="cuda")),
                 (A, B, torch.zeros(64, device="cuda"),                    # bias length
                  torch.zeros((64, 96), device="cuda"))):
        with pytest.raises(ValueError):
            gbr.gemm_bias_relu_tf32_noalloc(*args, stages=3)
    with pytest.raises(TypeError):
        gbr.gemm_bias_relu_tf32_noalloc(A, B, bias, torch.zeros((64, 96), device="cuda",
                                                                dtype=torch.bfloat16))
    assert gbr.launch_count() == before


def test_noalloc_timeout_is_reported_then_cleared():
    """A stage left unfilled on the host's instruction (50 ms limit): the
    kernel gives up, records the timeout in the no-alloc array's status words
    and returns; gbr_device_status reports it once, and the next call is
    correct again."""
    require_gpu()
    gbr = load_library()
    A, B, bias = inputs.gemm_normal(384, 512, 640, seed=24)
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    C = torch.empty((384, 512), device="cuda")
    gbr.selftest_noalloc_skip_load(dA, dB, db, C, stages=3, cta=1, item=2,
                                   limit_ns=50_000_000)
    assert gbr.device_status() == 6                    # GBR_ERR_TIMEOUT
    msg = gbr.last_error()
    assert "gemm_bias_relu_tf32_noalloc" in msg and "CTA 1" in msg
    assert gbr.device_status() == 0                    # read once, then cleared
    gbr.gemm_bias_relu_tf32_noalloc(dA, dB, db, C, stages=3)
    gbr.check_device()
    _check_oracle(C, A, B, bias)


def _noalloc_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        M = int(rng.integers(1, 3000))
        N = 32 * int(rng.integers(1, 60)) if rng.random() < 0.5 else 4 * int(rng.integers(1, 500))
        K = 4 * int(rng.integers(1, 500))
        S = int(rng.integers(1, 5))
        cases.append(pytest.param(M, N, K, S, id="n%02d-%dx%dx%d-s%d" % (i, M, N, K, S)))
    return cases


@pytest.mark.parametrize("M,N,K,S", _noalloc_cases(12, 9090))
def test_noalloc_random(M, N, K, S):
    """Seeded random shapes (N a whole number of 32-column B panels or only a
    multiple of 4, every ring depth the call accepts) against the oracle."""
    require_gpu()
    gbr = load_library()
    from mbarrier_gemm_pipelines_gb300 import _binding as b
    A, B, bias = inputs.gemm_normal(M, N, K, seed=M + N + K + S)
    C = torch.full((M, N), float("nan"), device="cuda")
    assert _noalloc(b.lib(), A.cuda(), B.cuda(), bias.cuda(), C, S) == b.OK, b.last_error()
    gbr.check_device()
    _check_oracle(C, A, B, bias)
