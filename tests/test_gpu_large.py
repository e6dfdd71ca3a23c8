"""Maximum-size edge cases: outputs with more than 2^31 elements (bf16) or
more than 2^32 bytes, a copy of more than 2^31 elements, and the largest
expert count of the grouped call.  Checked at sampled positions (the oracle
evaluates each one), including the last row and column, where 32-bit index
arithmetic would first go wrong."""
import numpy as np
import pytest
import torch

import oracle
from mbarrier_gemm_pipelines_gb300 import inputs
from gpu_helpers import TOL, load_library, rel_frobenius, require_gpu, sample_points

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbr():
    require_gpu()
    return load_library()


def _sampled(gbr, M, N, K, dtype, seed):
    A, B, bias = inputs.gemm_normal(M, N, K, seed=seed)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype=dtype, stages=3)
    gbr.check_device()
    ms, ns = sample_points(M, N, 2000, seed, extra_rows=(M - 1, M // 2 + 1), extra_cols=(N - 1,))
    got = C[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()].double().cpu().numpy()
    ref = oracle.gemm_bias_relu_points(A.float(), B.float(), bias, ms, ns)
    del C
    torch.cuda.empty_cache()
    assert rel_frobenius(got, ref) <= TOL[dtype]


def test_bf16_output_over_2_31_elements(gbr):
    _sampled(gbr, 49152, 49152, 128, "bf16", seed=80)        # 2.42e9 outputs, 4.8 GB


@pytest.mark.parametrize("dtype", ["ffma", "tf32"])
def test_fp32_output_over_2_32_bytes(gbr, dtype):
    _sampled(gbr, 36864, 32768, 64, dtype, seed=81)          # 1.2e9 outputs, 4.8 GB


def test_copy_over_2_31_elements(gbr):
    rows, cols = 65536, 33792                                # 2.21e9 fp32, 8.9 GB each way
    src = torch.empty((rows, cols), device="cuda")
    bits = src.view(torch.int32)
    col = torch.arange(cols, device="cuda", dtype=torch.int32)
    for r0 in range(0, rows, 4096):                          # every element distinct per row band
        r = torch.arange(r0, r0 + 4096, device="cuda", dtype=torch.int32)[:, None]
        bits[r0:r0 + 4096] = r * 33797 + col
    dst = gbr.staged_copy(src, tile=(128, 64), stages=4)
    gbr.check_device()
    assert torch.equal(dst.view(torch.int32), src.view(torch.int32))


def test_grouped_largest_expert_count(gbr):
    G = 32                                                   # kMaxGroups
    g = torch.Generator().manual_seed(82)
    counts = [int(c) for c in torch.randint(0, 300, (G,), generator=g)]
    counts[5] = 0
    _, X, W, b = inputs.grouped(tokens=sum(counts), experts=G, K=128, N=264, seed=82)
    C = gbr.gemm_bias_relu_grouped(X.cuda(), W.cuda(), b.cuda(), counts, stages=3)
    gbr.check_device()
    ref = oracle.gemm_bias_relu_grouped(X.float(), W.float(), b, counts)
    assert rel_frobenius(C.double().cpu().numpy(), ref) <= TOL["bf16"]
    with pytest.raises(gbr.GbrError):
        gbr.gemm_bias_relu_grouped(X.cuda(), torch.zeros((33, 128, 264), dtype=torch.bfloat16,
                                                         device="cuda"),
                                   torch.zeros((33, 264), device="cuda"), counts + [0], stages=3)
