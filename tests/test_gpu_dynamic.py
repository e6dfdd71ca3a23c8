"""Dynamic tile order (tiles taken from an atomic counter and handed to every
role through a shared-memory ring of tile ids): the same results as the
static order bit for bit, parity with the oracle, and the ring protocol
(stages and accumulators) holds in the trace."""
import pytest
import torch

import oracle
from mbarrier_gemm_pipelines_gb300 import inputs, trace
from gpu_helpers import (TOL, load_library, rel_frobenius, require_gpu, split_tail, to_host_f64,
                         tuned)
from trace_check import check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbr():
    require_gpu()
    return load_library()


class dynamic:
    def __init__(self, gbr):
        self.gbr = gbr

    def __enter__(self):
        self.gbr.gemm_dynamic_schedule(True)

    def __exit__(self, *exc):
        self.gbr.gemm_dynamic_schedule(False)
        return False


@pytest.mark.parametrize("dtype,pair,ks,S", [("bf16", 2, 2, 3), ("bf16", 2, 1, 6), ("bf16", 1, 1, 4),
                                             ("tf32", 2, 2, 3), ("tf32", 1, 1, 2)])
@pytest.mark.parametrize("M,N,K", [(383, 776, 1352), (2304, 2304, 512), (4096, 4096, 256)])
def test_dynamic_equals_static(gbr, dtype, pair, ks, S, M, N, K):
    A, B, bias = inputs.gemm_normal(M, N, K, seed=M + K)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    with tuned(gbr, pair, ks), split_tail(gbr, 0):
        C0 = gbr.gemm_bias_relu(dA, dB, db, dtype=dtype, stages=S)
        with dynamic(gbr):
            C1 = gbr.gemm_bias_relu(dA, dB, db, dtype=dtype, stages=S)
    gbr.check_device()
    assert torch.equal(C0, C1)
    if M * N * K <= 2304 * 2304 * 512:
        ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
        assert rel_frobenius(to_host_f64(C1), ref) <= TOL[dtype]


@pytest.mark.parametrize("pair", [1, 2])
def test_dynamic_grouped_skewed(gbr, pair):
    counts = [1500, 3, 0, 700, 40, 900, 1, 952]        # skewed expert sizes
    cnt_, X, W, b = inputs.grouped(tokens=sum(counts), experts=8, K=512, N=1032, seed=41)
    dX, dW, db = X.cuda(), W.cuda(), b.cuda()
    with tuned(gbr, pair), split_tail(gbr, 0):
        C0 = gbr.gemm_bias_relu_grouped(dX, dW, db, counts, stages=3)
        with dynamic(gbr):
            C1 = gbr.gemm_bias_relu_grouped(dX, dW, db, counts, stages=3)
    gbr.check_device()
    assert torch.equal(C0, C1)
    ref = oracle.gemm_bias_relu_grouped(X.float(), W.float(), b, counts)
    assert rel_frobenius(to_host_f64(C1), ref) <= TOL["bf16"]


@pytest.mark.parametrize("pair", [1, 2])
def test_dynamic_trace(gbr, pair):
    A, B, bias = inputs.gemm_normal(4096, 4096, 512, seed=42)
    A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    with tuned(gbr, pair), dynamic(gbr), trace.Recorder(cap=512) as rec:
        C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype="bf16", stages=3)
        ev, cnt = rec.events()
    gbr.check_device()
    ref = oracle.gemm_bias_relu_points(A.float(), B.float(), bias, [0, 4095, 1234], [0, 4095, 777])
    got = C[[0, 4095, 1234], [0, 4095, 777]].double().cpu().numpy()
    assert rel_frobenius(got, ref) <= TOL["bf16"]
    errs = check(ev, cnt, 3, cta_group=pair, accumulator=True)
    assert errs == [], errs[:5]


def test_dynamic_mode_is_validated(gbr):
    from mbarrier_gemm_pipelines_gb300 import _binding as b
    assert b.lib().gbr_gemm_dynamic_schedule(2) == b.ERR_INVALID
    b.lib().gbr_gemm_dynamic_schedule(0)
