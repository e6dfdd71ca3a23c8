"""Grouped (MoE-style) bf16 GEMM + bias + ReLU in one persistent launch against
the oracle applied expert by expert, element by element over the whole output
(the full-size MoE workload included).  Bar: relative Frobenius error 1e-2."""
import numpy as np
import pytest
import torch

import oracle
from mbarrier_gemm_pipelines_gb300 import inputs
from gpu_helpers import (TOL, load_library, rel_frobenius, require_gpu, split_tail, thin_tail,
                         to_host_f64, tuned)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbr():
    require_gpu()
    return load_library()


@pytest.mark.parametrize("counts,K,N", [
    ([130, 0, 7, 256, 1], 192, 520),      # ragged, an empty expert, a one-row expert
    ([64], 64, 256),
    ([300, 300, 300], 128, 264),
    ([0, 0, 129], 72, 512),
])
@pytest.mark.parametrize("pair", [1, 2])
def test_grouped_small(gbr, counts, K, N, pair):
    G = len(counts)
    cnt, X, W, b = inputs.grouped(tokens=sum(counts), experts=G, K=K, N=N, seed=sum(counts) + K)
    cnt = counts                                          # fixed counts for the edge cases
    with tuned(gbr, pair):
        C = gbr.gemm_bias_relu_grouped(X.cuda(), W.cuda(), b.cuda(), cnt, stages=3)
    gbr.check_device()
    ref = oracle.gemm_bias_relu_grouped(X.float(), W.float(), b, cnt)
    got = to_host_f64(C)
    assert rel_frobenius(got, ref) <= TOL["bf16"]
    assert np.abs(got - ref).max() <= 0.2 * np.abs(ref).max()


@pytest.mark.parametrize("pair", [1, 2])
def test_grouped_matches_dense_per_expert(gbr, pair):
    """Each expert's rows equal the dense kernel run on that expert alone (with
    the split tail and the transposed thin tails off, both add the same
    products in the same order)."""
    counts = [200, 77, 300]
    cnt, X, W, b = inputs.grouped(tokens=sum(counts), experts=3, K=256, N=512, seed=11)
    dX, dW, db = X.cuda(), W.cuda(), b.cuda()
    with tuned(gbr, pair), split_tail(gbr, 0), thin_tail(gbr, False):
        C = gbr.gemm_bias_relu_grouped(dX, dW, db, counts, stages=4)
        off = 0
        for e, n_e in enumerate(counts):
            Ce = gbr.gemm_bias_relu(dX[off:off + n_e].contiguous(), dW[e].contiguous(),
                                    db[e].contiguous(), dtype="bf16", stages=4)
            assert torch.equal(C[off:off + n_e], Ce)
            off += n_e
    gbr.check_device()


@pytest.mark.parametrize("pair", [1, 2])
def test_grouped_split_tail(gbr, pair):
    """The last round split along K (forced on), tiles of several experts among
    the split ones: parity with the oracle, and the unsplit result up to the
    order of fp32 additions.  (Thin tail tiles turn the split off, so they are
    off here.)"""
    counts = [300, 0, 513, 77, 1]
    cnt, X, W, b = inputs.grouped(tokens=sum(counts), experts=5, K=1024, N=1032, seed=21)
    dX, dW, db = X.cuda(), W.cuda(), b.cuda()
    with tuned(gbr, pair), thin_tail(gbr, False):
        with split_tail(gbr, 1):
            C = gbr.gemm_bias_relu_grouped(dX, dW, db, counts, stages=3)
        with split_tail(gbr, 0):
            C0 = gbr.gemm_bias_relu_grouped(dX, dW, db, counts, stages=3)
    gbr.check_device()
    ref = oracle.gemm_bias_relu_grouped(X.float(), W.float(), b, counts)
    got = to_host_f64(C)
    assert rel_frobenius(got, ref) <= TOL["bf16"]
    assert np.abs(got - ref).max() <= 0.2 * np.abs(ref).max()
    assert rel_frobenius(got, to_host_f64(C0)) <= TOL["bf16"] / 10


# Experts whose last 256-row tile holds 1, 16, 17, 100, 128 rows run it
# transposed (thin); 129 and 255 rows do not; one expert is empty.
THIN_COUNTS = [257, 272, 17, 100, 0, 128, 129, 511]


@pytest.mark.parametrize("K,N", [(200, 520), (1024, 264)])
def test_grouped_thin_tails(gbr, K, N):
    """Thin tail tiles (C^T = W^T X^T on the CTA pair) against the oracle,
    element by element, and against the same launch with every tile 256 rows
    (agreement to the order of fp32 additions); ragged K and N."""
    cnt, X, W, b = inputs.grouped(tokens=sum(THIN_COUNTS), experts=len(THIN_COUNTS), K=K, N=N,
                                  seed=K + N)
    dX, dW, db = X.cuda(), W.cuda(), b.cuda()
    with tuned(gbr, 2):
        C = gbr.gemm_bias_relu_grouped(dX, dW, db, THIN_COUNTS, stages=3)
        with thin_tail(gbr, False):
            C0 = gbr.gemm_bias_relu_grouped(dX, dW, db, THIN_COUNTS, stages=3)
    gbr.check_device()
    ref = oracle.gemm_bias_relu_grouped(X.float(), W.float(), b, THIN_COUNTS)
    got = to_host_f64(C)
    assert rel_frobenius(got, ref) <= TOL["bf16"]
    assert np.abs(got - ref).max() <= 0.2 * np.abs(ref).max()
    assert rel_frobenius(got, to_host_f64(C0)) <= TOL["bf16"] / 10
    # the rows of the thin tiles on their own (every expert's last rows)
    offs = oracle.group_offsets(THIN_COUNTS)
    for e, n_e in enumerate(THIN_COUNTS):
        t = n_e - 256 * ((n_e - 1) // 256) if n_e else 0
        if 0 < t <= 128:
            rows = slice(int(offs[e]) + n_e - t, int(offs[e]) + n_e)
            assert rel_frobenius(got[rows], ref[rows]) <= TOL["bf16"], (e, t)


def test_grouped_thin_tails_k_zero_and_switch(gbr):
    cnt, X, W, b = inputs.grouped(tokens=sum(THIN_COUNTS), experts=len(THIN_COUNTS), K=64, N=264,
                                  seed=5)
    X0 = torch.empty((sum(THIN_COUNTS), 0), dtype=torch.bfloat16, device="cuda")
    W0 = torch.empty((len(THIN_COUNTS), 0, 264), dtype=torch.bfloat16, device="cuda")
    with tuned(gbr, 2):
        C = gbr.gemm_bias_relu_grouped(X0, W0, b.cuda(), THIN_COUNTS, stages=3)
    gbr.check_device()
    ref = oracle.gemm_bias_relu_grouped(X0.cpu().float(), W0.cpu().float(), b, THIN_COUNTS)
    expect = torch.from_numpy(ref).float().to(torch.bfloat16)
    assert torch.equal(C.cpu(), expect)
    from mbarrier_gemm_pipelines_gb300 import _binding as bnd
    assert bnd.lib().gbr_gemm_thin_tail(2) == bnd.ERR_INVALID


def test_grouped_rejects(gbr):
    X = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((1, 64, 64), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((1, 64), device="cuda")
    with pytest.raises(ValueError):
        gbr.gemm_bias_relu_grouped(X, W, b, [9])     # counts must sum to the rows of X
    from mbarrier_gemm_pipelines_gb300 import _binding as bnd
    import ctypes
    cnt = (ctypes.c_int32 * 1)(8)
    C = torch.zeros((8, 64), device="cuda")
    assert bnd.lib().gemm_bias_relu_grouped(X.data_ptr(), W.data_ptr(), b.data_ptr(), C.data_ptr(),
                                            ctypes.cast(cnt, ctypes.c_void_p), 1, 64, 64,
                                            bnd.F32_FFMA, 2, None) == bnd.ERR_UNSUPPORTED
    assert bnd.lib().gemm_bias_relu_grouped(X.data_ptr(), W.data_ptr(), b.data_ptr(), C.data_ptr(),
                                            ctypes.cast(cnt, ctypes.c_void_p), 33, 64, 64,
                                            bnd.BF16, 2, None) == bnd.ERR_INVALID


@pytest.fixture(scope="module")
def moe():
    """The MoE workload (4096 tokens over 8 experts, Multinomial counts, seed
    4, K = 4096, N = 14336) and its oracle output, with the biases and with
    zero biases (the GEMM part alone), computed once for the module."""
    counts, X, W, b = inputs.workload("grouped_bf16")
    Xf, Wf = X.float(), W.float()
    ref = oracle.gemm_bias_relu_grouped(Xf, Wf, b, counts)
    ref0 = oracle.gemm_bias_relu_grouped(Xf, Wf, torch.zeros_like(b), counts)
    return counts, X, W, b, ref, ref0


def _check_moe(got, ref):
    assert rel_frobenius(got, ref) <= TOL["bf16"]
    assert (got >= 0).all()
    assert np.abs(got - ref).max() <= 20 * TOL["bf16"] * np.abs(ref).max()


@pytest.mark.parametrize("pair,S,ks", [(-1, 4, -1), (1, 4, -1), (2, 6, -1), (1, 2, 2), (2, 3, 2),
                                        (-1, 3, -1)])
def test_config5_moe(gbr, moe, pair, S, ks):
    """One launch over all experts' tiles; every output element of every
    expert against the oracle, with the biases and without them."""
    counts, X, W, b, ref, ref0 = moe
    dX, dW, db = X.cuda(), W.cuda(), b.cuda()
    with tuned(gbr, pair, ks):
        C = gbr.gemm_bias_relu_grouped(dX, dW, db, counts, stages=S)
        C0 = gbr.gemm_bias_relu_grouped(dX, dW, torch.zeros_like(db), counts, stages=S)
    gbr.check_device()
    _check_moe(to_host_f64(C), ref)
    _check_moe(to_host_f64(C0), ref0)
