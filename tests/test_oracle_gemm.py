"""Pins for the CPU GEMM+bias+ReLU oracle, independent of the oracle itself.

The operator is the SGEMM test bench of "pwwt.cn news/4436243", section 4.1:
C = ReLU(A[M,K] * B[K,N] + bias).  Each test checks the oracle against
something the mathematics fixes: exact rational arithmetic, closed forms
(identity, zero, diagonal, K = 0), an invariant of ReLU, and a library matmul.
"""
from fractions import Fraction

import numpy as np
import pytest

EPS64 = 2.0 ** -53


def _rand(rng, *shape, lo=-1.0, hi=1.0):
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def _exact(A, B, bias):
    M, K = A.shape
    N = B.shape[1]
    out = np.empty((M, N), dtype=object)
    mag = np.empty((M, N), dtype=np.float64)
    for m in range(M):
        for n in range(N):
            s = Fraction(float(bias[n]))
            a = abs(float(bias[n]))
            for k in range(K):
                t = Fraction(float(A[m, k])) * Fraction(float(B[k, n]))
                s += t
                a += abs(float(A[m, k]) * float(B[k, n]))
            out[m, n] = s if s > 0 else Fraction(0)
            mag[m, n] = a
    return out, mag


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 1, 0), (3, 5, 7, 1), (8, 2, 8, 2),
                                        (2, 8, 3, 3), (5, 7, 1, 4), (7, 3, 8, 5)])
def test_exact_rational_bruteforce(oracle_mod, M, N, K, seed):
    """Within the forward error bound of a K-term binary64 sum of the exact value."""
    rng = np.random.default_rng(seed)
    A, B, bias = _rand(rng, M, K), _rand(rng, K, N), _rand(rng, N)
    C = oracle_mod.gemm_bias_relu(A, B, bias)
    exact, mag = _exact(A, B, bias)
    for m in range(M):
        for n in range(N):
            bound = (K + 2) * EPS64 * mag[m, n]
            assert abs(Fraction(C[m, n]) - exact[m, n]) <= Fraction(bound), (m, n)


def test_small_integers_are_exact(oracle_mod):
    """Integer inputs: every partial sum is exact in binary64, so C is exact."""
    rng = np.random.default_rng(7)
    A = rng.integers(-9, 10, size=(6, 11)).astype(np.float32)
    B = rng.integers(-9, 10, size=(11, 4)).astype(np.float32)
    bias = rng.integers(-20, 21, size=(4,)).astype(np.float32)
    C = oracle_mod.gemm_bias_relu(A, B, bias)
    exact, _ = _exact(A, B, bias)
    assert all(Fraction(C[m, n]) == exact[m, n] for m in range(6) for n in range(4))


def test_identity(oracle_mod):
    rng = np.random.default_rng(11)
    K, N = 37, 29
    B, bias = _rand(rng, K, N), _rand(rng, N)
    C = oracle_mod.gemm_bias_relu(np.eye(K, dtype=np.float32), B, bias)
    expect = np.maximum(B.astype(np.float64) + bias.astype(np.float64), 0.0)
    assert np.array_equal(C, expect)


def test_zero_matrix(oracle_mod):
    rng = np.random.default_rng(12)
    B, bias = _rand(rng, 19, 23), _rand(rng, 23)
    C = oracle_mod.gemm_bias_relu(np.zeros((13, 19), np.float32), B, bias)
    assert np.array_equal(C, np.broadcast_to(np.maximum(bias.astype(np.float64), 0), C.shape))


def test_diagonal(oracle_mod):
    rng = np.random.default_rng(13)
    K, N = 17, 31
    d = _rand(rng, K)
    B, bias = _rand(rng, K, N), _rand(rng, N)
    C = oracle_mod.gemm_bias_relu(np.diag(d).astype(np.float32), B, bias)
    expect = np.maximum(d.astype(np.float64)[:, None] * B.astype(np.float64)
                        + bias.astype(np.float64)[None, :], 0.0)
    assert np.array_equal(C, expect)


def test_k_zero_is_relu_of_bias(oracle_mod):
    bias = np.array([-2.0, -0.0, 0.0, 0.5, 3.0], np.float32)
    C = oracle_mod.gemm_bias_relu(np.zeros((4, 0), np.float32), np.zeros((0, 5), np.float32), bias)
    assert np.array_equal(C, np.tile([0.0, 0.0, 0.0, 0.5, 3.0], (4, 1)))


def test_relu_invariant_and_numpy_cross_check(oracle_mod):
    """C >= 0; C equals the binary64 library product where it is positive."""
    rng = np.random.default_rng(14)
    M, N, K = 96, 80, 256
    A, B, bias = _rand(rng, M, K), _rand(rng, K, N), _rand(rng, N)
    C = oracle_mod.gemm_bias_relu(A, B, bias)
    pre = A.astype(np.float64) @ B.astype(np.float64) + bias.astype(np.float64)
    assert (C >= 0).all()
    tol = 1e-12 * np.abs(A).astype(np.float64) @ np.abs(B).astype(np.float64) + 1e-15
    pos = pre > tol
    neg = pre < -tol
    assert np.all(np.abs(C[pos] - pre[pos]) <= tol[pos])
    assert np.all(C[neg] == 0)
    assert pos.sum() > 0 and neg.sum() > 0


@pytest.mark.parametrize("n", [256, 512])
def test_library_matmul_rel_frobenius(oracle_mod, n):
    rng = np.random.default_rng(n)
    A, B, bias = _rand(rng, n, n), _rand(rng, n, n), _rand(rng, n)
    C = oracle_mod.gemm_bias_relu(A, B, bias)
    ref = np.maximum(A.astype(np.float64) @ B.astype(np.float64) + bias.astype(np.float64), 0)
    assert oracle_mod.rel_frobenius(C, ref) <= 1e-12


def test_thread_count_does_not_change_result(oracle_mod):
    rng = np.random.default_rng(15)
    A, B, bias = _rand(rng, 33, 70), _rand(rng, 70, 45), _rand(rng, 45)
    assert np.array_equal(oracle_mod.gemm_bias_relu(A, B, bias, nthreads=1),
                          oracle_mod.gemm_bias_relu(A, B, bias, nthreads=4))


def test_points_match_full_and_bruteforce(oracle_mod):
    rng = np.random.default_rng(16)
    M, N, K = 9, 6, 8
    A, B, bias = _rand(rng, M, K), _rand(rng, K, N), _rand(rng, N)
    mi = rng.integers(0, M, 20)
    ni = rng.integers(0, N, 20)
    P = oracle_mod.gemm_bias_relu_points(A, B, bias, mi, ni)
    full = oracle_mod.gemm_bias_relu(A, B, bias)
    assert np.array_equal(P, full[mi, ni])
    exact, mag = _exact(A, B, bias)
    for p in range(20):
        bound = (K + 2) * EPS64 * mag[mi[p], ni[p]]
        assert abs(Fraction(P[p]) - exact[mi[p], ni[p]]) <= Fraction(bound)


def test_points_reject_out_of_range(oracle_mod):
    A = np.zeros((2, 3), np.float32)
    with pytest.raises(IndexError):
        oracle_mod.gemm_bias_relu_points(A, np.zeros((3, 4), np.float32),
                                         np.zeros(4, np.float32), [2], [0])


def _block_embedding(X, W, b, counts):
    """Dense A', B' whose plain product (bias 0) is the grouped result."""
    G, K, N = W.shape
    T = X.shape[0]
    A = np.zeros((T, G * K + G), np.float32)
    Bd = np.zeros((G * K + G, N), np.float32)
    off = 0
    for e in range(G):
        n_e = int(counts[e])
        A[off:off + n_e, e * K:(e + 1) * K] = X[off:off + n_e]
        A[off:off + n_e, G * K + e] = 1.0
        Bd[e * K:(e + 1) * K] = W[e]
        Bd[G * K + e] = b[e]
        off += n_e
    return A, Bd


def test_grouped_equals_block_embedding(oracle_mod):
    """Grouped result equals a dense product on the block-diagonal embedding.

    The embedding adds only exact zeros and a bias row multiplied by exactly 1,
    so the two agree within the binary64 sum error bound."""
    rng = np.random.default_rng(17)
    G, K, N = 4, 24, 40
    counts = np.array([5, 0, 9, 3])
    X, W, b = _rand(rng, counts.sum(), K), _rand(rng, G, K, N), _rand(rng, G, N)
    C = oracle_mod.gemm_bias_relu_grouped(X, W, b, counts)
    A, Bd = _block_embedding(X, W, b, counts)
    ref = oracle_mod.gemm_bias_relu(A, Bd, np.zeros(N, np.float32))
    assert np.allclose(C, ref, rtol=0, atol=1e-13)
    pts_r = rng.integers(0, counts.sum(), 30)
    pts_c = rng.integers(0, N, 30)
    assert np.array_equal(oracle_mod.gemm_bias_relu_grouped_points(X, W, b, counts, pts_r, pts_c),
                          C[pts_r, pts_c])


def test_grouped_tiny_exact(oracle_mod):
    rng = np.random.default_rng(18)
    G, K, N = 3, 4, 3
    counts = np.array([2, 1, 2])
    X, W, b = _rand(rng, 5, K), _rand(rng, G, K, N), _rand(rng, G, N)
    C = oracle_mod.gemm_bias_relu_grouped(X, W, b, counts)
    off = 0
    for e in range(G):
        ex, mag = _exact(X[off:off + counts[e]], W[e], b[e])
        for i in range(counts[e]):
            for n in range(N):
                assert abs(Fraction(C[off + i, n]) - ex[i, n]) <= Fraction((K + 2) * EPS64 * mag[i, n])
        off += counts[e]


def test_copy_is_bitwise(oracle_mod):
    rng = np.random.default_rng(19)
    src = rng.uniform(-1e3, 1e3, size=(33, 17)).astype(np.float32)
    src.view(np.uint32)[0, 0] = 0x7FC00001    # a NaN payload must survive
    src.view(np.uint32)[0, 1] = 0x80000000    # and so must -0.0
    dst = oracle_mod.copy(src)
    assert np.array_equal(dst.view(np.uint32), src.view(np.uint32))
    out = np.empty_like(src)
    oracle_mod.copy_into(src, out, nthreads=3)
    assert np.array_equal(out.view(np.uint32), src.view(np.uint32))


def test_rel_frobenius_definition(oracle_mod):
    assert oracle_mod.rel_frobenius([3.0, 4.0], [3.0, 4.0]) == 0.0
    assert oracle_mod.rel_frobenius([3.0, 4.0], [0.0, 0.0]) == 5.0
    assert abs(oracle_mod.rel_frobenius([0.0, 4.0], [3.0, 4.0]) - 3.0 / 5.0) < 1e-15
