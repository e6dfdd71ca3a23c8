"""CPU oracle for the warp-specialized pipeline operators.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product package never
imports this module and this module never imports the product package; the
two share only the seeded input generators, which hold none of the method's
arithmetic.

Contents
--------
``gemm_bias_relu``          C = max(0, A @ B + bias) in binary64 (plain i-k-j
                            loop in ``oracle.c``).  Follows the SGEMM test
                            bench of "pwwt.cn news/4436243", section 4.1.
``gemm_bias_relu_points``   the same definition at chosen (m, n) positions.
``gemm_bias_relu_grouped``  the same definition applied per expert segment
                            (the MoE operator that motivates the same page,
                            section 1.1): rows [off_e, off_e + n_e) of X times
                            W[e] plus b[e].
``copy``                    the staged copy's result: memcpy ("Producer-
                            Consumer Warp Specialization for TMA Operations",
                            double-buffered load/store example).
``ring_sim``                a simulator of the mbarrier full/empty ring.

Pins (tests/test_oracle_*.py): exact rational brute force, identity, zero,
diagonal, K = 0, the ReLU invariant, a NumPy binary64 matmul cross-check, and
for the simulator the printed S = 2 schedule plus protocol invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc (OpenMP if present)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.oracle_gemm_bias_relu.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32]
        lib.oracle_gemm_bias_relu.restype = None
        lib.oracle_gemm_bias_relu_points.argtypes = [
            vp, vp, vp, i64, i64, i64, vp, vp, i64, vp, i32]
        lib.oracle_gemm_bias_relu_points.restype = None
        lib.oracle_copy.argtypes = [vp, vp, ctypes.c_size_t]
        lib.oracle_copy.restype = None
        lib.oracle_copy_parallel.argtypes = [vp, vp, ctypes.c_size_t, i32]
        lib.oracle_copy_parallel.restype = None
        lib.oracle_max_threads.restype = i32
        lib.oracle_has_openmp.restype = i32
        _lib = lib
        return lib


def _as_f32(x) -> np.ndarray:
    """Exact widening to a contiguous fp32 NumPy array (bf16 -> fp32 is exact)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu")
            if x.dtype != torch.float32:
                x = x.to(torch.float32)
            x = x.contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError("oracle inputs must already be exactly representable "
                        "in fp32 (got %s)" % x.dtype)
    return x


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def has_openmp() -> bool:
    return bool(_load().oracle_has_openmp())


def gemm_bias_relu(A, B, bias, nthreads: int = 0) -> np.ndarray:
    """C[m,n] = max(0, bias[n] + sum_k A[m,k] B[k,n]) in binary64."""
    A, B, bias = _as_f32(A), _as_f32(B), _as_f32(bias)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or bias.shape != (N,):
        raise ValueError("shape mismatch")
    C = np.empty((M, N), dtype=np.float64)
    _load().oracle_gemm_bias_relu(A.ctypes.data, B.ctypes.data, bias.ctypes.data,
                                  C.ctypes.data, M, N, K, nthreads)
    return C


def gemm_bias_relu_points(A, B, bias, m_idx, n_idx, nthreads: int = 0) -> np.ndarray:
    """The same definition evaluated only at positions (m_idx[p], n_idx[p])."""
    A, B, bias = _as_f32(A), _as_f32(B), _as_f32(bias)
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or bias.shape != (N,):
        raise ValueError("shape mismatch")
    mi = np.ascontiguousarray(np.asarray(m_idx, dtype=np.int64))
    ni = np.ascontiguousarray(np.asarray(n_idx, dtype=np.int64))
    if mi.shape != ni.shape or mi.ndim != 1:
        raise ValueError("index arrays must be 1-D and equal length")
    if mi.size and (mi.min() < 0 or mi.max() >= M or ni.min() < 0 or ni.max() >= N):
        raise IndexError("position out of range")
    out = np.empty(mi.shape, dtype=np.float64)
    _load().oracle_gemm_bias_relu_points(A.ctypes.data, B.ctypes.data, bias.ctypes.data,
                                         M, N, K, mi.ctypes.data, ni.ctypes.data,
                                         mi.size, out.ctypes.data, nthreads)
    return out


def group_offsets(counts) -> np.ndarray:
    """Row offset of each expert segment when rows are stored expert by expert."""
    c = np.asarray(counts, dtype=np.int64)
    return np.concatenate([[0], np.cumsum(c)[:-1]]).astype(np.int64)


def gemm_bias_relu_grouped(X, W, b, counts, nthreads: int = 0) -> np.ndarray:
    """Per expert e: C[rows of e] = max(0, X[rows of e] @ W[e] + b[e])."""
    X, W, b = _as_f32(X), _as_f32(W), _as_f32(b)
    G, K, N = W.shape
    counts = np.asarray(counts, dtype=np.int64)
    if counts.shape != (G,) or b.shape != (G, N) or X.shape[1] != K:
        raise ValueError("shape mismatch")
    if counts.sum() != X.shape[0]:
        raise ValueError("counts must sum to the number of rows of X")
    C = np.empty((X.shape[0], N), dtype=np.float64)
    for e, off in enumerate(group_offsets(counts)):
        n_e = int(counts[e])
        if n_e:
            C[off:off + n_e] = gemm_bias_relu(X[off:off + n_e], W[e], b[e], nthreads)
    return C


def gemm_bias_relu_grouped_points(X, W, b, counts, rows, cols, nthreads: int = 0) -> np.ndarray:
    """The grouped definition at global output positions (rows[p], cols[p])."""
    X, W, b = _as_f32(X), _as_f32(W), _as_f32(b)
    counts = np.asarray(counts, dtype=np.int64)
    offs = group_offsets(counts)
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    expert = np.searchsorted(offs + counts, rows, side="right")
    out = np.empty(rows.shape, dtype=np.float64)
    for e in np.unique(expert):
        sel = np.nonzero(expert == e)[0]
        out[sel] = gemm_bias_relu_points(X, W[e], b[e], rows[sel], cols[sel], nthreads)
    return out


def copy(src: np.ndarray) -> np.ndarray:
    """The staged copy's expected output: the same bytes."""
    src = np.ascontiguousarray(src)
    dst = np.empty_like(src)
    _load().oracle_copy(src.ctypes.data, dst.ctypes.data, src.nbytes)
    return dst


def copy_into(src: np.ndarray, dst: np.ndarray, nthreads: int = 1) -> None:
    """memcpy of src into dst, cut into nthreads pieces (timing helper)."""
    if src.nbytes != dst.nbytes:
        raise ValueError("size mismatch")
    if nthreads <= 1:
        _load().oracle_copy(src.ctypes.data, dst.ctypes.data, src.nbytes)
    else:
        _load().oracle_copy_parallel(src.ctypes.data, dst.ctypes.data, src.nbytes, nthreads)


def rel_frobenius(got, ref) -> float:
    """||got - ref||_F / ||ref||_F in binary64 (absolute norm if ||ref|| = 0)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = float(np.linalg.norm((got - ref).ravel()))
    den = float(np.linalg.norm(ref.ravel()))
    return num / den if den > 0 else num
