"""ctypes binding of ``libgbr.so`` (declared in ``include/gbr.h``).

Argument marshalling only: every step of every operator runs in the CUDA
kernels of the library.  There is no CPU or PyTorch fallback; if the library
is missing or the tensors are not on a CUDA device the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build

# gbr_dtype
F32_FFMA, F32_TF32, BF16, F32_FFMA_SYNC, F32_FFMA_CPASYNC = 0, 1, 2, 3, 4
DTYPE_NAMES = {"ffma": F32_FFMA, "tf32": F32_TF32, "bf16": BF16, "ffma_sync": F32_FFMA_SYNC,
               "ffma_cpasync": F32_FFMA_CPASYNC}
# gbr_status
OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_ALIGN, ERR_SMEM, ERR_CUDA, ERR_TIMEOUT = range(7)
STATUS_NAMES = {0: "GBR_OK", 1: "GBR_ERR_INVALID", 2: "GBR_ERR_UNSUPPORTED", 3: "GBR_ERR_ALIGN",
                4: "GBR_ERR_SMEM", 5: "GBR_ERR_CUDA", 6: "GBR_ERR_TIMEOUT"}
OP_GEMM, OP_COPY = 0, 1

# Every function the header declares: name -> (restype, argtypes).
_vp, _i64, _i32, _u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64
SIGNATURES = {
    "gemm_bias_relu": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _vp]),
    "gemm_bias_relu_grouped": (_i32, [_vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32, _i32, _vp]),
    "gemm_bias_relu_host": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _vp]),
    "staged_copy": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp]),
    "gbr_device_status": (_i32, [_vp]),
    "gbr_last_error": (ctypes.c_char_p, []),
    "gbr_max_stages": (_i32, [_i32, _i32, _i32, _i32]),
    "gbr_launch_count": (ctypes.c_longlong, []),
    "gbr_sm_count": (_i32, []),
    "gbr_set_wait_timeout_ns": (_i32, [_u64]),
    "gbr_copy_tuning": (_i32, [_i32, _i32, _i32]),
    "gbr_gemm_tuning": (_i32, [_i32, _i32, _i32, _i32]),
    "gbr_gemm_split_tail": (_i32, [_i32]),
    "gbr_gemm_dynamic_schedule": (_i32, [_i32]),
    "gbr_launch_overlap": (_i32, [_i32]),
    "gbr_gemm_thin_tail": (_i32, [_i32]),
    "gbr_ffma_tuning": (_i32, [_i32]),
    "gbr_trace_buffer": (_i32, [_vp, _u64]),
    "gbr_selftest_wait_timeout": (_i32, [_u64, _vp]),
    "gbr_selftest_gemm_skip_load": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32, _i32,
                                           _i32, _u64, _vp]),
    "gbr_selftest_copy_skip_load": (_i32, [_vp, _vp, _i64, _i64, _i32, _i32, _i32, _u64, _vp]),
    "gemm_bias_relu_tf32_noalloc": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp]),
    "gbr_selftest_noalloc_skip_load": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _i32,
                                              _i32, _u64, _vp]),
}

_lib = None
_lock = threading.Lock()


class GbrError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__("%s: %s" % (STATUS_NAMES.get(code, str(code)), msg))
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """Loads libgbr.so (it must have been built: ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError("libgbr.so is not built (%s); run __graft_entry__.build()" % path)
            h = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(h, name)
                fn.restype = res
                fn.argtypes = args
            _lib = h
        return _lib


def last_error() -> str:
    return (lib().gbr_last_error() or b"").decode()


def check(code: int) -> None:
    if code != OK:
        raise GbrError(code, last_error())


def _stream_ptr(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _cuda_tensor(t, name, dtypes):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (this library has no CPU path)" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if t.dtype not in dtypes:
        raise TypeError("%s has dtype %s, expected one of %s" % (name, t.dtype, dtypes))
    return t


def gemm_bias_relu(A, B, bias, C=None, dtype="bf16", stages=4, stream=None):
    """C = ReLU(A @ B + bias) on the GPU; returns C."""
    import torch
    dt = DTYPE_NAMES[dtype] if isinstance(dtype, str) else int(dtype)
    in_t = torch.bfloat16 if dt == BF16 else torch.float32
    _cuda_tensor(A, "A", (in_t,))
    _cuda_tensor(B, "B", (in_t,))
    _cuda_tensor(bias, "bias", (torch.float32,))
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(bias.shape) != (N,):
        raise ValueError("shape mismatch: A %s, B %s, bias %s" % (tuple(A.shape), tuple(B.shape),
                                                                  tuple(bias.shape)))
    if C is None:
        C = torch.empty((M, N), dtype=in_t, device=A.device)
    _cuda_tensor(C, "C", (in_t,))
    if tuple(C.shape) != (M, N):
        raise ValueError("C must be [M, N]")
    check(lib().gemm_bias_relu(A.data_ptr(), B.data_ptr(), bias.data_ptr(), C.data_ptr(),
                               M, N, K, dt, int(stages), _stream_ptr(stream)))
    return C


def gemm_bias_relu_host(A, B, bias, C=None, dtype="bf16", stages=4, stream=None, sync=True):
    """C = ReLU(A @ B + bias) for CPU tensors (page-locked for full copy speed):
    the library copies in, computes and copies out, overlapped, on the current
    CUDA device.  With sync=False the caller must synchronise `stream` before
    reading C or changing the inputs."""
    import torch
    dt = DTYPE_NAMES[dtype] if isinstance(dtype, str) else int(dtype)
    in_t = torch.bfloat16 if dt == BF16 else torch.float32
    for t, n, want in ((A, "A", in_t), (B, "B", in_t), (bias, "bias", torch.float32)):
        if not isinstance(t, torch.Tensor) or t.is_cuda:
            raise ValueError("%s must be a CPU tensor (host buffer)" % n)
        if not t.is_contiguous() or t.dtype != want:
            raise TypeError("%s must be contiguous %s" % (n, want))
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(bias.shape) != (N,):
        raise ValueError("shape mismatch")
    if C is None:
        C = torch.empty((M, N), dtype=in_t).pin_memory()
    if C.is_cuda or tuple(C.shape) != (M, N) or C.dtype != in_t or not C.is_contiguous():
        raise ValueError("C must be a contiguous CPU [M, N] tensor of the input type")
    s = _stream_ptr(stream)
    check(lib().gemm_bias_relu_host(A.data_ptr(), B.data_ptr(), bias.data_ptr(), C.data_ptr(),
                                    M, N, K, dt, int(stages), s))
    if sync:
        import torch as _t
        (stream or _t.cuda.current_stream()).synchronize()
    return C


def gemm_bias_relu_grouped(X, W, bias, counts, C=None, stages=4, stream=None):
    """Per expert e: C[rows of e] = ReLU(X[rows of e] @ W[e] + bias[e]); returns C."""
    import torch
    _cuda_tensor(X, "X", (torch.bfloat16,))
    _cuda_tensor(W, "W", (torch.bfloat16,))
    _cuda_tensor(bias, "bias", (torch.float32,))
    G, K, N = W.shape
    counts = [int(c) for c in counts]
    if len(counts) != G or X.shape[1] != K or tuple(bias.shape) != (G, N):
        raise ValueError("shape mismatch")
    T = sum(counts)
    if X.shape[0] != T:
        raise ValueError("X must have sum(counts) rows")
    if C is None:
        C = torch.empty((T, N), dtype=torch.bfloat16, device=X.device)
    _cuda_tensor(C, "C", (torch.bfloat16,))
    arr = (ctypes.c_int32 * G)(*counts)
    check(lib().gemm_bias_relu_grouped(X.data_ptr(), W.data_ptr(), bias.data_ptr(), C.data_ptr(),
                                       ctypes.cast(arr, ctypes.c_void_p), G, K, N, BF16, int(stages),
                                       _stream_ptr(stream)))
    return C


def staged_copy(src, dst=None, tile=(128, 64), stages=4, stream=None):
    """dst = src through the TMA staging ring (4-byte elements); returns dst."""
    import torch
    ok = (torch.float32, torch.int32)
    _cuda_tensor(src, "src", ok)
    if src.dim() != 2:
        raise ValueError("src must be 2-D")
    if dst is None:
        dst = torch.empty_like(src)
    _cuda_tensor(dst, "dst", ok)
    if dst.shape != src.shape:
        raise ValueError("dst must match src")
    rows, cols = src.shape
    check(lib().staged_copy(src.data_ptr(), dst.data_ptr(), rows, cols, int(tile[0]), int(tile[1]),
                            int(stages), _stream_ptr(stream)))
    return dst


def device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status code."""
    return int(lib().gbr_device_status(_stream_ptr(stream)))


def check_device(stream=None) -> None:
    check(device_status(stream))


def max_stages(op, dtype=0, tile_rows=0, tile_cols=0) -> int:
    r = int(lib().gbr_max_stages(op, dtype, tile_rows, tile_cols))
    if r < 0:
        raise GbrError(-r, last_error())
    return r


def launch_count() -> int:
    return int(lib().gbr_launch_count())


def sm_count() -> int:
    r = int(lib().gbr_sm_count())
    if r < 0:
        raise GbrError(-r, last_error())
    return r


def set_wait_timeout_ns(ns: int) -> None:
    check(lib().gbr_set_wait_timeout_ns(int(ns)))


def copy_tuning(store_lag: int = -1, ctas_per_sm: int = -1, l2_hint: int = -1) -> None:
    """Staged-copy knobs (see gbr.h): slot-release lag, CTAs per SM, L2 hint."""
    check(lib().gbr_copy_tuning(int(store_lag), int(ctas_per_sm), int(l2_hint)))


def gemm_tuning(cta_pair: int = -1, group_m: int = -1, l2_hint: int = -1,
                k_per_stage: int = -1) -> None:
    """Tensor-core GEMM variant: cta_pair -1 auto, 1 one CTA per tile, 2 CTA pair;
    group_m raster band height in tiles; l2_hint operand-load L2 policy;
    k_per_stage 128-byte K slices per ring stage (see gbr.h)."""
    check(lib().gbr_gemm_tuning(int(cta_pair), int(group_m), int(l2_hint), int(k_per_stage)))


def gemm_split_tail(mode: int = -1) -> None:
    """Split the last round of tensor-core GEMM tiles along K: -1 auto, 0 never,
    1 whenever possible (see gbr.h)."""
    check(lib().gbr_gemm_split_tail(int(mode)))


def gemm_dynamic_schedule(on: bool) -> None:
    """Tensor-core GEMM tiles from an atomic counter (True) or the static order (see gbr.h)."""
    check(lib().gbr_gemm_dynamic_schedule(int(bool(on))))


def ffma_tuning(consumer_warps: int = -1) -> None:
    """FFMA GEMM consumer layout: 8 warps of 8x8 (-1, default) or 16 warps of 8x4 (see gbr.h)."""
    check(lib().gbr_ffma_tuning(int(consumer_warps)))


def gemm_thin_tail(on: bool) -> None:
    """Grouped CTA-pair launches: run experts' last M-tiles of <= 128 rows
    transposed (True, default) or as 256-row tiles (False) (see gbr.h)."""
    check(lib().gbr_gemm_thin_tail(int(bool(on))))


def launch_overlap(on: bool) -> None:
    """Programmatic dependent launch of the library's kernels (True, default)
    or ordinary launches (False) (see gbr.h)."""
    check(lib().gbr_launch_overlap(int(bool(on))))


def selftest_wait_timeout(timeout_ns: int, stream=None) -> None:
    check(lib().gbr_selftest_wait_timeout(int(timeout_ns), _stream_ptr(stream)))


def selftest_gemm_skip_load(A, B, bias, dtype, stages, cta, item, limit_ns, stream=None):
    """Runs gemm_bias_relu with one stage of CTA `cta`, ring item `item`, left
    unfilled (see gbr.h); returns the (undefined) output tensor."""
    import torch
    code = DTYPE_NAMES[dtype] if isinstance(dtype, str) else int(dtype)
    want = (torch.bfloat16,) if code == BF16 else (torch.float32,)
    _cuda_tensor(A, "A", want)
    _cuda_tensor(B, "B", want)
    _cuda_tensor(bias, "bias", (torch.float32,))
    M, K = A.shape
    N = B.shape[1]
    C = torch.empty((M, N), dtype=A.dtype, device=A.device)
    check(lib().gbr_selftest_gemm_skip_load(A.data_ptr(), B.data_ptr(), bias.data_ptr(),
                                            C.data_ptr(), M, N, K, code, int(stages), int(cta),
                                            int(item), int(limit_ns), _stream_ptr(stream)))
    return C


def selftest_copy_skip_load(src, stages, cta, item, limit_ns, stream=None):
    """Runs staged_copy (128 x 64 tiles) with one stage of CTA `cta`, ring item
    `item`, left unfilled (see gbr.h); returns the (undefined) output tensor."""
    import torch
    _cuda_tensor(src, "src", (torch.float32,))
    dst = torch.empty_like(src)
    rows, cols = src.shape
    check(lib().gbr_selftest_copy_skip_load(src.data_ptr(), dst.data_ptr(), rows, cols,
                                            int(stages), int(cta), int(item), int(limit_ns),
                                            _stream_ptr(stream)))
    return dst


def _noalloc_shapes(A, B, bias, C):
    """The dimension checks of gemm_bias_relu, for the no-alloc entry points
    (which take C from the caller): nothing is launched when they fail."""
    import torch
    for t, n in ((A, "A"), (B, "B"), (bias, "bias"), (C, "C")):
        _cuda_tensor(t, n, (torch.float32,))
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K or tuple(bias.shape) != (N,):
        raise ValueError("shape mismatch: A %s, B %s, bias %s" % (tuple(A.shape), tuple(B.shape),
                                                                  tuple(bias.shape)))
    if tuple(C.shape) != (M, N):
        raise ValueError("C must be [M, N] = [%d, %d], got %s" % (M, N, tuple(C.shape)))
    return M, N, K


def gemm_bias_relu_tf32_noalloc(A, B, bias, C, stages=4, stream=None):
    """TF32 C = ReLU(A @ B + bias) that allocates no device memory (C is required).

    For callers that may not allocate: serving loops that must stay out of
    allocators, plug-ins whose host framework owns all device allocation,
    processes whose device memory is reserved by another allocator.  Its
    status words live in a fixed device array that every call on the device
    shares; calls that overlap on the GPU race, so serialise them.  One CTA
    per tile, never split: stages 1..4."""
    M, N, K = _noalloc_shapes(A, B, bias, C)
    check(lib().gemm_bias_relu_tf32_noalloc(A.data_ptr(), B.data_ptr(), bias.data_ptr(),
                                            C.data_ptr(), M, N, K, int(stages),
                                            _stream_ptr(stream)))
    return C


def selftest_noalloc_skip_load(A, B, bias, C, stages, cta, item, limit_ns, stream=None):
    """Runs gemm_bias_relu_tf32_noalloc with one stage of CTA `cta`, ring item
    `item`, left unfilled (see gbr.h); C's contents are then undefined."""
    M, N, K = _noalloc_shapes(A, B, bias, C)
    check(lib().gbr_selftest_noalloc_skip_load(A.data_ptr(), B.data_ptr(), bias.data_ptr(),
                                               C.data_ptr(), M, N, K, int(stages), int(cta),
                                               int(item), int(limit_ns), _stream_ptr(stream)))
    return C
