"""gemm_bias_relu_host: host buffers in, host buffer out, with the copies and
the GEMM overlapped chunk by chunk.  Checked against the oracle, and
bit-for-bit against the device-buffer call (with the split tail off, both
add every output's products in the same order)."""
import numpy as np
import pytest
import torch

import oracle
from mbarrier_gemm_pipelines_gb300 import inputs
from gpu_helpers import (TOL, load_library, rel_frobenius, require_gpu, split_tail,
                         to_host_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbr():
    require_gpu()
    return load_library()


def _host_inputs(M, N, K, dtype, seed, pin=True):
    A, B, bias = inputs.gemm_normal(M, N, K, seed=seed)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    if pin:
        A, B, bias = A.pin_memory(), B.pin_memory(), bias.pin_memory()
    return A, B, bias


@pytest.mark.parametrize("dtype", ["ffma", "tf32", "bf16"])
@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (300, 264, 200), (2600, 264, 200), (4100, 136, 72)])
def test_host_matches_oracle_and_device_path(gbr, dtype, M, N, K):
    A, B, bias = _host_inputs(M, N, K, dtype, seed=M + N + K)
    with split_tail(gbr, 0):
        C = gbr.gemm_bias_relu_host(A, B, bias, dtype=dtype, stages=3)
        D = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype=dtype, stages=3)
    gbr.check_device()
    assert torch.equal(C, D.cpu())
    ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    assert rel_frobenius(to_host_f64(C), ref) <= TOL[dtype]


def test_host_pageable_inputs(gbr):
    A, B, bias = _host_inputs(700, 256, 128, "bf16", seed=3, pin=False)
    C = torch.empty((700, 256), dtype=torch.bfloat16)
    gbr.gemm_bias_relu_host(A, B, bias, C, dtype="bf16", stages=3)
    gbr.check_device()
    ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    assert rel_frobenius(to_host_f64(C), ref) <= TOL["bf16"]


def test_host_eight_chunks(gbr):
    """8192 rows: eight 1024-row chunks in flight at once; every element."""
    M, N, K = 8192, 1024, 1024
    A, B, bias = _host_inputs(M, N, K, "bf16", seed=9)
    C = gbr.gemm_bias_relu_host(A, B, bias, dtype="bf16", stages=3)
    gbr.check_device()
    ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    got = to_host_f64(C)
    assert rel_frobenius(got, ref) <= TOL["bf16"]
    assert np.abs(got - ref).max() <= 20 * TOL["bf16"] * np.abs(ref).max()


def test_host_k_zero_and_empty(gbr):
    bias = torch.linspace(-2, 2, 264).pin_memory()
    A = torch.empty((300, 0), dtype=torch.bfloat16)
    B = torch.empty((0, 264), dtype=torch.bfloat16)
    C = gbr.gemm_bias_relu_host(A, B, bias, dtype="bf16", stages=2)
    gbr.check_device()
    expect = np.maximum(np.tile(bias.numpy(), (300, 1)), 0)
    expect = torch.from_numpy(expect).to(torch.bfloat16).double().numpy()
    assert np.array_equal(to_host_f64(C), expect)
    E = gbr.gemm_bias_relu_host(torch.empty((0, 8)), torch.empty((8, 8)), torch.zeros(8),
                                dtype="ffma", stages=2)
    assert E.shape == (0, 8)


def test_host_errors(gbr):
    from mbarrier_gemm_pipelines_gb300 import _binding as b
    lib = b.lib()
    h = torch.zeros(64 * 64).pin_memory()
    assert lib.gemm_bias_relu_host(None, None, None, None, 64, 64, 64, 0, 2, None) == b.ERR_INVALID
    assert lib.gemm_bias_relu_host(h.data_ptr(), h.data_ptr(), h.data_ptr(), h.data_ptr(),
                                   64, 64, 64, 0, 99, None) == b.ERR_SMEM
    assert lib.gemm_bias_relu_host(h.data_ptr(), h.data_ptr(), h.data_ptr(), h.data_ptr(),
                                   64, 62, 64, 0, 2, None) == b.ERR_ALIGN
    with pytest.raises(ValueError):
        gbr.gemm_bias_relu_host(h.cuda().view(64, 64), h.view(64, 64), torch.zeros(64), dtype="ffma")
    gbr.check_device()


def test_host_calls_from_two_threads(gbr):
    """Two host threads, each on its own stream, calling at once: the library's
    streams are shared, and each call's enqueue sequence is taken as a whole."""
    import threading
    jobs = []
    for t in range(2):
        A, B, bias = _host_inputs(1800, 520, 304, "bf16", seed=60 + t)
        jobs.append((A, B, bias, torch.empty((1800, 520), dtype=torch.bfloat16).pin_memory(),
                     torch.cuda.Stream()))
    errors = []

    def run(job):
        try:
            A, B, bias, C, st = job
            for _ in range(3):
                gbr.gemm_bias_relu_host(A, B, bias, C, dtype="bf16", stages=3, stream=st)
        except Exception as e:   # surfaced below
            errors.append(e)

    threads = [threading.Thread(target=run, args=(j,)) for j in jobs]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    gbr.check_device()
    for A, B, bias, C, _ in jobs:
        ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
        assert rel_frobenius(to_host_f64(C), ref) <= TOL["bf16"]


def test_host_steps_on_two_streams_pipeline(gbr):
    """Consecutive calls on two streams (as the benchmark issues them) each
    produce their own correct result."""
    A, B, bias = _host_inputs(2048, 512, 512, "bf16", seed=70)
    outs = [torch.empty((2048, 512), dtype=torch.bfloat16).pin_memory() for _ in range(4)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    with split_tail(gbr, 0):   # deterministic, so that the four results are comparable bit for bit
        for i, C in enumerate(outs):
            gbr.gemm_bias_relu_host(A, B, bias, C, dtype="bf16", stages=3, stream=streams[i % 2],
                                    sync=False)
        torch.cuda.synchronize()
    gbr.check_device()
    ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    for C in outs:
        assert rel_frobenius(to_host_f64(C), ref) <= TOL["bf16"]
        assert torch.equal(C, outs[0])
