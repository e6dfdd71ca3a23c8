"""The calls are stream-ordered and capture into CUDA graphs: each operator is
captured once after a warm-up call and replayed; replays give the eager
results (bit for bit where the result is deterministic)."""
import pytest
import torch

import oracle
from mbarrier_gemm_pipelines_gb300 import inputs
from gpu_helpers import TOL, load_library, rel_frobenius, require_gpu, split_tail, to_host_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbr():
    require_gpu()
    return load_library()


def _capture(fn, replays=3):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                                  # warm-up: per-device setup happens outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(replays):
        g.replay()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("dtype,M,N,K,split", [("ffma", 256, 256, 256, -1), ("bf16", 640, 776, 1352, 1),
                                               ("tf32", 520, 264, 4096, -1)])
def test_gemm_in_graph(gbr, dtype, M, N, K, split):
    A, B, bias = inputs.gemm_normal(M, N, K, seed=90)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    C = torch.empty((M, N), dtype=dA.dtype, device="cuda")
    with split_tail(gbr, split):
        eager = gbr.gemm_bias_relu(dA, dB, db, dtype=dtype, stages=3).clone()
        C.zero_()
        _capture(lambda: gbr.gemm_bias_relu(dA, dB, db, C, dtype=dtype, stages=3,
                                            stream=torch.cuda.current_stream()))
    gbr.check_device()
    ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    assert rel_frobenius(to_host_f64(C), ref) <= TOL[dtype]
    if split == -1 and dtype == "ffma":
        assert torch.equal(C, eager)


def test_copy_and_grouped_in_graph(gbr):
    src = torch.randn(2048, 1024, device="cuda")
    dst = torch.empty_like(src)
    counts = [300, 0, 77]
    _, X, W, b = inputs.grouped(tokens=sum(counts), experts=3, K=256, N=520, seed=91)
    dX, dW, db = X.cuda(), W.cuda(), b.cuda()
    Cg = torch.empty((sum(counts), 520), dtype=torch.bfloat16, device="cuda")

    def work():
        st = torch.cuda.current_stream()
        gbr.staged_copy(src, dst, tile=(128, 64), stages=4, stream=st)
        gbr.gemm_bias_relu_grouped(dX, dW, db, counts, Cg, stages=3, stream=st)

    _capture(work)
    gbr.check_device()
    assert torch.equal(dst, src)
    ref = oracle.gemm_bias_relu_grouped(X.float(), W.float(), b, counts)
    assert rel_frobenius(to_host_f64(Cg), ref) <= TOL["bf16"]


def test_host_path_in_graph(gbr):
    A, B, bias = inputs.gemm_normal(2600, 264, 200, seed=92)
    A, B = A.to(torch.bfloat16).pin_memory(), B.to(torch.bfloat16).pin_memory()
    bias = bias.pin_memory()
    C = torch.zeros((2600, 264), dtype=torch.bfloat16).pin_memory()
    _capture(lambda: gbr.gemm_bias_relu_host(A, B, bias, C, dtype="bf16", stages=3,
                                             stream=torch.cuda.current_stream(), sync=False))
    gbr.check_device()
    ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    assert rel_frobenius(to_host_f64(C), ref) <= TOL["bf16"]


def test_small_gemm_graph_replays(gbr):
    """The 256^3 FFMA workload replayed 200 times from one graph.  Its four
    128 x 128 tiles keep 4 SMs busy for ~28 us per call whether issued eagerly
    or from the graph: the call is bound by those SMs, not by the host."""
    A, B, bias = inputs.workload("gemm_small")
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    C = torch.empty((256, 256), device="cuda")
    fn = lambda: gbr.gemm_bias_relu(dA, dB, db, C, dtype="ffma", stages=2,
                                    stream=torch.cuda.current_stream())
    g = _capture(fn)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(200):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    per_replay_us = e0.elapsed_time(e1) * 1e3 / 200
    gbr.check_device()
    assert rel_frobenius(to_host_f64(C), oracle.gemm_bias_relu(A, B, bias)) <= TOL["ffma"]
    assert per_replay_us < 100.0, per_replay_us
