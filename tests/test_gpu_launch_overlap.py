"""Programmatic dependent launch (gbr_launch_overlap).

With it on, a library kernel may be scheduled while the previous kernel in the
stream is still running; its CTAs set up, then wait (griddepcontrol.wait) for
that kernel to complete before touching global memory.  These tests chain
kernels that read what the previous one wrote (read after write) and that
overwrite what the previous one is still reading (write after read), across
all the library's kernels and torch's, and require the results of the
non-overlapped launches bit for bit."""
import pytest
import torch

from mbarrier_gemm_pipelines_gb300 import inputs
from gpu_helpers import load_library, require_gpu, split_tail

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbr():
    require_gpu()
    lib = load_library()
    yield lib
    lib.launch_overlap(True)


def _copy(gbr, x, stages):
    """Bit copy of a contiguous tensor through the staged copy (as int32 words)."""
    y = torch.empty_like(x)
    gbr.staged_copy(x.view(torch.int32).view(x.shape[0], -1), y.view(torch.int32).view(x.shape[0], -1),
                    tile=(128, 64), stages=stages)
    return y


def _chain(gbr, dtype):
    """copy -> GEMM reading the copy -> copy of the GEMM's output -> torch
    kernel -> GEMM reading that as A (each reads what the previous wrote),
    then a copy that overwrites the source of the copy before it."""
    M = N = K = 1024
    A, B, bias = inputs.gemm_normal(M, N, K, seed=21)
    dev_dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    A, B, bias = A.to(dev_dt).cuda(), B.to(dev_dt).cuda(), bias.cuda()
    A2 = _copy(gbr, A, 4)
    C1 = gbr.gemm_bias_relu(A2, B, bias, dtype=dtype, stages=3)
    C1c = _copy(gbr, C1, 2)
    C1c.mul_(0.5)
    C2 = gbr.gemm_bias_relu(C1c, B, bias, dtype=dtype, stages=3)
    X = torch.randn(4096, 1024, device="cuda")
    Z = torch.randn_like(X)
    X0 = X.clone()
    Y = torch.empty_like(X)
    gbr.staged_copy(X, Y, tile=(128, 64), stages=4)      # reads X
    gbr.staged_copy(Z, X, tile=(128, 64), stages=4)      # then overwrites X
    torch.cuda.synchronize()
    gbr.check_device()
    assert torch.equal(Y, X0) and torch.equal(X, Z)
    assert torch.equal(A2, A)
    return [A2, C1, C1c, C2]


@pytest.mark.parametrize("dtype", ["ffma", "tf32", "bf16"])
def test_overlapped_chain_equals_plain(gbr, dtype):
    # Split tail off: its L2 reductions add partial sums in arrival order, so
    # only the unsplit GEMM is deterministic to the bit.
    with split_tail(gbr, 0):
        gbr.launch_overlap(True)
        got = _chain(gbr, dtype)
        gbr.launch_overlap(False)
        try:
            ref = _chain(gbr, dtype)
        finally:
            gbr.launch_overlap(True)
    for g, r in zip(got, ref):
        assert torch.equal(g, r)


def test_back_to_back_copies_ping_pong(gbr):
    """Forty dependent copies, each reading the previous one's output."""
    a = torch.randn(2048, 2048, device="cuda")
    b = torch.empty_like(a)
    ref = a.clone()
    for i in range(40):
        src, dst = (a, b) if i % 2 == 0 else (b, a)
        gbr.staged_copy(src, dst, tile=(128, 64), stages=(i % 4) + 1)
    torch.cuda.synchronize()
    gbr.check_device()
    assert torch.equal(a, ref) and torch.equal(b, ref)


def test_switch_is_validated(gbr):
    with pytest.raises(gbr.GbrError):
        gbr.check(gbr.lib().gbr_launch_overlap(2))
    gbr.launch_overlap(True)


def _random_sequence(gbr, seed, n_ops=60):
    """A seeded random program over four 512 x 512 fp32 buffers: staged copies,
    FFMA and TF32 GEMMs and torch kernels, each reading buffers earlier ops
    wrote; returns the buffers at the end."""
    g = torch.Generator().manual_seed(seed)
    bufs = [torch.rand(512, 512, generator=g).cuda() for _ in range(4)]
    bias = (torch.rand(512, generator=g) - 0.5).cuda()
    for _ in range(n_ops):
        op = int(torch.randint(0, 4, (1,), generator=g))
        i, j, k = (int(x) for x in torch.randperm(4, generator=g)[:3])
        if op == 0:
            gbr.staged_copy(bufs[i], bufs[k], tile=(128, 64), stages=int(torch.randint(1, 8, (1,), generator=g)))
        elif op in (1, 2):
            gbr.gemm_bias_relu(bufs[i], bufs[j], bias, bufs[k], dtype="ffma" if op == 1 else "tf32",
                               stages=3)
            bufs[k].div_(bufs[k].amax().clamp_min(1e-3))     # torch kernels: keep values in [0, 1]
        else:
            bufs[k].mul_(0.75).add_(bufs[i], alpha=0.25)
    torch.cuda.synchronize()
    gbr.check_device()
    return [b.clone() for b in bufs]


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_dependent_sequence_equals_plain(gbr, seed):
    with split_tail(gbr, 0):
        gbr.launch_overlap(True)
        got = _random_sequence(gbr, seed)
        gbr.launch_overlap(False)
        try:
            ref = _random_sequence(gbr, seed)
        finally:
            gbr.launch_overlap(True)
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
