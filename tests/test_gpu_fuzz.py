"""Seeded random problems against the binary64 oracle, element by element.

Each case draws its shape and every launch option at once: the kernel (FFMA in
its three loaders, TF32, bf16), one CTA or a CTA pair per tile, one or two
128-byte K slices per ring stage, the ring depth, the split tail (auto, never,
forced), the dynamic tile counter and programmatic dependent launch.  M is any
size from 1 row (a fifth of the draws take several rounds of tiles over the
SMs), K may be 0, and N and K are multiples of 16 bytes (the TMA row-pitch
rule: 8 bf16 or 4 fp32 elements); half the draws make N a whole number of B
panels (64 bf16 or 32 fp32 columns), where the panels of a K slice come in one
3-D box, the rest take the per-panel boxes.  The grouped cases draw expert
counts with empty and one-row experts the same way; the staged-copy cases draw
shape, tile, ring depth and the copy's knobs; the host-buffer cases draw shape,
kernel and pinned or pageable buffers; the traced cases run the event-trace
kernel instances and check their ring events as well as their outputs; the
graph cases capture random call sequences into CUDA graphs and replay them.  The
draws come from fixed seeds, so a failing case id names a problem that can be
rerun."""
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


class options:
    """Sets the launch options of one case for a with-block, then restores the
    defaults (automatic variant, auto split, static schedule, overlap on)."""

    def __init__(self, gbr, pair, ks, split, dynamic, overlap):
        self.gbr = gbr
        self.ctx = [tuned(gbr, pair, ks), split_tail(gbr, split)]
        self.dynamic, self.overlap = dynamic, overlap

    def __enter__(self):
        for c in self.ctx:
            c.__enter__()
        self.gbr.gemm_dynamic_schedule(self.dynamic)
        self.gbr.launch_overlap(self.overlap)
        return self

    def __exit__(self, *exc):
        self.gbr.launch_overlap(True)
        self.gbr.gemm_dynamic_schedule(False)
        for c in reversed(self.ctx):
            c.__exit__(*exc)
        return False


def _stage_limit(dtype, pair, ks):
    """Deepest ring each variant holds in shared memory (the library refuses
    deeper ones with an error, which these draws stay clear of)."""
    if dtype == "ffma_sync":
        return 1
    if dtype.startswith("ffma"):
        return 4
    if pair == 1:
        return 4 if ks == 1 else 2
    return 6 if ks == 1 else 3


def _dense_cases(n, seed):
    rng = np.random.default_rng(seed)
    kinds = ["ffma", "ffma_cpasync", "ffma_sync", "tf32", "tf32", "bf16", "bf16", "bf16"]
    cases = []
    for i in range(n):
        dtype = kinds[rng.integers(len(kinds))]
        q = 8 if dtype == "bf16" else 4                    # elements per 16 bytes
        panel = 64 if dtype == "bf16" else 32
        M = int(rng.integers(1500, 5000)) if rng.random() < 0.2 else int(rng.integers(1, 1500))
        N = (panel * int(rng.integers(1, 2400 // panel)) if rng.random() < 0.5
             else q * int(rng.integers(1, 2400 // q)))
        K = 0 if rng.random() < 0.05 else q * int(rng.integers(1, 2080 // q))
        umma = dtype in ("tf32", "bf16")
        pair = int(rng.choice([1, 2])) if umma else -1
        ks = int(rng.choice([1, 2])) if umma else -1
        S = int(rng.integers(1, _stage_limit(dtype, pair, ks) + 1))
        split = int(rng.choice([-1, 0, 1]))
        dynamic = bool(umma and rng.random() < 0.3)
        overlap = bool(rng.random() < 0.7)
        cases.append(pytest.param(dtype, M, N, K, pair, ks, S, split, dynamic, overlap,
                                  id="d%02d-%s-%dx%dx%d-p%d-k%d-s%d-t%d-%s%s" % (
                                      i, dtype, M, N, K, pair, ks, S, split,
                                      "dyn" if dynamic else "st", "-ov" if overlap else "")))
    return cases


@pytest.mark.parametrize("dtype,M,N,K,pair,ks,S,split,dynamic,overlap", _dense_cases(96, 20261203))
def test_dense_random(gbr, dtype, M, N, K, pair, ks, S, split, dynamic, overlap):
    A, B, bias = inputs.gemm_normal(M, N, K, seed=M * 7 + N * 3 + K)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    with options(gbr, pair, ks, split, dynamic, overlap):
        C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype=dtype, stages=S)
    gbr.check_device()
    got = to_host_f64(C)
    ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    if dtype == "bf16":                    # the kernel rounds its output to bf16
        ref_cmp = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    else:
        ref_cmp = ref
    assert got.shape == (M, N)
    assert (got >= 0).all()
    if K == 0:
        assert np.array_equal(got, ref_cmp)
        return
    assert rel_frobenius(got, ref) <= TOL[dtype]
    scale = np.abs(ref).max() + 1e-30
    assert np.abs(got - ref).max() <= 20 * TOL[dtype] * scale


def _grouped_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        G = int(rng.integers(1, 10))
        counts = []
        for _ in range(G):
            r = rng.random()
            counts.append(0 if r < 0.15 else 1 if r < 0.25 else int(rng.integers(2, 700)))
        K = 8 * int(rng.integers(1, 200))
        N = 64 * int(rng.integers(1, 20)) if rng.random() < 0.5 else 8 * int(rng.integers(1, 160))
        pair = int(rng.choice([-1, 1, 2]))
        S = int(rng.integers(1, 5 if pair == 1 else 7))
        split = int(rng.choice([-1, 0, 1]))
        thin = bool(rng.random() < 0.7)
        dynamic = bool(rng.random() < 0.3)
        overlap = bool(rng.random() < 0.7)
        cases.append(pytest.param(counts, K, N, pair, S, split, thin, dynamic, overlap,
                                  id="g%02d-%s-%dx%d-p%d-s%d-t%d-%s-%s%s" % (
                                      i, "_".join(map(str, counts)), K, N, pair, S, split,
                                      "thin" if thin else "wide", "dyn" if dynamic else "st",
                                      "-ov" if overlap else "")))
    return cases


@pytest.mark.parametrize("counts,K,N,pair,S,split,thin,dynamic,overlap",
                         _grouped_cases(48, 31415))
def test_grouped_random(gbr, counts, K, N, pair, S, split, thin, dynamic, overlap):
    G, T = len(counts), sum(counts)
    _, X, W, b = inputs.grouped(tokens=max(T, 1), experts=G, K=K, N=N, seed=T + K + N)
    X = X[:T].contiguous()                 # all experts empty: a 0-row X
    with options(gbr, pair, -1, split, dynamic, overlap), thin_tail(gbr, thin):
        C = gbr.gemm_bias_relu_grouped(X.cuda(), W.cuda(), b.cuda(), counts, stages=S)
    gbr.check_device()
    got = to_host_f64(C)
    assert got.shape == (T, N)
    if T == 0:
        return
    ref = oracle.gemm_bias_relu_grouped(X.float(), W.float(), b, counts)
    assert (got >= 0).all()
    assert rel_frobenius(got, ref) <= TOL["bf16"]
    scale = np.abs(ref).max() + 1e-30
    assert np.abs(got - ref).max() <= 20 * TOL["bf16"] * scale


def _copy_cases(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        rows = 0 if rng.random() < 0.03 else int(rng.integers(1, 6000))
        cols = 4 * int(rng.integers(1, 1100))
        tr = int(rng.choice([1, 5, 8, 16, 32, 64, 100, 128, 256]))
        tc = 4 * int(rng.choice([1, 2, 3, 8, 16, 24, 32, 64]))
        dtype = "i32" if rng.random() < 0.3 else "f32"
        lag = int(rng.choice([-1, 0, 1]))
        hint = int(rng.choice([-1, 0, 1, 2, 3]))
        ctas = int(rng.choice([-1, 1]))
        u = rng.random()                                  # ring depth: a fraction of the limit
        cases.append(pytest.param(rows, cols, tr, tc, dtype, lag, hint, ctas, u,
                                  id="c%02d-%dx%d-t%dx%d-%s-l%d-h%d-c%d" % (
                                      i, rows, cols, tr, tc, dtype, lag, hint, ctas)))
    return cases


@pytest.mark.parametrize("rows,cols,tr,tc,dtype,lag,hint,ctas,u", _copy_cases(40, 4242))
def test_copy_random(gbr, rows, cols, tr, tc, dtype, lag, hint, ctas, u):
    smax = min(gbr.max_stages(gbr.OP_COPY, 0, tr, tc), 8)
    if smax == 0:                  # one tile does not fit a CTA's shared memory: rejected
        with pytest.raises(gbr.GbrError) as e:
            gbr.staged_copy(torch.zeros((8, 8), device="cuda"), tile=(tr, tc), stages=1)
        assert e.value.code == 4   # GBR_ERR_SMEM
        return
    S = min(1 + int(u * smax), smax)
    if lag == 1 and S < 2:
        lag = 0
    g = inputs._gen(rows * 31 + cols * 7 + tr + tc)
    src = inputs.uniform((rows, cols), -1e3, 1e3, g)
    if dtype == "i32":
        src = src.view(torch.int32)
    expect = oracle.copy(src.numpy())
    dst = torch.full((rows, cols), -1, dtype=src.dtype, device="cuda")
    gbr.copy_tuning(lag, ctas, hint)
    try:
        gbr.staged_copy(src.cuda(), dst, tile=(tr, tc), stages=S)
        gbr.check_device()
    finally:
        gbr.copy_tuning(-1, -1, -1)
    assert np.array_equal(dst.cpu().view(torch.int32).numpy(), expect.view(np.int32))


def _host_cases(n, seed):
    rng = np.random.default_rng(seed)
    kinds = ["ffma", "tf32", "bf16", "bf16"]
    cases = []
    for i in range(n):
        dtype = kinds[rng.integers(len(kinds))]
        q = 8 if dtype == "bf16" else 4
        M = int(rng.integers(1, 5000))
        N = q * int(rng.integers(1, 800 // q))
        K = 0 if rng.random() < 0.1 else q * int(rng.integers(1, 800 // q))
        S = int(rng.integers(1, 4))
        pinned = bool(rng.random() < 0.7)
        cases.append(pytest.param(dtype, M, N, K, S, pinned,
                                  id="h%02d-%s-%dx%dx%d-s%d-%s" % (
                                      i, dtype, M, N, K, S, "pin" if pinned else "page")))
    return cases


@pytest.mark.parametrize("dtype,M,N,K,S,pinned", _host_cases(16, 777))
def test_host_random(gbr, dtype, M, N, K, S, pinned):
    """gemm_bias_relu_host (copies in, GEMM in row chunks, copy out) against
    the device-buffer call bit for bit (split tail off: both add every output's
    products in the same order) and against the oracle."""
    A, B, bias = inputs.gemm_normal(M, N, K, seed=M + 3 * N + 5 * K)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    if pinned:
        A, B, bias = A.pin_memory(), B.pin_memory(), bias.pin_memory()
    with split_tail(gbr, 0):
        C = gbr.gemm_bias_relu_host(A, B, bias, dtype=dtype, stages=S)
        D = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype=dtype, stages=S)
    gbr.check_device()
    assert torch.equal(C, D.cpu())
    got = to_host_f64(C)
    ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    if K == 0:
        if dtype == "bf16":
            ref = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        assert np.array_equal(got, ref)
        return
    assert rel_frobenius(got, ref) <= TOL[dtype]


def _trace_cases(n, seed):
    rng = np.random.default_rng(seed)
    kinds = ["copy", "ffma", "ffma_cpasync", "tf32", "bf16", "bf16", "grouped"]
    cases = []
    for i in range(n):
        kind = kinds[rng.integers(len(kinds))]
        pair = int(rng.choice([1, 2]))
        ks = int(rng.choice([1, 2]))
        split = int(rng.choice([-1, 0, 1]))
        dyn = bool(kind in ("tf32", "bf16", "grouped") and rng.random() < 0.3)
        q = 8 if kind in ("bf16", "grouped") else 4
        M = int(rng.integers(1, 3000))
        N = q * int(rng.integers(1, 2000 // q))
        K = q * int(rng.integers(1, 1600 // q))
        u = rng.random()
        cases.append(pytest.param(kind, M, N, K, pair, ks, split, dyn, u,
                                  id="t%02d-%s-%dx%dx%d-p%d-k%d-t%d-%s" % (
                                      i, kind, M, N, K, pair, ks, split, "dyn" if dyn else "st")))
    return cases


@pytest.mark.parametrize("kind,M,N,K,pair,ks,split,dyn,u", _trace_cases(24, 5151))
def test_trace_random(gbr, kind, M, N, K, pair, ks, split, dyn, u):
    """Seeded random problems run by the traced kernel instances: the output
    against the oracle, the recorded ring events through the protocol checker
    and, unit by unit, through the oracle's ring-simulator replay."""
    from mbarrier_gemm_pipelines_gb300 import trace
    from test_gpu_trace import replay_units
    from trace_check import check
    if kind == "copy":
        tr, tc = 8 * (1 + int(u * 16)), 4 * (1 + int(u * 32))     # up to 128 x 128
        S = min(gbr.max_stages(gbr.OP_COPY, 0, tr, tc), 1 + int(u * 7))
        src = inputs.uniform((M, 4 * (N // 4)), -1e3, 1e3, inputs._gen(M + N))
        with trace.Recorder() as rec:
            dst = gbr.staged_copy(src.cuda(), tile=(tr, tc), stages=S)
            ev, cnt = rec.events()
        gbr.check_device()
        assert np.array_equal(dst.cpu().numpy(), oracle.copy(src.numpy()))
        assert check(ev, cnt, S) == []
        assert replay_units(ev, S) >= 1
        return
    if kind == "grouped":
        G = 1 + int(u * 8)
        counts = [int(c) for c in np.random.default_rng(M).integers(0, 2 * M // G + 2, G)]
        _, X, W, b = inputs.grouped(tokens=max(sum(counts), 1), experts=G, K=K, N=N, seed=M + K)
        X = X[:sum(counts)].contiguous()
        S = 1 + int(u * (4 if pair == 1 else 3))
        gbr.gemm_dynamic_schedule(dyn)
        try:
            with tuned(gbr, pair), split_tail(gbr, split), trace.Recorder() as rec:
                C = gbr.gemm_bias_relu_grouped(X.cuda(), W.cuda(), b.cuda(), counts, stages=S)
                ev, cnt = rec.events()
        finally:
            gbr.gemm_dynamic_schedule(False)
        gbr.check_device()
        if sum(counts) == 0:
            return
        ref = oracle.gemm_bias_relu_grouped(X.float(), W.float(), b, counts)
        assert rel_frobenius(to_host_f64(C), ref) <= TOL["bf16"]
        assert check(ev, cnt, S, cta_group=pair, accumulator=True) == []
        assert replay_units(ev, S, cta_group=pair, accumulator=True) >= 1
        return
    A, B, bias = inputs.gemm_normal(M, N, K, seed=M + 2 * N + 3 * K)
    if kind == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    umma = kind in ("tf32", "bf16")
    S = 1 + int(u * ((4 if ks == 1 else 2) if pair == 1 else (6 if ks == 1 else 3))) if umma \
        else 1 + int(u * 4)
    gbr.gemm_dynamic_schedule(dyn)
    try:
        with tuned(gbr, pair if umma else -1, ks if umma else -1), split_tail(gbr, split):
            with trace.Recorder() as rec:
                C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype=kind, stages=S)
                ev, cnt = rec.events()
    finally:
        gbr.gemm_dynamic_schedule(False)
    gbr.check_device()
    ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    assert rel_frobenius(to_host_f64(C), ref) <= TOL[kind]
    if umma:
        assert check(ev, cnt, S, cta_group=pair, accumulator=True) == []
        assert replay_units(ev, S, cta_group=pair, accumulator=True) >= 1
    else:
        assert check(ev, cnt, S) == []
        assert replay_units(ev, S) >= 1


def _graph_cases(n, seed):
    rng = np.random.default_rng(seed)
    return [pytest.param(int(rng.integers(0, 2 ** 31)), id="g%02d" % i) for i in range(n)]


@pytest.mark.parametrize("case_seed", _graph_cases(12, 6262))
def test_graph_random(gbr, case_seed):
    """A random sequence of three calls (dense GEMM with a random kernel,
    split mode and tile order; grouped GEMM; staged copy) captured into one
    CUDA graph after an eager run, then replayed twice: each output matches
    the oracle, and the eager output bit for bit where the call is
    deterministic (every call but a tensor-core split tail, forced or chosen
    by the automatic rule, whose parts are added in arrival order)."""
    rng = np.random.default_rng(case_seed)
    ops = []
    for k in range(3):
        kind = ["dense", "dense", "grouped", "copy"][rng.integers(4)]
        if kind == "dense":
            dtype = ["ffma", "tf32", "bf16"][rng.integers(3)]
            q = 8 if dtype == "bf16" else 4
            M, N, K = int(rng.integers(1, 2000)), q * int(rng.integers(1, 1200 // q)), \
                q * int(rng.integers(1, 1600 // q))
            split = int(rng.choice([-1, 0, 1]))
            dyn = bool(dtype != "ffma" and rng.random() < 0.4)
            A, B, bias = inputs.gemm_normal(M, N, K, seed=int(rng.integers(0, 10 ** 6)))
            if dtype == "bf16":
                A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
            dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
            C = torch.empty((M, N), dtype=dA.dtype, device="cuda")
            ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)

            def call(st, dA=dA, dB=dB, db=db, C=C, dtype=dtype, split=split, dyn=dyn):
                gbr.gemm_split_tail(split)
                gbr.gemm_dynamic_schedule(dyn)
                try:
                    gbr.gemm_bias_relu(dA, dB, db, C, dtype=dtype, stages=3, stream=st)
                finally:
                    gbr.gemm_split_tail(-1)
                    gbr.gemm_dynamic_schedule(False)
            exact = dtype == "ffma" or dyn or split == 0    # no arrival-order split sums
            ops.append((call, C, ref, TOL[dtype], exact))
        elif kind == "grouped":
            G = int(rng.integers(1, 6))
            counts = [int(c) for c in rng.integers(0, 600, G)]
            Kg, Ng = 8 * int(rng.integers(1, 100)), 8 * int(rng.integers(1, 100))
            _, X, W, b = inputs.grouped(tokens=max(sum(counts), 1), experts=G, K=Kg, N=Ng,
                                        seed=int(rng.integers(0, 10 ** 6)))
            X = X[:sum(counts)].contiguous()
            dX, dW, db = X.cuda(), W.cuda(), b.cuda()
            Cg = torch.empty((sum(counts), Ng), dtype=torch.bfloat16, device="cuda")
            ref = (oracle.gemm_bias_relu_grouped(X.float(), W.float(), b, counts)
                   if sum(counts) else np.zeros((0, Ng)))

            def call(st, dX=dX, dW=dW, db=db, counts=counts, Cg=Cg):
                gbr.gemm_bias_relu_grouped(dX, dW, db, counts, Cg, stages=3, stream=st)
            ops.append((call, Cg, ref, TOL["bf16"], True))
        else:
            rows, cols = int(rng.integers(1, 3000)), 4 * int(rng.integers(1, 600))
            src = inputs.uniform((rows, cols), -1e3, 1e3, inputs._gen(rows + cols))
            dsrc = src.cuda()
            dst = torch.empty_like(dsrc)

            def call(st, dsrc=dsrc, dst=dst):
                gbr.staged_copy(dsrc, dst, tile=(64, 64), stages=4, stream=st)
            ops.append((call, dst, src.numpy().astype(np.float64), 0.0, True))

    def work():
        st = torch.cuda.current_stream()
        for call, *_ in ops:
            call(st)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        work()                                  # eager run (also does per-device set-up)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    gbr.check_device()
    eager = [out.clone() for _, out, *_ in ops]
    for _, out, *_ in ops:
        out.fill_(0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        work()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    gbr.check_device()
    for (call, out, ref, tol, exact), e in zip(ops, eager):
        got = to_host_f64(out)
        if tol == 0.0:
            assert np.array_equal(got, ref)
        elif got.size:
            assert rel_frobenius(got, ref) <= tol
        if exact:
            assert torch.equal(out, e)
