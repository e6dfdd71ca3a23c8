"""GEMM + bias + ReLU on the GPU (through the C ABI) against the binary64 oracle.

Bars (relative Frobenius error): FFMA 1e-5, TF32 5e-3, bf16 1e-2.  Every
problem, the full-size workloads (fp32 4096^3, bf16 8192^3, in the launch
configuration the benchmark uses) included, is compared element by element over
the whole output."""
import numpy as np
import pytest
import torch

import oracle
from mbarrier_gemm_pipelines_gb300 import inputs
from gpu_helpers import (TOL, ffma_warps, load_library, rel_frobenius, require_gpu, split_tail,
                         to_host_f64, tuned)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbr():
    require_gpu()
    return load_library()


def _run(gbr, A, B, bias, dtype, stages):
    C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype=dtype, stages=stages)
    gbr.check_device()
    return to_host_f64(C)


def _check_full(got, A, B, bias, dtype):
    ref = oracle.gemm_bias_relu(A, B, bias)
    err = rel_frobenius(got, ref)
    assert err <= TOL[dtype], err
    assert (got >= 0).all()
    # element-wise: no single output far off (catches a wrong tile at a ragged edge)
    scale = np.abs(ref).max() + 1e-30
    assert np.abs(got - ref).max() <= 20 * TOL[dtype] * scale
    return err


def test_config1_ffma_256_s2(gbr):
    """fp32 256^3, U[-1,1] from seed 0, 2-stage ring, BK = 32."""
    A, B, bias = inputs.workload("gemm_small")
    got = _run(gbr, A, B, bias, "ffma", 2)
    _check_full(got, A, B, bias, "ffma")


# Ragged in every dimension; K and N multiples of 8 so that bf16 rows keep
# 16-byte pitches (the TMA rule).
SHAPES = [(128, 128, 32), (256, 512, 256), (200, 136, 104), (129, 264, 40), (1, 8, 8),
          (300, 520, 200), (640, 384, 1000), (383, 776, 1352)]


VARIANTS = [("ffma", -1), ("ffma_cpasync", -1), ("tf32", 1), ("tf32", 2), ("bf16", 1), ("bf16", 2)]


@pytest.mark.parametrize("dtype,pair", VARIANTS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_small_shapes(gbr, dtype, pair, M, N, K):
    A, B, bias = inputs.gemm_uniform(M, N, K, seed=M * 31 + N * 7 + K)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    with tuned(gbr, pair):
        got = _run(gbr, A, B, bias, dtype, 2)
    _check_full(got, A.float(), B.float(), bias, dtype)


@pytest.mark.parametrize("dtype", ["ffma", "ffma_cpasync", "ffma_sync"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_ffma_layouts_agree(gbr, dtype, M, N, K):
    """The FFMA consumer layouts (8 warps of 8x8, the default, and 16 warps
    of 8x4) add each output's products in the same order: the same bits, and
    parity with the oracle."""
    A, B, bias = inputs.gemm_uniform(M, N, K, seed=M * 13 + N * 5 + K)
    S = 1 if dtype == "ffma_sync" else 3
    outs = []
    for warps in (8, 16):
        with ffma_warps(gbr, warps):
            outs.append(_run(gbr, A, B, bias, dtype, S))
    assert np.array_equal(outs[0], outs[1])
    _check_full(outs[1], A, B, bias, "ffma")


def test_ffma_tuning_is_validated(gbr):
    with pytest.raises(gbr.GbrError):
        gbr.ffma_tuning(12)
    gbr.ffma_tuning(-1)


@pytest.mark.parametrize("dtype,pair,ks", [v + (1,) for v in VARIANTS] +
                         [("tf32", 1, 2), ("tf32", 2, 2), ("bf16", 1, 2), ("bf16", 2, 2)])
def test_stage_sweep(gbr, dtype, pair, ks):
    """Every ring depth, one CTA or a pair per tile, one or two 128-byte K
    slices per stage (K = 640 leaves a ragged last stage in both)."""
    M, N, K = 384, 512, 640
    A, B, bias = inputs.gemm_normal(M, N, K, seed=5)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    smax = gbr.max_stages(gbr.OP_GEMM, {"ffma": 0, "ffma_cpasync": 4, "tf32": 1, "bf16": 2}[dtype])
    assert smax >= 4
    if pair == 1:
        smax = 4                                   # one CTA per tile holds 4 stages
    if ks == 2:
        smax = 2 if pair == 1 else 3               # stages twice as large
    with tuned(gbr, pair, ks):
        for S in range(1, smax + 1):
            got = _run(gbr, A, B, bias, dtype, S)
            _check_full(got, A.float(), B.float(), bias, dtype)


@pytest.mark.parametrize("dtype", ["tf32", "bf16"])
def test_pair_and_single_agree(gbr, dtype):
    """The CTA-pair kernel (M = 256 MMAs) and the one-CTA kernel add the same
    products in the same K order, so their outputs agree to the output rounding."""
    A, B, bias = inputs.gemm_normal(520, 776, 1352, seed=6)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    outs = []
    for pair in (1, 2):
        with tuned(gbr, pair):
            outs.append(_run(gbr, A, B, bias, dtype, 3))
    assert rel_frobenius(outs[1], outs[0]) <= TOL[dtype] / 10
    _check_full(outs[1], A.float(), B.float(), bias, dtype)


@pytest.mark.parametrize("dtype", ["tf32", "bf16"])
@pytest.mark.parametrize("pair", [1, 2])
def test_b_panel_boxes_agree(gbr, dtype, pair):
    """B loaded as one 3-D box of whole panels per K slice (N a multiple of
    the panel width) and as one 2-D box per panel (N ragged: the same B with
    8 zero columns appended) gives the same bits in the shared columns; both
    match the oracle.  N = 1536 makes the last tile's CTAs reach past N (its
    boxes zero-fill whole panels)."""
    M, N, K = 384, 1536, 392
    A, B, bias = inputs.gemm_normal(M, N, K, seed=9)
    Bpad = torch.cat([B, torch.zeros(K, 8)], dim=1)
    biaspad = torch.cat([bias, torch.zeros(8)])
    if dtype == "bf16":
        A, B, Bpad = A.to(torch.bfloat16), B.to(torch.bfloat16), Bpad.to(torch.bfloat16)
    with tuned(gbr, pair), split_tail(gbr, 0):   # the two tile counts would split differently
        whole = _run(gbr, A, B, bias, dtype, 3)
        ragged = _run(gbr, A, Bpad, biaspad, dtype, 3)
    assert np.array_equal(whole, ragged[:, :N])
    _check_full(whole, A.float(), B.float(), bias, dtype)


# Tile counts that leave a partial last round of units, K long enough to split:
# a few tiles only (every unit runs a split run), more tiles than units (whole
# tiles first, then the split round), ragged edges in M and N.
SPLIT_SHAPES = [(383, 776, 1352), (520, 264, 4096), (130, 2056, 3000), (2304, 2304, 1024),
                (256, 256, 8192)]


@pytest.mark.parametrize("dtype,pair", [("tf32", 1), ("tf32", 2), ("bf16", 1), ("bf16", 2),
                                        ("ffma", -1)])
@pytest.mark.parametrize("M,N,K", SPLIT_SHAPES)
def test_split_tail(gbr, dtype, pair, M, N, K):
    """Last round split along K (forced on): parity with the oracle element by
    element, and the unsplit kernel's result up to the order of fp32 additions."""
    A, B, bias = inputs.gemm_normal(M, N, K, seed=M + N + K)
    if dtype == "bf16":
        A, B = A.to(torch.bfloat16), B.to(torch.bfloat16)
    with tuned(gbr, pair):
        with split_tail(gbr, 1):
            got = _run(gbr, A, B, bias, dtype, 3)
        with split_tail(gbr, 0):
            whole = _run(gbr, A, B, bias, dtype, 3)
    _check_full(got, A.float(), B.float(), bias, dtype)
    assert rel_frobenius(got, whole) <= TOL[dtype] / 10


@pytest.mark.parametrize("M,N,K", SPLIT_SHAPES)
def test_ffma_split_tail_is_ordered(gbr, M, N, K):
    """The FFMA split tail (whole tiles in one launch, the last round's
    k-blocks dealt to every CTA in a second) adds each tile's parts in part
    order: the same bits on every call and with either consumer layout."""
    A, B, bias = inputs.gemm_normal(M, N, K, seed=M * 3 + N + K)
    outs = []
    with split_tail(gbr, 1):
        for warps in (8, 8, 16):
            with ffma_warps(gbr, warps):
                outs.append(_run(gbr, A, B, bias, "ffma", 3))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_split_tail_mode_is_validated(gbr):
    with pytest.raises(gbr.GbrError):
        gbr.gemm_split_tail(2)
    gbr.gemm_split_tail(-1)


def test_forced_single_rejects_deep_ring(gbr):
    A = torch.zeros((256, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    bias = torch.zeros(256, device="cuda")
    with tuned(gbr, 1):
        with pytest.raises(gbr.GbrError) as e:
            gbr.gemm_bias_relu(A, B, bias, dtype="bf16", stages=5)
    assert e.value.code == 4
    C = gbr.gemm_bias_relu(A, B, bias, dtype="bf16", stages=6)   # auto: the pair kernel
    gbr.check_device()
    assert bool((C == 0).all())


@pytest.mark.parametrize("dtype,pair", VARIANTS)
def test_k_zero_is_relu_bias(gbr, dtype, pair):
    bias = torch.linspace(-2, 2, 264)
    t = torch.bfloat16 if dtype == "bf16" else torch.float32
    A = torch.empty((270, 0), dtype=t)
    B = torch.empty((0, 264), dtype=t)
    with tuned(gbr, pair):
        C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype=dtype, stages=2)
    gbr.check_device()
    expect = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    if dtype == "bf16":
        expect = torch.from_numpy(expect).to(torch.bfloat16).double().numpy()
    assert np.array_equal(to_host_f64(C), expect)


def test_bf16_output_rounding(gbr):
    """The bf16 result is the fp32 result rounded once: with exactly
    representable small-integer inputs the accumulation is exact, so the output
    must equal the oracle rounded to bf16."""
    g = inputs._gen(9)
    A = torch.randint(-4, 5, (256, 128), generator=g).to(torch.bfloat16)
    B = torch.randint(-4, 5, (128, 512), generator=g).to(torch.bfloat16)
    bias = torch.randint(-50, 51, (512,), generator=g).float() * 0.25
    C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype="bf16", stages=3)
    gbr.check_device()
    ref = oracle.gemm_bias_relu(A.float(), B.float(), bias)
    expect = torch.from_numpy(ref).float().to(torch.bfloat16)
    assert torch.equal(C.cpu(), expect)


def test_ffma_integer_inputs_exact(gbr):
    g = inputs._gen(10)
    A = torch.randint(-8, 9, (200, 96), generator=g).float()
    B = torch.randint(-8, 9, (96, 140), generator=g).float()
    bias = torch.randint(-100, 101, (140,), generator=g).float()
    C = gbr.gemm_bias_relu(A.cuda(), B.cuda(), bias.cuda(), dtype="ffma", stages=3)
    gbr.check_device()
    assert np.array_equal(to_host_f64(C), oracle.gemm_bias_relu(A, B, bias))


def test_errors_are_reported(gbr):
    from mbarrier_gemm_pipelines_gb300 import _binding as b
    lib = b.lib()
    A = torch.zeros((64, 64), device="cuda")
    bias = torch.zeros(64, device="cuda")
    C = torch.zeros((64, 64), device="cuda")
    # stages outside [1, max]
    assert lib.gemm_bias_relu(A.data_ptr(), A.data_ptr(), bias.data_ptr(), C.data_ptr(),
                              64, 64, 64, 0, 0, None) == b.ERR_SMEM
    assert lib.gemm_bias_relu(A.data_ptr(), A.data_ptr(), bias.data_ptr(), C.data_ptr(),
                              64, 64, 64, 2, 9, None) == b.ERR_SMEM
    # row pitch not a multiple of 16 bytes
    assert lib.gemm_bias_relu(A.data_ptr(), A.data_ptr(), bias.data_ptr(), C.data_ptr(),
                              64, 62, 64, 0, 2, None) == b.ERR_ALIGN
    # misaligned base
    assert lib.gemm_bias_relu(A.data_ptr() + 4, A.data_ptr(), bias.data_ptr(), C.data_ptr(),
                              64, 64, 64, 0, 2, None) == b.ERR_ALIGN
    # C overlapping an input
    assert lib.gemm_bias_relu(A.data_ptr(), A.data_ptr(), bias.data_ptr(), A.data_ptr(),
                              64, 64, 64, 0, 2, None) == b.ERR_INVALID
    assert "overlap" in b.last_error()
    assert lib.gemm_bias_relu(A.data_ptr(), A.data_ptr(), bias.data_ptr(), C.data_ptr(),
                              64, 64, 64, 7, 2, None) == b.ERR_INVALID
    assert "dtype 7" in b.last_error()
    assert lib.gemm_bias_relu(None, None, None, None, 0, 64, 64, 0, 2, None) == b.OK
    gbr.check_device()


# ------------------------------------------------------------------ full size
# The full-size workloads are compared element by element over the whole of C:
# the oracle's binary64 product is computed once per workload (with the bias,
# and with a zero bias so that the GEMM part alone, which the N(0, 0.1) bias
# would otherwise dominate, meets the same bar) and every variant's output is
# checked against all of it.

def _full_oracle(A, B, bias):
    A32, B32 = A.float(), B.float()
    return oracle.gemm_bias_relu(A32, B32, bias), oracle.gemm_bias_relu(A32, B32, torch.zeros_like(bias))


@pytest.fixture(scope="module")
def fp32_4096():
    A, B, bias = inputs.workload("gemm_fp32")
    ref, ref0 = _full_oracle(A, B, bias)
    return A, B, bias, ref, ref0


@pytest.fixture(scope="module")
def bf16_8192():
    A, B, bias = inputs.workload("gemm_bf16")
    ref, ref0 = _full_oracle(A, B, bias)
    return A, B, bias, ref, ref0


def _check_against(got, ref, dtype):
    err = rel_frobenius(got, ref)
    assert err <= TOL[dtype], err
    assert (got >= 0).all()
    scale = np.abs(ref).max() + 1e-30
    assert np.abs(got - ref).max() <= 20 * TOL[dtype] * scale
    return err


def _full_size(gbr, case, dtype, stages):
    """Runs the workload with its bias and with a zero bias and compares both
    outputs with the oracle over every element."""
    A, B, bias, ref, ref0 = case
    d_A, d_B, d_bias = A.cuda(), B.cuda(), bias.cuda()
    C = gbr.gemm_bias_relu(d_A, d_B, d_bias, dtype=dtype, stages=stages)
    gbr.check_device()
    _check_against(to_host_f64(C), ref, dtype)
    C0 = gbr.gemm_bias_relu(d_A, d_B, torch.zeros_like(d_bias), dtype=dtype, stages=stages)
    gbr.check_device()
    _check_against(to_host_f64(C0), ref0, dtype)
    return C


@pytest.mark.parametrize("dtype,S,pair", [("ffma", 3, -1), ("ffma", 4, -1), ("ffma_cpasync", 4, -1),
                                           ("ffma16", 4, -1), ("tf32", 3, -1), ("tf32", 4, -1),
                                           ("tf32", 3, 1), ("tf32", 4, 1)])
def test_config3_fp32_4096(gbr, fp32_4096, dtype, S, pair):
    """fp32 4096^3, A, B ~ N(0,1)/sqrt(K), bias ~ N(0, 0.1), seed 2: strict fp32
    FFMA (TMA or cp.async producer; "ffma16": the 16-warp consumer layout) and
    TF32 (CTA pair or one CTA per tile), S in {3, 4}; every output element
    against the oracle."""
    warps = 16 if dtype == "ffma16" else -1
    with tuned(gbr, pair), ffma_warps(gbr, warps):
        _full_size(gbr, fp32_4096, "ffma" if dtype == "ffma16" else dtype, S)


@pytest.mark.parametrize("S,pair,ks", [(4, -1, -1), (5, -1, -1), (6, -1, -1), (4, 1, -1),
                                        (3, 2, 2)])
def test_config4_bf16_8192(gbr, bf16_8192, S, pair, ks):
    """bf16 8192^3, 4-6 stage ring of 64-K stages (the pair kernel by default;
    one CTA per tile at S=4), and the library default 3 x 128 K; every output
    element against the oracle."""
    with tuned(gbr, pair, ks):
        _full_size(gbr, bf16_8192, "bf16", S)


def test_config3_ffma_default_is_deterministic(gbr, fp32_4096):
    """fp32 4096^3 FFMA at S = 3, the default (the split tail is on: 1024
    tiles on 152 CTAs): two calls in a row give the same bits."""
    A, B, bias = (t.cuda() for t in fp32_4096[:3])
    C1 = gbr.gemm_bias_relu(A, B, bias, dtype="ffma", stages=3)
    C2 = gbr.gemm_bias_relu(A, B, bias, dtype="ffma", stages=3)
    gbr.check_device()
    assert torch.equal(C1, C2)


def test_config4_default_is_deterministic(gbr, bf16_8192):
    """The library default for bf16 8192^3 (no split tail there) gives the
    same bits on back-to-back calls."""
    A, B, bias, _, _ = bf16_8192
    d_A, d_B, d_bias = A.cuda(), B.cuda(), bias.cuda()
    C1 = gbr.gemm_bias_relu(d_A, d_B, d_bias, dtype="bf16", stages=3)
    C2 = gbr.gemm_bias_relu(d_A, d_B, d_bias, dtype="bf16", stages=3)
    gbr.check_device()
    assert torch.equal(C1, C2)


def test_wait_timeout_is_reported_and_context_survives(gbr):
    gbr.selftest_wait_timeout(50_000_000)   # 50 ms limit on a wait nothing completes
    assert gbr.device_status() == 6          # GBR_ERR_TIMEOUT
    assert "timed out" in gbr.last_error()
    assert gbr.device_status() == 0          # cleared
    A, B, bias = inputs.gemm_uniform(128, 256, 64, seed=1)
    got = _run(gbr, A, B, bias, "tf32", 2)
    _check_full(got, A, B, bias, "tf32")


def test_launch_order_does_not_matter(gbr):
    """Deep ring, then shallow ring, then deep ring again on the same kernels:
    a kernel's shared-memory limit must only ever be raised, never lowered by a
    smaller launch."""
    from mbarrier_gemm_pipelines_gb300 import _binding as b
    A, B, bias = inputs.gemm_normal(384, 512, 640, seed=12)
    Ab, Bb = A.to(torch.bfloat16), B.to(torch.bfloat16)
    for dtype, S_list in (("bf16", (6, 1, 6, 3, 1, 3)), ("tf32", (6, 1, 6)), ("ffma", (7, 1, 7))):
        a, bb = (Ab, Bb) if dtype == "bf16" else (A, B)
        for S in S_list:
            got = _run(gbr, a, bb, bias, dtype, S)
            _check_full(got, a.float(), bb.float(), bias, dtype)
    src = torch.arange(512 * 64, dtype=torch.float32).reshape(512, 64).cuda()
    for S in (7, 2, 7):
        dst = gbr.staged_copy(src, tile=(128, 64), stages=S)
        gbr.check_device()
        assert torch.equal(dst, src)
    # the allocation-free TF32 variant sets limits on the same one-CTA kernels
    dA, dB, db = A.cuda(), B.cuda(), bias.cuda()
    C = torch.empty((384, 512), device="cuda")
    with tuned(gbr, 1):
        for S in (4, 1):
            assert b.lib().gemm_bias_relu_tf32_noalloc(
                dA.data_ptr(), dB.data_ptr(), db.data_ptr(), C.data_ptr(), 384, 512, 640, S,
                torch.cuda.current_stream().cuda_stream) == b.OK
            gbr.check_device()
            got = _run(gbr, A, B, bias, "tf32", 4)
            _check_full(got, A, B, bias, "tf32")


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_homogeneous_baseline_small(gbr, M, N, K):
    """The section 1.1 loop (all threads load, sync, compute, sync) computes the
    same C as the pipeline, to the FFMA bar."""
    A, B, bias = inputs.gemm_uniform(M, N, K, seed=M * 17 + N * 3 + K)
    got = _run(gbr, A, B, bias, "ffma_sync", 1)
    _check_full(got, A, B, bias, "ffma")


def test_homogeneous_baseline_4096_and_limits(gbr, fp32_4096):
    A, B, bias, _, _ = fp32_4096
    _full_size(gbr, fp32_4096, "ffma_sync", 1)
    assert gbr.max_stages(gbr.OP_GEMM, 3) == 1
    with pytest.raises(gbr.GbrError) as e:
        gbr.gemm_bias_relu(A[:64, :64].contiguous().cuda(), B[:64, :64].contiguous().cuda(),
                           bias[:64].contiguous().cuda(), dtype="ffma_sync", stages=2)
    assert e.value.code == 4
    bias_only = torch.linspace(-1, 1, 136)
    C = gbr.gemm_bias_relu(torch.empty((50, 0)).cuda(), torch.empty((0, 136)).cuda(),
                           bias_only.cuda(), dtype="ffma_sync", stages=1)
    gbr.check_device()
    assert torch.equal(C.cpu(), torch.clamp(bias_only, min=0).expand(50, 136))
