"""Failure detection on the real pipelines, without a GPU fault.

One stage of one CTA is left unfilled: the producer registers the stage's
expected bytes on the full barrier but issues no TMA load (planted through the
library's self-test entry points).  The consumer's bounded wait must give up,
the kernel must record the site, CTA and item, let its own copies in flight
land, free its Tensor Memory and return; the status is then reported on the
host and the context keeps working (the next normal call is correct).  Nothing
here faults, traps or hangs a GPU: every wait involved has a time limit.
"""
import re

import numpy as np
import pytest
import torch

import oracle
from mbarrier_gemm_pipelines_gb300 import inputs
from gpu_helpers import (TOL, load_library, rel_frobenius, require_gpu, split_tail, to_host_f64,
                         tuned)

pytestmark = pytest.mark.gpu

LIMIT_NS = 50_000_000      # 50 ms per wait
SITE_PRODUCER_EMPTY, SITE_FFMA_CONSUMER, SITE_MMA_FULL = 0x11, 0x21, 0x31
SITE_EPI_ACC_FULL, SITE_STORER_FULL = 0x41, 0x51


def _producer_gave_up(site, got_item, item, stages):
    """The producer may give up first instead: the unfilled stage is never
    released, so its wait for that slot (the item `stages` later, or one
    earlier where the copy releases a slot one store late) runs out too.  Its
    wait starts microseconds after the consumer's and the waits poll with a
    suspend hint, so which of the two records first is a race."""
    return site == SITE_PRODUCER_EMPTY and item + stages - 1 <= got_item <= item + stages


@pytest.fixture(scope="module")
def gbr():
    require_gpu()
    return load_library()


def _status(gbr):
    code = gbr.device_status()
    msg = gbr.last_error()
    return code, msg


def _parse(msg):
    m = re.search(r"site 0x([0-9a-f]+), CTA (\d+), item (\d+)", msg)
    assert m, msg
    return int(m.group(1), 16), int(m.group(2)), int(m.group(3))


def _check_gemm(gbr, A, B, bias, dtype, stages):
    C = gbr.gemm_bias_relu(A, B, bias, dtype=dtype, stages=stages)
    assert gbr.device_status() == 0
    ref = oracle.gemm_bias_relu(to_host_f64(A).astype(np.float32),
                                    to_host_f64(B).astype(np.float32),
                                    bias.cpu().numpy())
    assert rel_frobenius(to_host_f64(C), ref) <= TOL[dtype]


@pytest.mark.parametrize("cta,item", [(0, 0), (3, 1), (5, 3)])
def test_copy_unfilled_stage_times_out_and_recovers(gbr, cta, item):
    # 8192 x 1024 fp32 in 128 x 64 tiles: 1024 tiles, so CTA 5 of the
    # persistent grid (at most one 4-stage ring of 32 KiB tiles per SM) handles
    # at least six of them.
    src = torch.randn(8192, 1024, device="cuda")
    gbr.selftest_copy_skip_load(src, 4, cta, item, LIMIT_NS)
    code, msg = _status(gbr)
    assert code == 6, msg
    site, got_cta, got_item = _parse(msg)
    assert got_cta == cta
    assert (site, got_item) == (SITE_STORER_FULL, item) or _producer_gave_up(site, got_item, item, 4)
    assert gbr.device_status() == 0          # cleared
    dst = gbr.staged_copy(src, tile=(128, 64), stages=4)
    gbr.check_device()
    assert torch.equal(dst, src)


def test_copy_injection_outside_the_launch_is_a_no_op(gbr):
    src = torch.randn(1024, 512, device="cuda")   # 64 tiles: CTA 100000 does not exist
    dst = gbr.selftest_copy_skip_load(src, 3, 100000, 0, LIMIT_NS)
    assert gbr.device_status() == 0
    assert torch.equal(dst, src)


@pytest.mark.parametrize("dtype,stages,cta,item", [
    ("ffma", 3, 0, 0), ("ffma", 4, 2, 5),
    ("bf16", 3, 0, 0), ("bf16", 4, 2, 6),
    ("tf32", 3, 1, 4),
])
def test_gemm_unfilled_stage_times_out_and_recovers(gbr, dtype, stages, cta, item):
    # 512 x 512 x 1024: every CTA holds one output tile and runs >= 8 k-blocks.
    A, B, bias = inputs.gemm_uniform(512, 512, 1024, seed=40 + item)
    dev_dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dA, dB, db = A.to(dev_dt).cuda(), B.to(dev_dt).cuda(), bias.cuda()
    gbr.selftest_gemm_skip_load(dA, dB, db, dtype, stages, cta, item, LIMIT_NS)
    code, msg = _status(gbr)
    assert code == 6, msg
    site, got_cta, got_item = _parse(msg)
    assert got_cta == cta
    if _producer_gave_up(site, got_item, item, stages):
        pass
    elif dtype == "ffma":
        assert (site, got_item) == (SITE_FFMA_CONSUMER, item)
    else:
        # The MMA issuer waits for the stage; the epilogue waits (longer) for
        # the tile's accumulator, so either may give up first.
        assert (site, got_item) in ((SITE_MMA_FULL, item), (SITE_EPI_ACC_FULL, 0))
    assert gbr.device_status() == 0
    _check_gemm(gbr, dA, dB, db, dtype, stages)


def test_gemm_selftest_rejects_bad_arguments(gbr):
    A = torch.zeros(128, 128, device="cuda")
    bias = torch.zeros(128, device="cuda")
    with pytest.raises(Exception):
        gbr.selftest_gemm_skip_load(A, A, bias, "ffma", 3, -1, 0, LIMIT_NS)
    with pytest.raises(Exception):
        gbr.selftest_gemm_skip_load(A, A, bias, "ffma", 3, 0, 0, 0)
    with pytest.raises(Exception):
        gbr.selftest_gemm_skip_load(A, A, bias, "ffma_sync", 3, 0, 0, LIMIT_NS)
    assert gbr.device_status() == 0


def test_repeated_injection_leaves_the_context_usable(gbr):
    """Five timed-out launches in a row (Tensor Memory must be freed each time,
    or the next tcgen05 launch could not allocate), then a correct GEMM."""
    A, B, bias = inputs.gemm_uniform(256, 512, 512, seed=50)
    dA, dB, db = A.to(torch.bfloat16).cuda(), B.to(torch.bfloat16).cuda(), bias.cuda()
    for r in range(5):
        gbr.selftest_gemm_skip_load(dA, dB, db, "bf16", 3, r % 4, r, LIMIT_NS)
        assert gbr.device_status() == 6
    _check_gemm(gbr, dA, dB, db, "bf16", 3)


@pytest.mark.parametrize("dtype,stages,ks,unit,item", [
    ("bf16", 3, 2, 0, 0), ("bf16", 3, 2, 3, 5), ("bf16", 6, 1, 1, 9), ("bf16", 6, 1, 2, 15),
    ("tf32", 3, 2, 2, 3), ("tf32", 6, 1, 0, 11),
])
def test_pair_unfilled_stage_times_out_and_recovers(gbr, dtype, stages, ks, unit, item):
    """The CTA-pair kernel (cta_group::2, the default tensor-core path): both
    CTAs of pair `unit` leave ring item `item` unfilled.  The even CTA's MMA
    lane (or an epilogue or producer wait of either CTA) gives up; the even
    CTA then waits for every load either CTA issued, both free their Tensor
    Memory and return.  512 x 512 x 1024: four 256 x 256 tiles, one per pair,
    8 k-blocks of 128 K or 16 of 64 K each."""
    A, B, bias = inputs.gemm_uniform(512, 512, 1024, seed=60 + item)
    dev_dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dA, dB, db = A.to(dev_dt).cuda(), B.to(dev_dt).cuda(), bias.cuda()
    with tuned(gbr, 2, ks):
        gbr.selftest_gemm_skip_load(dA, dB, db, dtype, stages, unit, item, LIMIT_NS)
        code, msg = _status(gbr)
        assert code == 6, msg
        site, got_cta, got_item = _parse(msg)
        assert got_cta in (2 * unit, 2 * unit + 1)
        assert ((site, got_item) in ((SITE_MMA_FULL, item), (SITE_EPI_ACC_FULL, 0))
                or _producer_gave_up(site, got_item, item, stages)), (hex(site), got_item)
        assert gbr.device_status() == 0
        _check_gemm(gbr, dA, dB, db, dtype, stages)


def test_pair_repeated_injection_leaves_the_context_usable(gbr):
    """Five timed-out CTA-pair launches in a row, alternating 128-K and 64-K
    stages (both CTAs' Tensor Memory must be freed each time), then correct
    GEMMs on the pair and on one CTA per tile."""
    A, B, bias = inputs.gemm_uniform(512, 1024, 768, seed=51)
    dA, dB, db = A.to(torch.bfloat16).cuda(), B.to(torch.bfloat16).cuda(), bias.cuda()
    for r in range(5):
        ks, S = (2, 3) if r % 2 == 0 else (1, 5)
        with tuned(gbr, 2, ks):
            gbr.selftest_gemm_skip_load(dA, dB, db, "bf16", S, r % 8, r + 1, LIMIT_NS)
            assert gbr.device_status() == 6
    with tuned(gbr, 2):
        _check_gemm(gbr, dA, dB, db, "bf16", 3)
    with tuned(gbr, 1):
        _check_gemm(gbr, dA, dB, db, "bf16", 4)


def _random_injections(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        dtype = ["ffma", "bf16", "bf16", "tf32"][rng.integers(4)]
        pair = int(rng.choice([1, 2])) if dtype != "ffma" else -1
        ks = int(rng.choice([1, 2])) if dtype != "ffma" else -1
        q = 8 if dtype == "bf16" else 4
        M, N = int(rng.integers(1, 1200)), q * int(rng.integers(1, 1200 // q))
        K = q * int(rng.integers(1, 1600 // q))
        if dtype == "ffma":
            S = int(rng.integers(1, 5))
            tile_m, tile_n, kb = 128, 128, -(-K // 32)
        else:
            S = int(rng.integers(1, (4 if ks == 1 else 2) + 1 if pair == 1 else (6 if ks == 1 else 3) + 1))
            tile_m, tile_n = 128 * pair, 256
            kb = -(-K // ((64 if dtype == "bf16" else 32) * ks))
        tiles = -(-M // tile_m) * -(-N // tile_n)
        units = 152 if pair != 2 else 76
        unit = int(rng.integers(0, min(tiles, units)))
        item = int(rng.integers(0, kb))         # within the unit's first tile
        cases.append(pytest.param(dtype, pair, ks, S, M, N, K, unit, item,
                                  id="i%02d-%s-p%d-k%d-s%d-%dx%dx%d-u%d-j%d" % (
                                      i, dtype, pair, ks, S, M, N, K, unit, item)))
    return cases


@pytest.mark.parametrize("dtype,pair,ks,S,M,N,K,unit,item", _random_injections(16, 8181))
def test_random_unfilled_stage_times_out_and_recovers(gbr, dtype, pair, ks, S, M, N, K, unit, item):
    """Seeded random shapes, variants, ring depths and injection points (a
    unit that has a tile, an item within its first tile): the wait gives up,
    the site is reported on one of the unit's CTAs, and a normal GEMM on the
    same data afterwards matches the oracle."""
    A, B, bias = inputs.gemm_uniform(M, N, K, seed=M + N + K)
    dev_dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dA, dB, db = A.to(dev_dt).cuda(), B.to(dev_dt).cuda(), bias.cuda()
    with tuned(gbr, pair, ks), split_tail(gbr, 0):
        gbr.selftest_gemm_skip_load(dA, dB, db, dtype, S, unit, item, LIMIT_NS)
        code, msg = _status(gbr)
        assert code == 6, msg
        site, got_cta, got_item = _parse(msg)
        cta_group = 2 if pair == 2 else 1
        assert unit * cta_group <= got_cta < (unit + 1) * cta_group, (got_cta, unit)
        assert gbr.device_status() == 0
        _check_gemm(gbr, dA, dB, db, dtype, S)
