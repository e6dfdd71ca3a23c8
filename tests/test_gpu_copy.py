"""Staged copy (TMA gmem -> smem -> gmem through the S-slot ring) against the
oracle's memcpy: bit-exact.

Workload of record: fp32 [16384, 4096] (256 MiB) U[-1e3, 1e3] from seed 1,
tiles 128x64, S in {2, 4} and 7 (S = 8 does not fit a CTA's shared memory at
this tile and must be rejected)."""
import numpy as np
import pytest
import torch

import oracle
from mbarrier_gemm_pipelines_gb300 import inputs
from gpu_helpers import load_library, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gbr():
    require_gpu()
    return load_library()


def _bits(t):
    return t.contiguous().view(torch.int32).cpu().numpy()


@pytest.mark.parametrize("rows,cols,tile,S", [
    (128, 64, (128, 64), 1),
    (1000, 200, (128, 64), 2),       # ragged in both dimensions
    (257, 68, (128, 64), 3),
    (384, 256, (64, 128), 4),
    (5, 4, (128, 64), 2),            # smaller than one tile
    (3000, 1028, (128, 64), 7),
    (777, 132, (256, 32), 5),
    (64, 4096, (16, 256), 6),
])
def test_copy_small_bit_exact(gbr, rows, cols, tile, S):
    src = inputs.uniform((rows, cols), -1e3, 1e3, inputs._gen(rows * 7919 + cols))
    expect = oracle.copy(src.numpy())
    dst = torch.full((rows, cols), float("nan"), device="cuda")
    gbr.staged_copy(src.cuda(), dst, tile=tile, stages=S)
    gbr.check_device()
    assert np.array_equal(_bits(dst), expect.view(np.int32))


@pytest.mark.parametrize("tile,S", [((1, 8), 3), ((5, 12), 4), ((3, 4), 8), ((7, 36), 2),
                                    ((1, 4), 1), ((33, 20), 5)])
def test_copy_tiles_not_multiple_of_128_bytes(gbr, tile, S):
    """Tiles of 16 to 3696 bytes that are not whole multiples of 128: every
    ring slot still starts on a 128-byte boundary (TMA's shared-memory
    alignment), and the copy is bit-exact."""
    rows, cols = 1000, 612
    src = inputs.uniform((rows, cols), -1e3, 1e3, inputs._gen(tile[0] * 131 + tile[1] + S))
    expect = oracle.copy(src.numpy())
    dst = torch.full((rows, cols), float("nan"), device="cuda")
    gbr.staged_copy(src.cuda(), dst, tile=tile, stages=S)
    gbr.check_device()
    assert np.array_equal(_bits(dst), expect.view(np.int32))


def test_copy_special_values(gbr):
    bits = np.array([0x7FC00001, 0x80000000, 0x7F800000, 0xFF800000, 0x00000001, 0x7F7FFFFF,
                     0xFFFFFFFF, 0x3F800000], dtype=np.uint32)
    src = torch.from_numpy(np.tile(bits, (33, 16)).view(np.int32)).contiguous()
    dst = torch.zeros_like(src, device="cuda")
    gbr.staged_copy(src.cuda(), dst, tile=(16, 32), stages=2)
    gbr.check_device()
    assert np.array_equal(dst.cpu().numpy(), oracle.copy(src.numpy()))


@pytest.mark.parametrize("S", [2, 4, 7])
@pytest.mark.parametrize("store_lag,l2_hint", [(-1, -1), (0, -1), (-1, 3), (1, 1)])
def test_copy_full_size_bit_exact(gbr, S, store_lag, l2_hint):
    src = inputs.workload("copy")
    expect = oracle.copy(src.numpy())
    d_src = src.cuda()
    dst = torch.empty_like(d_src)
    gbr.copy_tuning(store_lag, -1, l2_hint)
    try:
        gbr.staged_copy(d_src, dst, tile=(128, 64), stages=S)
        gbr.check_device()
    finally:
        gbr.copy_tuning(-1, -1, -1)
    assert np.array_equal(_bits(dst), expect.view(np.int32))


def test_copy_stage_limits(gbr):
    smax = gbr.max_stages(gbr.OP_COPY, 0, 128, 64)
    assert smax == 7
    src = torch.zeros((256, 64), device="cuda")
    with pytest.raises(gbr.GbrError) as e:
        gbr.staged_copy(src, tile=(128, 64), stages=8)
    assert e.value.code == 4   # GBR_ERR_SMEM
    with pytest.raises(gbr.GbrError) as e:
        gbr.staged_copy(src, tile=(128, 64), stages=0)
    assert e.value.code == 4


def test_copy_rejects_bad_arguments(gbr):
    from mbarrier_gemm_pipelines_gb300 import _binding as b
    lib = b.lib()
    x = torch.zeros((64, 64), device="cuda")
    y = torch.zeros((64, 64), device="cuda")
    assert lib.staged_copy(x.data_ptr() + 4, y.data_ptr(), 8, 8, 8, 8, 2, None) == b.ERR_ALIGN
    assert lib.staged_copy(x.data_ptr(), y.data_ptr(), 8, 6, 8, 8, 2, None) == b.ERR_ALIGN
    assert lib.staged_copy(x.data_ptr(), x.data_ptr() + 64, 8, 8, 8, 8, 2, None) == b.ERR_INVALID
    assert lib.staged_copy(x.data_ptr(), y.data_ptr(), 8, 8, 300, 8, 2, None) == b.ERR_INVALID
    assert lib.staged_copy(x.data_ptr(), y.data_ptr(), 0, 8, 8, 8, 2, None) == b.OK
    assert lib.staged_copy(None, None, 0, 0, 8, 8, 2, None) == b.OK
    gbr.check_device()
