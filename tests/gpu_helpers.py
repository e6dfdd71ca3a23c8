"""Shared helpers of the GPU parity tests (no arithmetic of the operators)."""
import numpy as np
import pytest
import torch

# Parity bars (relative Frobenius error against the binary64 oracle).
TOL = {"ffma": 1e-5, "ffma_sync": 1e-5, "ffma_cpasync": 1e-5, "tf32": 5e-3, "bf16": 1e-2}


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    major, minor = torch.cuda.get_device_capability(0)
    if (major, minor) != (10, 3):
        pytest.fail("this library targets sm_103a; found sm_%d%d" % (major, minor))


def load_library():
    import mbarrier_gemm_pipelines_gb300 as gbr
    gbr.build()
    gbr.lib()
    return gbr


def to_host_f64(t):
    return t.detach().to("cpu").to(torch.float64).numpy()


def rel_frobenius(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((got - ref).ravel())
    return num / den if den > 0 else num


def sample_points(M, N, n, seed, extra_rows=(), extra_cols=()):
    """n random (m, n) positions plus the corners and the given rows/columns."""
    rng = np.random.default_rng(seed)
    ms = list(rng.integers(0, M, n))
    ns = list(rng.integers(0, N, n))
    for m in (0, M - 1):
        for c in (0, N - 1):
            ms.append(m)
            ns.append(c)
    for r in extra_rows:
        cols = rng.integers(0, N, 64)
        ms += [r] * len(cols)
        ns += list(cols)
    for c in extra_cols:
        rows = rng.integers(0, M, 64)
        ms += list(rows)
        ns += [c] * len(rows)
    return np.array(ms, dtype=np.int64), np.array(ns, dtype=np.int64)


class tuned:
    """Forces the tensor-core GEMM variant (1: one CTA per tile, 2: CTA pair)
    for the duration of a with-block, then restores the automatic choice."""

    def __init__(self, gbr, pair, k_per_stage=-1):
        self.gbr, self.pair, self.ks = gbr, pair, k_per_stage

    def __enter__(self):
        self.gbr.gemm_tuning(self.pair, -1, -1, self.ks)
        return self

    def __exit__(self, *exc):
        self.gbr.gemm_tuning(-1, -1, -1, -1)
        return False


class split_tail:
    """Sets the tensor-core GEMMs' split-tail mode (-1 auto, 0 never, 1 whenever
    possible) for the duration of a with-block, then restores auto."""

    def __init__(self, gbr, mode):
        self.gbr, self.mode = gbr, mode

    def __enter__(self):
        self.gbr.gemm_split_tail(self.mode)
        return self

    def __exit__(self, *exc):
        self.gbr.gemm_split_tail(-1)
        return False


class thin_tail:
    """Sets the grouped CTA-pair launches' thin tail tiles on or off for the
    duration of a with-block, then restores the default (on)."""

    def __init__(self, gbr, on):
        self.gbr, self.on = gbr, on

    def __enter__(self):
        self.gbr.gemm_thin_tail(self.on)
        return self

    def __exit__(self, *exc):
        self.gbr.gemm_thin_tail(True)
        return False


class ffma_warps:
    """Selects the FFMA kernels' consumer layout (8 warps of 8x8, the default,
    or 16 warps of 8x4) for the duration of a with-block, then restores the
    default."""

    def __init__(self, gbr, warps):
        self.gbr, self.warps = gbr, warps

    def __enter__(self):
        self.gbr.ffma_tuning(self.warps)
        return self

    def __exit__(self, *exc):
        self.gbr.ffma_tuning(-1)
        return False
