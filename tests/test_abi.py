"""The C-ABI library builds for sm_103a, loads, and exports every function
declared in include/gbr.h; the binding declares each of them.  No GPU needed
(no compute call is made)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbr.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*?\*?\s*\b([a-z_][a-z0-9_]*)\s*\(",
                       text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


@pytest.fixture(scope="module")
def built():
    from mbarrier_gemm_pipelines_gb300 import _build
    return _build.build()


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("gemm_bias_relu", "gemm_bias_relu_grouped", "staged_copy",
                     "gbr_device_status", "gbr_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(built):
    lib = ctypes.CDLL(built)
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_covers_header(built):
    from mbarrier_gemm_pipelines_gb300 import _binding
    assert set(_declared()) == set(_binding.SIGNATURES)
    lib = _binding.lib()
    assert lib.gbr_last_error() == b""
    assert lib.gbr_launch_count() == 0


def test_oracle_and_product_do_not_import_each_other():
    pkg = os.path.join(ROOT, "mbarrier_gemm_pipelines_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", src, flags=re.M), f
                assert "liboracle" not in src and "oracle.c" not in src, f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            src = open(os.path.join(ROOT, "oracle", f)).read()
            assert "mbarrier_gemm_pipelines_gb300" not in src, f
            assert "gbr.h" not in src and "libgbr" not in src, f


def test_built_for_sm103a_only():
    from mbarrier_gemm_pipelines_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_product_fails_loudly_without_cuda(built):
    import torch
    import mbarrier_gemm_pipelines_gb300 as gbr
    A = torch.zeros(8, 8)
    with pytest.raises((ValueError, RuntimeError)):
        gbr.gemm_bias_relu(A, A, torch.zeros(8), dtype="ffma")
