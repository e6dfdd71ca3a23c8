"""The C ABI used from a plain C program (no Python in the call path): the
program allocates its own device buffers and calls gemm_bias_relu (FFMA and
bf16), staged_copy and gbr_device_status; its outputs are then checked
against the oracle here."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import TOL, load_library, rel_frobenius, require_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_calls_the_abi(tmp_path):
    require_gpu()
    gbr = load_library()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.dirname(gbr.library_path())
    exe = str(tmp_path / "c_abi_example")
    res = subprocess.run([cc, "-std=c99", "-O2", "-I" + os.path.join(ROOT, "include"),
                          "-I" + os.path.join(cuda, "include"),
                          os.path.join(ROOT, "tests", "c_abi_example.c"), "-o", exe,
                          "-L" + libdir, "-lgbr", "-L" + os.path.join(cuda, "lib64"), "-lcudart",
                          "-Wl,-rpath," + libdir + ":" + os.path.join(cuda, "lib64")],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    out = str(tmp_path / "out.bin")
    res = subprocess.run([exe, out], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0 and res.stdout.strip() == "ok", res.stdout + res.stderr
    M, N, K = 300, 264, 200
    raw = np.fromfile(out, dtype=np.uint8)
    off = 0

    def take(n, dt):
        nonlocal off
        a = raw[off:off + n * np.dtype(dt).itemsize].view(dt)
        off += n * np.dtype(dt).itemsize
        return a

    A = take(M * K, np.float32).reshape(M, K)
    B = take(K * N, np.float32).reshape(K, N)
    bias = take(N, np.float32)
    C = take(M * N, np.float32).reshape(M, N)
    Cb = take(M * N, np.uint16).reshape(M, N)
    copy = take(M * K, np.float32).reshape(M, K)
    ref = oracle.gemm_bias_relu(A, B, bias)
    assert rel_frobenius(C, ref) <= TOL["ffma"]
    Ab = torch.from_numpy(A).to(torch.bfloat16).float().numpy()
    Bb = torch.from_numpy(B).to(torch.bfloat16).float().numpy()
    Cbf = (Cb.astype(np.uint32) << 16).view(np.float32)
    assert rel_frobenius(Cbf, oracle.gemm_bias_relu(Ab, Bb, bias)) <= TOL["bf16"]
    assert np.array_equal(copy.view(np.uint32), A.view(np.uint32))
