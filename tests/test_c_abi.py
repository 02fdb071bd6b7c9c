"""The C ABI from plain C: a program built against include/gemm.h and linked
with libgb300gemm.so runs the GEMM on cudaMalloc'd buffers; its output is
compared with the oracle.  The CPU test only checks that the program compiles
against the header."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from dense_gemm_engineering_gb300 import build, inputs
from gpu_util import check_close

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c_abi", "gemm_from_c.c")
CUDA = "/usr/local/cuda"


def _compile(out):
    cc = shutil.which("gcc") or "cc"
    cmd = [cc, "-std=c11", "-O1", "-Wall", "-Werror", "-I", build.INCLUDE,
           "-I", os.path.join(CUDA, "include"), SRC, "-o", out,
           "-L", build.BUILD, "-lgb300gemm", f"-Wl,-rpath,{build.BUILD}",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    return subprocess.run(cmd, capture_output=True, text=True)


def test_header_compiles_as_c(tmp_path):
    cc = shutil.which("gcc") or "cc"
    r = subprocess.run([cc, "-std=c11", "-fsyntax-only", "-Wall", "-Werror", "-I", build.INCLUDE,
                        "-I", os.path.join(CUDA, "include"), SRC], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
@pytest.mark.parametrize("layout,dtype,M,N,K", [("abt", "f16", 300, 520, 200),
                                                 ("ab", "bf16", 520, 384, 136)])
def test_gemm_from_plain_c(tmp_path, layout, dtype, M, N, K):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    exe = str(tmp_path / "gemm_from_c")
    r = _compile(exe)
    assert r.returncode == 0, r.stderr
    A, B = inputs.operands(M, N, K, layout, dtype, "uniform", 31)
    A.tofile(tmp_path / "A.bin")
    B.tofile(tmp_path / "B.bin")
    r = subprocess.run([exe, layout, dtype, str(M), str(N), str(K), str(tmp_path / "A.bin"),
                        str(tmp_path / "B.bin"), str(tmp_path / "D.bin")],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
    D = np.fromfile(tmp_path / "D.bin", dtype=np.uint16).reshape(M, N)
    ref = oracle.gemm(A, B, layout=layout, dtype=dtype)
    check_close(D, ref, dtype, "plain C caller")


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_gemm_from_plain_c(tmp_path, fmt):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    exe = str(tmp_path / "gemm_from_c")
    r = _compile(exe)
    assert r.returncode == 0, r.stderr
    M, N, K, alpha = 300, 520, 272, 0.75
    A, B = inputs.operands(M, N, K, "abt", fmt, "uniform", 32)
    A.tofile(tmp_path / "A.bin")
    B.tofile(tmp_path / "B.bin")
    r = subprocess.run([exe, "fp8", fmt, str(M), str(N), str(K), str(tmp_path / "A.bin"),
                        str(tmp_path / "B.bin"), str(tmp_path / "D.bin"), str(alpha)],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
    D = np.fromfile(tmp_path / "D.bin", dtype=np.uint16).reshape(M, N)
    ref = oracle.gemm_fp8(A, B, fmt=fmt, out_dtype="bf16", alpha=alpha)
    check_close(D, ref, "bf16", "plain C caller, FP8")


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_block_scaled_gemm_from_plain_c(tmp_path, fmt):
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    exe = str(tmp_path / "gemm_from_c")
    r = _compile(exe)
    assert r.returncode == 0, r.stderr
    M, N, K, alpha = 300, 520, 272, 0.75
    A, B, SA, SB = inputs.mx_operands(M, N, K, fmt, "uniform", 33)
    for name, x in (("A", A), ("B", B), ("SA", SA), ("SB", SB)):
        np.ascontiguousarray(x).tofile(tmp_path / f"{name}.bin")
    r = subprocess.run([exe, "mx", fmt, str(M), str(N), str(K), str(tmp_path / "A.bin"),
                        str(tmp_path / "B.bin"), str(tmp_path / "D.bin"), str(alpha),
                        str(tmp_path / "SA.bin"), str(tmp_path / "SB.bin")],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
    D = np.fromfile(tmp_path / "D.bin", dtype=np.uint16).reshape(M, N)
    ref = oracle.gemm_mx(A, B, SA, SB, fmt=fmt, out_dtype="bf16", alpha=alpha)
    check_close(D, ref, "bf16", "plain C caller, block-scaled FP8")
