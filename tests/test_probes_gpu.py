"""Measurement probes that back statements about the kernel: each builds with
nvcc for sm_103a and runs to completion on the GPU (their counters are read
with ncu; see the probe's header)."""
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_smem_store_conflict_probe_runs(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = str(tmp_path / "smem_store_conflicts")
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-o", exe,
                    os.path.join(HERE, "probes", "smem_store_conflicts.cu")], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "status no error, copy waits that ran out: 0" in r.stdout


def test_cluster_exchange_probe_runs(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    exe = str(tmp_path / "cluster_exchange")
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-o", exe,
                    os.path.join(HERE, "probes", "cluster_exchange.cu")], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "waits that ran out / sink: 0" in r.stdout
    # every mode of every cluster size reported a time
    assert r.stdout.count(" per exchange;") == 11, r.stdout
