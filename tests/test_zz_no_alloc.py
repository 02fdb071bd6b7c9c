"""gemm_run_no_alloc: the GEMM for callers that cannot allocate device memory.

Such callers (graph capture, fixed memory budgets, plugins whose host owns all
allocations) get the split tail's scratch from a fixed array inside the
library.  These checks call the entry point through the C ABI and compare its
output with the existing gemm_run_workspace path, within the tolerance every
parity test here uses, on two calls in a row.  This file is collected last so
that a run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from dense_gemm_engineering_gb300 import binding, build, inputs
from gpu_util import check_close, from_device, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.load()
    torch.cuda.set_device(0)


def _raw_no_alloc(A, B, D, layout, opts):
    """Direct C-ABI call (ctypes, integer addresses), returning the status."""
    lib = binding.load()
    o = binding.GemmOptions(**opts)
    M, K = A.shape
    N = D.shape[1]
    return lib.gemm_run_no_alloc(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                 A.stride(0), B.stride(0), D.stride(0),
                                 0 if A.dtype == torch.float16 else 1, layout,
                                 ctypes.pointer(o), torch.cuda.current_stream().cuda_stream)


CASES = [
    # M, N, K, layout, dtype, options (split tail active: tiles mod clusters > 0)
    (1024, 1024, 2048, 0, "f16", {"cta_group": 2, "max_clusters": 7, "tail_split": 3}),
    (768, 1280, 1000, 1, "bf16", {"cta_group": 2, "max_clusters": 7, "tail_split": 4}),
    (4096, 4096, 4096, 0, "f16", {"tail_split": 2}),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}_{c[4]}")
def test_no_alloc_matches_workspace_path_twice(case):
    M, N, K, layout, dtype, opts = case
    lay = "abt" if layout == 0 else "ab"
    A, B = inputs.operands(M, N, K, lay, dtype, "uniform" if dtype == "f16" else "normal", 123)
    dA, dB = to_device(A, dtype), to_device(B, dtype)
    tdt = dA.dtype
    ref = binding.gemm_run(dA, dB, layout=layout, options=opts or None)  # existing entry point
    torch.cuda.synchronize()
    ref_bits = from_device(ref)
    for _ in range(2):  # two calls in a row share (and reuse) the scratch
        D = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        assert _raw_no_alloc(dA, dB, D, layout, opts) == 0
        torch.cuda.synchronize()
        check_close(from_device(D), ref_bits, dtype, "gemm_run_no_alloc vs gemm_run_workspace")
    assert binding.gemm_device_status(clear=True) == 0


def test_no_alloc_split_tail_in_a_cuda_graph():
    # A captured launch replays with the same epoch for its split-tail
    # counters; the range that finishes a tile resets its counter, so every
    # replay writes the whole of D again.
    M, N, K, opts = 1024, 1024, 2048, {"cta_group": 2, "max_clusters": 7, "tail_split": 3}
    A, B = inputs.operands(M, N, K, "abt", "f16", "uniform", 124)
    dA, dB = to_device(A, "f16"), to_device(B, "f16")
    ref_bits = from_device(binding.gemm_run(dA, dB, layout=0, options=opts))
    D = torch.empty((M, N), dtype=torch.float16, device="cuda")
    assert _raw_no_alloc(dA, dB, D, 0, opts) == 0  # plan cached outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        status = _raw_no_alloc(dA, dB, D, 0, opts)
    assert status == 0
    for i in range(3):
        D.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        check_close(from_device(D), ref_bits, "f16", f"graph replay {i}")
    assert binding.gemm_device_status(clear=True) == 0


def test_no_alloc_rejects_plans_beyond_its_scratch():
    # 4096^3 in 256-wide tiles on 76 clusters leaves 28 tail tiles; a forced
    # 16-way split would need 28 x 16 x 256 KiB = 112 MiB of scratch, beyond the
    # fixed 20 MiB.
    opts = {"cta_group": 2, "block_n": 256, "tail_split": 16}
    need = binding.gemm_workspace_size(4096, 4096, 4096, 0, 0, opts)
    if need <= 20 << 20:
        pytest.skip("this GPU's plan fits in the scratch")
    A = torch.zeros((4096, 4096), dtype=torch.float16, device="cuda")
    D = torch.zeros((4096, 4096), dtype=torch.float16, device="cuda")
    assert _raw_no_alloc(A, A, D, 0, opts) == -10
    assert binding.gemm_status_string(-10)
