"""gemm_run_no_alloc: the GEMM for callers that cannot allocate device memory.

Some callers may not call cudaMalloc where they run a GEMM: a plugin whose
host framework owns every byte of device memory, a latency-critical loop in
which an allocation can synchronise the device, a process with a device
budget fixed at start-up.  For them the split tail's scratch is a fixed
array inside the library.  These checks call that entry point through the C
ABI, on plans that really use the scratch, and compare its output with the
existing entry point's (gemm_run_workspace with a caller-owned workspace) and
with the CPU oracle, within the tolerance every parity test here uses, on two
calls in a row.  This file is collected last so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import oracle
from dense_gemm_engineering_gb300 import binding, build, inputs
from gpu_util import check_close, from_device, to_device

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 20 << 20


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
    # M, N, K, layout, dtype, options: each plan has a split tail (tiles mod
    # clusters > 0 and tail_split >= 2), so the scratch is in use
    (1024, 1024, 2048, 0, "f16", {"cta_group": 2, "max_clusters": 7, "tail_split": 3}),
    (768, 1280, 1000, 1, "bf16", {"cta_group": 2, "max_clusters": 7, "tail_split": 4}),
    # 256 tiles of 256 x 256 on 76 clusters: 28 tail tiles in 2 K-ranges each
    (4096, 4096, 4096, 0, "f16", {"cta_group": 2, "block_n": 256, "tail_split": 2}),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}_{c[4]}")
def test_no_alloc_matches_existing_entry_point_and_oracle_twice(case):
    M, N, K, layout, dtype, opts = case
    dt = 0 if dtype == "f16" else 1
    need = binding.gemm_workspace_size(M, N, K, dt, layout, opts)
    assert 0 < need <= SCRATCH_BYTES, need
    plan = binding.gemm_plan(M, N, K, dt, layout, opts)
    assert plan["tail_split"] >= 2 and plan["num_tiles"] % plan["num_clusters"] != 0
    lay = "abt" if layout == 0 else "ab"
    A, B = inputs.operands(M, N, K, lay, dtype, "uniform" if dtype == "f16" else "normal", 123)
    dA, dB = to_device(A, dtype), to_device(B, dtype)
    tdt = dA.dtype
    # the existing entry point, with a caller-owned (zeroed) workspace
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    existing = binding.gemm_run(dA, dB, layout=layout, options=opts, workspace=ws)
    torch.cuda.synchronize()
    existing_bits = from_device(existing)
    ref = oracle.gemm(A, B, layout=lay, dtype=dtype)
    check_close(existing_bits, ref, dtype, "gemm_run_workspace vs oracle")
    for i in range(2):  # two calls in a row share (and reuse) the scratch
        D = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        assert _raw_no_alloc(dA, dB, D, layout, opts) == 0
        torch.cuda.synchronize()
        got = from_device(D)
        check_close(got, existing_bits, dtype, f"call {i}: gemm_run_no_alloc vs gemm_run_workspace")
        check_close(got, ref, dtype, f"call {i}: gemm_run_no_alloc vs oracle")
    assert binding.gemm_device_status(clear=True) == 0


def test_no_alloc_rejects_plans_beyond_its_scratch():
    # 4096^3 in 256-wide tiles on 76 clusters leaves 28 tail tiles; a forced
    # 16-way split would need 28 x 16 x 256 KiB = 112 MiB of scratch, beyond the
    # fixed 20 MiB.
    opts = {"cta_group": 2, "block_n": 256, "tail_split": 16}
    need = binding.gemm_workspace_size(4096, 4096, 4096, 0, 0, opts)
    if need <= SCRATCH_BYTES:
        pytest.skip("this GPU's plan fits in the scratch")
    A = torch.zeros((4096, 4096), dtype=torch.float16, device="cuda")
    D = torch.zeros((4096, 4096), dtype=torch.float16, device="cuda")
    assert _raw_no_alloc(A, A, D, 0, opts) == -10
    assert binding.gemm_status_string(-10)
