"""GPU parity of the FP8 (E4M3 / E5M2) A.Bt GEMM against the CPU oracle.

D = round(alpha * A . Bt) with FP8 A (M x K) and B (N x K), FP32 accumulation
and a 16-bit D.  Exact small-integer cases are compared bit for bit; the rest
within the output type's tolerance (|got - ref| <= 1e-2 + rtol |ref|, the same
bound as the 16-bit GEMM: FP32 accumulation of exact FP8 products, then one
rounding to the output type).
"""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_engineering_gb300 import binding, build, inputs
from gpu_util import check_close, from_device, sample_tiles

pytestmark = pytest.mark.gpu

FORMATS = ["e4m3", "e5m2"]
OUTS = ["bf16", "f16"]
TDT = {"bf16": torch.bfloat16, "f16": torch.float16}
VARIANTS = [{}, {"cta_group": 2, "block_n": 256}, {"cta_group": 2, "block_n": 224},
            {"cta_group": 1, "block_n": 256}]
VID = ["auto", "cg2_n256", "cg2_n224", "cg1_n256"]


@pytest.fixture(scope="module", autouse=True)
def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.load()
    torch.cuda.set_device(0)
    yield
    assert binding.gemm_device_status(clear=True) == 0


def to_dev8(bits: np.ndarray) -> torch.Tensor:
    """uint8 patterns (2-D, unit inner stride, padded rows kept) -> device view."""
    rows, cols = bits.shape
    ld = bits.strides[0] if rows > 1 else cols
    base = np.lib.stride_tricks.as_strided(bits, shape=(rows, ld), strides=(ld, 1)) \
        if ld != cols else bits
    return torch.from_numpy(np.ascontiguousarray(base)).cuda()[:, :cols]


def run8(A, B, fmt, out, alpha=1.0, options=None, D=None):
    dA, dB = to_dev8(A), to_dev8(B)
    D = binding.gemm_fp8(dA, dB, D, fmt=fmt, out_dtype=TDT[out], alpha=alpha, options=options)
    torch.cuda.synchronize()
    return D


def parity8(M, N, K, fmt, out, dist="uniform", seed=0, alpha=1.0, options=None, lda=None,
            ldb=None):
    # FP8 rows are byte arrays: TMA needs row strides that are multiples of 16
    # bytes, so a ragged K gets padded rows (the padding holds NaN).
    ld16 = -(-K // 16) * 16
    A, B = inputs.operands(M, N, K, "abt", fmt, dist, seed, lda=lda or ld16, ldb=ldb or ld16)
    got = from_device(run8(A, B, fmt, out, alpha, options))
    ref, ref64 = oracle.gemm_fp8(A, B, fmt=fmt, out_dtype=out, alpha=alpha, want_f64=True)
    return check_close(got, ref, out, f"fp8 {M}x{N}x{K} {fmt}->{out} {options}", ref64)


def small_int8(M, N, K, fmt, seed):
    rng = np.random.default_rng(seed)
    a = rng.integers(-2, 3, size=(M, K)).astype(np.float32)
    b = rng.integers(-2, 3, size=(N, K)).astype(np.float32)
    return inputs.f32_to_fp8_bits(a, fmt), inputs.f32_to_fp8_bits(b, fmt)


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("out", OUTS)
def test_exact_small_integers(variant, fmt, out):
    # |D| <= 4 * 64 = 256: exact in FP32 and in both output types.
    for (M, N, K) in [(128, 128, 64), (384, 520, 64)]:
        A, B = small_int8(M, N, K, fmt, M + K)
        got = from_device(run8(A, B, fmt, out, options=variant or None))
        ref = oracle.gemm_fp8(A, B, fmt=fmt, out_dtype=out)
        assert np.array_equal(got, ref), f"{M}x{N}x{K} {fmt}->{out} {variant}"


SHAPES = [(128, 128, 128), (256, 256, 1024), (300, 520, 136), (1000, 1104, 1000),
          (129, 264, 4000), (1, 16, 16), (777, 32, 2048)]


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("fmt", FORMATS)
def test_shapes(variant, shape, fmt):
    M, N, K = shape
    parity8(M, N, K, fmt, "bf16", seed=M + N + K, options=variant or None)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("out", OUTS)
def test_alpha_scales_the_fp32_sum(fmt, out):
    for alpha in (0.0625, 0.37, 3.0):
        parity8(500, 704, 1024, fmt, out, dist="normal", seed=21, alpha=alpha)


def test_square_4096_full():
    parity8(4096, 4096, 4096, "e4m3", "bf16", seed=2)


def test_large_sampled_tiles():
    # 8192 x 8192 x 4096 E4M3: compare a seeded cover of the persistent
    # schedule's positions (cluster, round, ring stage, phase, TMEM buffer).
    M, N, K = 8192, 8192, 4096
    A, B = inputs.operands(M, N, K, "abt", "e4m3", "normal", 7)
    D = from_device(run8(A, B, "e4m3", "bf16", alpha=0.5))
    plan = binding.gemm_plan(M, N, K, binding.GEMM_E4M3, binding.LAYOUT_ABT)
    g, o = plan["raster_group"], plan["raster_order"]
    tiles = sample_tiles(M, N, K, plan["block_m"], plan["block_n"], g,
                         plan["num_clusters"], plan["stages"],
                         lambda t: binding.gemm_tile_origin(M, N, plan["block_m"], plan["block_n"],
                                                            g, t, o), seed=3, block_k=128)
    for (m0, n0) in tiles:
        m1, n1 = min(m0 + plan["block_m"], M), min(n0 + plan["block_n"], N)
        ref, ref64 = oracle.gemm_fp8(A, B, fmt="e4m3", out_dtype="bf16", alpha=0.5,
                                     rows=(m0, m1), cols=(n0, n1), want_f64=True)
        check_close(D[m0:m1, n0:n1], ref, "bf16", f"tile ({m0},{n0})", ref64)


@pytest.mark.parametrize("split", [2, 3])
def test_split_tail(split):
    # 10 tiles on 4 clusters: 2 whole rounds, the last 2 tiles split along K.
    opts = {"cta_group": 2, "block_n": 256, "max_clusters": 4, "tail_split": split}
    parity8(1280, 512, 2048, "e4m3", "bf16", seed=split, options=opts)
    plan = binding.gemm_plan(1280, 512, 2048, binding.GEMM_E4M3, binding.LAYOUT_ABT, opts)
    assert plan["tail_split"] == split


def test_strided_operands_and_guarded_output():
    # Row strides above the row length (padding is NaN in FP8); D is a view in
    # a larger buffer filled with a sentinel that must survive.
    M, N, K = 300, 200, 160
    A, B = inputs.operands(M, N, K, "abt", "e5m2", "uniform", 9, lda=K + 32, ldb=K + 16)
    sentinel = 0x5A5A
    ldd = N + 40
    buf = torch.full((M + 3, ldd), sentinel, dtype=torch.int16, device="cuda")
    D = buf.view(torch.bfloat16)[1:M + 1, 8:8 + N]
    run8(A, B, "e5m2", "bf16", D=D)
    host = buf.cpu().numpy().view(np.uint16)
    inside = np.zeros_like(host, dtype=bool)
    inside[1:M + 1, 8:8 + N] = True
    assert (host[~inside] == sentinel).all()
    ref = oracle.gemm_fp8(A, B, fmt="e5m2", out_dtype="bf16")
    check_close(host[1:M + 1, 8:8 + N], ref, "bf16", "strided")


def test_k_zero_writes_zeros():
    A = torch.empty((40, 0), dtype=torch.uint8, device="cuda")
    B = torch.empty((48, 0), dtype=torch.uint8, device="cuda")
    D = torch.full((40, 48), 7.0, dtype=torch.bfloat16, device="cuda")
    binding.gemm_fp8(A, B, D, fmt="e4m3")
    torch.cuda.synchronize()
    assert (D == 0).all()


def test_torch_float8_tensors_are_accepted():
    A, B = inputs.operands(256, 384, 512, "abt", "e4m3", "uniform", 11)
    dA = to_dev8(A).view(torch.float8_e4m3fn)
    dB = to_dev8(B).view(torch.float8_e4m3fn)
    got = from_device(binding.gemm_fp8(dA, dB))
    torch.cuda.synchronize()
    ref = oracle.gemm_fp8(A, B, fmt="e4m3", out_dtype="bf16")
    check_close(got, ref, "bf16", "float8 tensors")


def test_option_limits():
    A = torch.zeros((256, 128), dtype=torch.uint8, device="cuda")
    for bad in ({"consumers": 2}, {"multicast": 2}, {"block_n": 192}, {"block_n": 128},
                {"cta_group": 1, "block_n": 224}):
        with pytest.raises(binding.GemmError) as e:
            binding.gemm_fp8(A, A, fmt="e4m3", options=bad)
        assert e.value.status == -8, bad
