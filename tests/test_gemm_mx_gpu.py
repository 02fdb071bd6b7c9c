"""GPU parity of the block-scaled FP8 (MX) A.Bt GEMM against the CPU oracle.

D[i,j] = round(alpha * sum_k (A[i,k] 2^(SA[i][k/32]-127)) (B[j,k] 2^(SB[j][k/32]-127)))
with FP8 A (M x K) and B (N x K), one UE8M0 scale per 32 K elements of each
row, FP32 accumulation and a 16-bit D.  The scales reach the GEMM in the
layouts written by gemm_mx_pack_scales (A) and gemm_mx_pack_scales_b (B), whose
outputs are checked byte for byte against the layouts' definitions.  Exact cases are compared bit for bit; the
rest within the output type's tolerance (|got - ref| <= 1e-2 + rtol |ref|:
every scaled product is exact in FP32, so only the FP32 accumulation and the
one rounding to the output type separate the two sides).
"""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_engineering_gb300 import binding, build, inputs
from gpu_util import check_close, decode, from_device, sample_tiles

pytestmark = pytest.mark.gpu

FORMATS = ["e4m3", "e5m2"]
OUTS = ["bf16", "f16"]
TDT = {"bf16": torch.bfloat16, "f16": torch.float16}


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


def tiled_scales(S: np.ndarray, K: int) -> np.ndarray:
    """The tiled scale layout, from its definition: atom (rb, kc) of 512 bytes
    at (rb * ceil(K/128) + kc) * 512; row rb*128 + r, group kc*4 + g at byte
    (r % 32) * 16 + (r / 32) * 4 + g; 127 past the last row or group."""
    rows, groups = S.shape
    rb_n, kc_n = -(-rows // 128), -(-K // 128)
    full = np.full((rb_n * 128, kc_n * 4), 127, dtype=np.uint8)
    full[:rows, :groups] = S
    out = np.empty(rb_n * kc_n * 512, dtype=np.uint8)
    for rb in range(rb_n):
        for kc in range(kc_n):
            blk = full[rb * 128:(rb + 1) * 128, kc * 4:(kc + 1) * 4]  # (r, g)
            atom = blk.reshape(4, 32, 4).transpose(1, 0, 2)           # (r % 32, r / 32, g)
            o = (rb * kc_n + kc) * 512
            out[o:o + 512] = atom.reshape(-1)
    return out


def tiled_scales_b(S: np.ndarray, K: int) -> np.ndarray:
    """The B-scale layout, from its definition: block (t, kc) of 4096 bytes at
    (t * ceil(K/128) + kc) * 4096; column 224 t + 32 c + l (c < 7), group
    kc*4 + g at byte (r/8)*256 + (r%8)*16 + (c/4)*128 + (c%4)*4 + g for
    r = l, l+32, l+64, l+96; 127 elsewhere."""
    N, groups = S.shape
    t_n, kc_n = -(-N // 224), -(-K // 128)
    full = np.full((t_n * 224 + 32, kc_n * 4), 127, dtype=np.uint8)
    full[:N, :groups] = S
    out = np.full(t_n * kc_n * 4096, 127, dtype=np.uint8)
    r = np.arange(128)
    for t in range(t_n):
        for kc in range(kc_n):
            o = (t * kc_n + kc) * 4096
            for c in range(7):
                for g in range(4):
                    byte = (r // 8) * 256 + (r % 8) * 16 + (c // 4) * 128 + (c % 4) * 4 + g
                    out[o + byte] = full[t * 224 + 32 * c + r % 32, kc * 4 + g]
    return out


def pack(S: np.ndarray, K: int) -> torch.Tensor:
    return binding.mx_pack_scales(to_dev8(S), K)


def pack_b(S: np.ndarray, K: int) -> torch.Tensor:
    return binding.mx_pack_scales_b(to_dev8(S), K)


def run_mx(A, B, SA, SB, K, fmt, out, alpha=1.0, options=None, D=None):
    D = binding.gemm_mx(to_dev8(A), to_dev8(B), pack(SA, K), pack_b(SB, K), D, fmt=fmt,
                        out_dtype=TDT[out], alpha=alpha, options=options)
    torch.cuda.synchronize()
    return D


def parity_mx(M, N, K, fmt, out, dist="uniform", seed=0, alpha=1.0, options=None, lo=124,
              hi=130):
    # FP8 rows are byte arrays: TMA needs row strides that are multiples of 16
    # bytes, so a ragged K gets padded rows (the padding holds NaN).
    ld16 = -(-K // 16) * 16
    A, B, SA, SB = inputs.mx_operands(M, N, K, fmt, dist, seed, lda=ld16, ldb=ld16, lo=lo, hi=hi)
    got = from_device(run_mx(A, B, SA, SB, K, fmt, out, alpha, options))
    ref, ref64 = oracle.gemm_mx(A, B, SA, SB, fmt=fmt, out_dtype=out, alpha=alpha, want_f64=True)
    return check_close(got, ref, out, f"mx {M}x{N}x{K} {fmt}->{out} {options}", ref64)


@pytest.mark.parametrize("shape", [(1, 32), (128, 128), (300, 1000), (129, 4096), (5, 33),
                                   (700, 200)], ids=lambda s: f"{s[0]}x{s[1]}")
def test_pack_layout_byte_exact(shape):
    rows, K = shape
    groups = -(-K // 32)
    S = inputs.mx_scales(rows, 2, rows, K, lo=0, hi=254, ld=groups + 3)  # padded rows (255)
    got = pack(S, K).cpu().numpy()[:binding.mx_scales_size(rows, K)]
    assert np.array_equal(got, tiled_scales(S, K))
    got_b = pack_b(S, K).cpu().numpy()[:binding.mx_scales_b_size(rows, K)]
    assert np.array_equal(got_b, tiled_scales_b(S, K))


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("out", OUTS)
def test_exact_small_integers(fmt, out):
    # |A|, |B| <= 2 and scales 2^-2 .. 2^2: every partial sum is a multiple of
    # 2^-4 below 2^12, exact in FP32; one rounding to the output on each side.
    rng = np.random.default_rng(3)
    for (M, N, K) in [(256, 224, 64), (384, 520, 160), (200, 904, 256)]:
        a = rng.integers(-2, 3, size=(M, K)).astype(np.float32)
        b = rng.integers(-2, 3, size=(N, K)).astype(np.float32)
        A, B = inputs.f32_to_fp8_bits(a, fmt), inputs.f32_to_fp8_bits(b, fmt)
        g = -(-K // 32)
        SA = rng.integers(125, 130, size=(M, g)).astype(np.uint8)
        SB = rng.integers(125, 130, size=(N, g)).astype(np.uint8)
        got = from_device(run_mx(A, B, SA, SB, K, fmt, out))
        ref = oracle.gemm_mx(A, B, SA, SB, fmt=fmt, out_dtype=out)
        assert np.array_equal(got, ref), f"{M}x{N}x{K} {fmt}->{out}"


SHAPES = [(256, 224, 128), (300, 520, 136), (1000, 1104, 1000), (129, 264, 4000), (1, 16, 16),
          (777, 32, 2048), (512, 1000, 384), (256, 896, 512)]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("fmt", FORMATS)
def test_shapes(shape, fmt):
    M, N, K = shape
    parity_mx(M, N, K, fmt, "bf16", seed=M + N + K)


@pytest.mark.parametrize("options", [{"max_clusters": 3}, {"max_clusters": 1},
                                     {"raster_group": 1}, {"raster_group": 5, "max_clusters": 7}],
                         ids=["c3", "c1", "g1", "g5c7"])
def test_schedules(options):
    # Many rounds per cluster: every ring stage, phase and TMEM buffer (for the
    # accumulators and for the scales) is reused with different tiles.
    parity_mx(1000, 1600, 1152, "e4m3", "bf16", seed=11, options=options)


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("out", OUTS)
def test_alpha_scales_the_fp32_sum(fmt, out):
    for alpha in (0.0625, 0.37, 3.0):
        parity_mx(500, 704, 1024, fmt, out, dist="normal", seed=21, alpha=alpha)


def test_wide_scale_range():
    # Scales 2^-27 .. 2^27 per group: the groups of one dot product differ by
    # up to 2^108, so a scale applied to the wrong group shows at once.  With
    # such a range the sum cancels heavily, and FP32 accumulation can only be
    # held to a fraction of the sum of |terms| (computed by the oracle on
    # |A| and |B|): the bound adds 2^-16 of it to the output tolerance, far
    # below the size of any misplaced group's contribution.
    M, N, K = 512, 672, 1024
    A, B, SA, SB = inputs.mx_operands(M, N, K, "e4m3", "normal", 23, lo=100, hi=154)
    got = decode(from_device(run_mx(A, B, SA, SB, K, "e4m3", "bf16")), "bf16")
    ref, ref64 = oracle.gemm_mx(A, B, SA, SB, fmt="e4m3", out_dtype="bf16", want_f64=True)
    _, mag = oracle.gemm_mx(A & np.uint8(0x7F), B & np.uint8(0x7F), SA, SB, fmt="e4m3",
                            out_dtype="bf16", want_f64=True)
    err = np.abs(got - ref64)
    assert (err <= 1e-2 + 8e-3 * np.abs(ref64) + 2.0 ** -16 * mag).all()
    plain = err <= 1e-2 + 8e-3 * np.abs(decode(ref, "bf16"))
    assert plain.mean() > 0.999


def test_square_4096_full():
    parity_mx(4096, 4096, 4096, "e4m3", "bf16", seed=2)


def test_large_sampled_tiles():
    # 8192 x 8192 x 8192 E4M3 (the benchmark shape): a seeded cover of the
    # persistent schedule's positions (cluster, round, ring stage, phase, TMEM
    # buffer) plus the edge tiles, each checked against the oracle.
    M = N = K = 8192
    A, B, SA, SB = inputs.mx_operands(M, N, K, "e4m3", "normal", 7)
    D = from_device(run_mx(A, B, SA, SB, K, "e4m3", "bf16", alpha=0.5))
    plan = binding.gemm_mx_plan(M, N, K, binding.GEMM_E4M3)
    g, o = plan["raster_group"], plan["raster_order"]
    tiles = sample_tiles(M, N, K, plan["block_m"], plan["block_n"], g, plan["num_clusters"],
                         plan["stages"],
                         lambda t: binding.gemm_tile_origin(M, N, plan["block_m"],
                                                            plan["block_n"], g, t, o),
                         seed=3, extra_random=8, block_k=128)
    for (m0, n0) in tiles:
        m1, n1 = min(m0 + plan["block_m"], M), min(n0 + plan["block_n"], N)
        ref, ref64 = oracle.gemm_mx(A, B, SA, SB, fmt="e4m3", out_dtype="bf16", alpha=0.5,
                                    rows=(m0, m1), cols=(n0, n1), want_f64=True)
        check_close(D[m0:m1, n0:n1], ref, "bf16", f"tile ({m0},{n0})", ref64)


@pytest.mark.parametrize("shape", [(8192, 4096, 14336), (8192, 14336, 4096)],
                         ids=["narrowing_8192x4096x14336", "widening_8192x14336x4096"])
def test_mlp_shapes_sampled_tiles(shape):
    # M = 8192 against MLP-like weights: a seeded cover of the schedule's
    # positions plus the edge tiles (N = 4096 ends in a partial 224-wide tile).
    M, N, K = shape
    A, B, SA, SB = inputs.mx_operands(M, N, K, "e4m3", "normal", 8)
    D = from_device(run_mx(A, B, SA, SB, K, "e4m3", "bf16"))
    plan = binding.gemm_mx_plan(M, N, K, binding.GEMM_E4M3)
    g, o = plan["raster_group"], plan["raster_order"]
    tiles = sample_tiles(M, N, K, plan["block_m"], plan["block_n"], g, plan["num_clusters"],
                         plan["stages"],
                         lambda t: binding.gemm_tile_origin(M, N, plan["block_m"],
                                                            plan["block_n"], g, t, o),
                         seed=4, extra_random=4, block_k=128)
    for (m0, n0) in tiles:
        m1, n1 = min(m0 + plan["block_m"], M), min(n0 + plan["block_n"], N)
        ref, ref64 = oracle.gemm_mx(A, B, SA, SB, fmt="e4m3", out_dtype="bf16",
                                    rows=(m0, m1), cols=(n0, n1), want_f64=True)
        check_close(D[m0:m1, n0:n1], ref, "bf16", f"tile ({m0},{n0})", ref64)


def test_plan():
    plan = binding.gemm_mx_plan(4096, 4096, 4096, binding.GEMM_E4M3)
    assert (plan["cta_group"], plan["block_m"], plan["block_n"]) == (2, 256, 224)
    assert plan["num_tiles"] == 16 * 19
    assert 1 <= plan["num_clusters"] <= 76 and plan["stages"] >= 4


def test_nan_scale_poisons_its_row():
    # UE8M0 255 is NaN (OCP Microscaling): row 5's group 3 poisons row 5 only.
    M, N, K = 256, 224, 256
    A, B, SA, SB = inputs.mx_operands(M, N, K, "e4m3", "uniform", 31)
    SA = SA.copy()
    SA[5, 3] = 255
    got = run_mx(A, B, SA, SB, K, "e4m3", "bf16").float().cpu().numpy()
    assert np.isnan(got[5]).all()
    assert not np.isnan(np.delete(got, 5, axis=0)).any()


def test_strided_operands_and_guarded_output():
    # Row strides above the row length (padding is NaN in FP8, 255 = NaN in
    # the row-major scales); D is a view in a larger buffer filled with a
    # sentinel that must survive.
    M, N, K = 300, 200, 160
    A, B, SA, SB = inputs.mx_operands(M, N, K, "e5m2", "uniform", 9, lda=K + 32, ldb=K + 16)
    SA = inputs.mx_scales(9, 2, M, K, ld=9)
    sentinel = 0x5A5A
    ldd = N + 40
    buf = torch.full((M + 3, ldd), sentinel, dtype=torch.int16, device="cuda")
    D = buf.view(torch.bfloat16)[1:M + 1, 8:8 + N]
    run_mx(A, B, SA, SB, K, "e5m2", "bf16", D=D)
    host = buf.cpu().numpy().view(np.uint16)
    inside = np.zeros_like(host, dtype=bool)
    inside[1:M + 1, 8:8 + N] = True
    assert (host[~inside] == sentinel).all()
    ref = oracle.gemm_mx(A, B, SA, SB, fmt="e5m2", out_dtype="bf16")
    check_close(host[1:M + 1, 8:8 + N], ref, "bf16", "strided")


def test_k_zero_writes_zeros():
    A = torch.empty((40, 0), dtype=torch.uint8, device="cuda")
    B = torch.empty((48, 0), dtype=torch.uint8, device="cuda")
    S = torch.zeros(16, dtype=torch.uint8, device="cuda")
    D = torch.full((40, 48), 7.0, dtype=torch.bfloat16, device="cuda")  # K = 0: no scales read
    binding.gemm_mx(A, B, S, S, D, fmt="e4m3")
    torch.cuda.synchronize()
    assert (D == 0).all()


def test_torch_float8_tensors_are_accepted():
    M, N, K = 256, 448, 512
    A, B, SA, SB = inputs.mx_operands(M, N, K, "e4m3", "uniform", 41)
    dA = to_dev8(A).view(torch.float8_e4m3fn)
    dB = to_dev8(B).view(torch.float8_e4m3fn)
    got = from_device(binding.gemm_mx(dA, dB, pack(SA, K), pack_b(SB, K)))
    torch.cuda.synchronize()
    ref = oracle.gemm_mx(A, B, SA, SB, fmt="e4m3", out_dtype="bf16")
    check_close(got, ref, "bf16", "float8 tensors")


def test_option_limits():
    A = torch.zeros((256, 128), dtype=torch.uint8, device="cuda")
    S = torch.full((binding.mx_scales_b_size(256, 128),), 127, dtype=torch.uint8, device="cuda")
    for bad in ({"cta_group": 1}, {"block_n": 256}, {"block_n": 192}, {"consumers": 2},
                {"multicast": 2}, {"tail_split": 2}):
        with pytest.raises(binding.GemmError) as e:
            binding.gemm_mx(A, A, S, S, fmt="e4m3", options=bad)
        assert e.value.status == -8, bad


def test_scale_argument_errors():
    lib = binding.load()
    M, N, K = 256, 224, 128
    A = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    B = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    # One buffer large enough for the scales and for D at any offset used below,
    # so that no check under test can cause an access outside an allocation.
    big = torch.full((1 << 20,), 127, dtype=torch.uint8, device="cuda")
    S = big.data_ptr()
    call = lambda sa, sb, d=D.data_ptr(): lib.gemm_mx_run(
        A.data_ptr(), B.data_ptr(), sa, sb, d, M, N, K, K, K, N, binding.GEMM_E4M3,
        binding.GEMM_BF16, 1.0, None, None)
    assert call(None, S) == -1
    assert call(S, None) == -1
    assert call(S + 4, S) == -4
    assert call(S, S + 8) == -4
    assert call(S, S + 16384, S + 256) == -5     # D over the scales of A
    assert call(S + 16384, S, S + 512) == -5     # D over the scales of B (8 KiB)
    assert lib.gemm_mx_run(A.data_ptr(), B.data_ptr(), S, S, D.data_ptr(), M, N, K, K, K, N,
                           binding.GEMM_BF16, binding.GEMM_BF16, 1.0, None, None) == -2
    torch.cuda.synchronize()


def test_cuda_graph_capture_and_replay():
    M, N, K = 512, 672, 1024
    A, B, SA, SB = inputs.mx_operands(M, N, K, "e4m3", "uniform", 53)
    dA, dB, dSA, dSB = to_dev8(A), to_dev8(B), pack(SA, K), pack_b(SB, K)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    binding.gemm_mx(dA, dB, dSA, dSB, D, fmt="e4m3")  # plan cached outside the capture
    torch.cuda.synchronize()
    D.fill_(7.0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.gemm_mx(dA, dB, dSA, dSB, D, fmt="e4m3")
    g.replay()
    torch.cuda.synchronize()
    ref = oracle.gemm_mx(A, B, SA, SB, fmt="e4m3", out_dtype="bf16")
    check_close(from_device(D), ref, "bf16", "graph replay")
