"""GPU parity: the sm_103a kernel through the C ABI against the CPU oracle.

Every case draws seeded inputs, runs the CUDA path (binding -> libgb300gemm.so)
and compares element by element with the oracle on the same 16-bit inputs,
within |got - ref| <= 1e-2 + rtol * |ref| (rtol 1e-3 for FP16 output, 8e-3 for
BF16 output).  Small-integer cases, whose FP32 sums are exact, must match the
oracle bit for bit.  The five workloads are checked at full size in the launch
configuration the benchmark uses: in full where the oracle takes seconds, and
on seeded whole-tile samples (every scheduler position and ring stage/phase at
tile start) for the 8192 x 17408 x 5120 shape.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_engineering_gb300 import binding, build, configs, inputs
from gpu_util import (TORCH_DTYPE, check_close, check_strict, decode, from_device,
                      oracle_with_bound, sample_tiles, to_device)

pytestmark = pytest.mark.gpu

VARIANTS = [
    {"cta_group": 2, "block_n": 256, "raster_group": 0, "max_clusters": 0, "tail_split": 0},
    {"cta_group": 1, "block_n": 256, "raster_group": 0, "max_clusters": 0, "tail_split": 0},
    {"cta_group": 2, "block_n": 128, "raster_group": 0, "max_clusters": 0, "tail_split": 0},
    {"cta_group": 1, "block_n": 128, "raster_group": 0, "max_clusters": 0, "tail_split": 0},
    {"cta_group": 2, "block_n": 224, "raster_group": 0, "max_clusters": 0, "tail_split": 0},
    {"cta_group": 2, "block_n": 192, "raster_group": 0, "max_clusters": 0, "tail_split": 0},
    {"cta_group": 1, "block_n": 224, "raster_group": 0, "max_clusters": 0, "tail_split": 0},
    {"cta_group": 2, "block_n": 256, "raster_group": 0, "max_clusters": 0, "tail_split": 0,
     "consumers": 2},
    {"cta_group": 1, "block_n": 128, "cluster_ksplit": 4},
    {"cta_group": 1, "block_n": 256, "cluster_ksplit": 2},
    {"cta_group": 1, "block_n": 64, "cluster_ksplit": 1},
    {"cta_group": 1, "block_n": 32, "cluster_ksplit": 1},
    {"cta_group": 1, "block_n": 64, "cluster_ksplit": 2},
]
VID = ["cg2_n256", "cg1_n256", "cg2_n128", "cg1_n128", "cg2_n224", "cg2_n192", "cg1_n224",
       "cg2_n256_2cons", "cg1_n128_ks4", "cg1_n256_ks2", "cg1_n64", "cg1_n32", "cg1_n64_ks2"]


def k_major_only(variant, layout):
    """Widths 32, 192 and 224 exist for K-major B (A.Bt) only."""
    return layout == "ab" and variant["block_n"] % 128 != 0 and variant["block_n"] != 64


@pytest.fixture(scope="module", autouse=True)
def device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    binding.load()
    major, minor = torch.cuda.get_device_capability(0)
    assert (major, minor) == (10, 3), f"expected an sm_103 GPU, got sm_{major}{minor}"
    torch.cuda.set_device(0)
    yield
    assert binding.gemm_device_status(clear=True) == 0


def run(A_bits, B_bits, layout, dtype, options=None, D=None):
    A = to_device(A_bits, dtype)
    B = to_device(B_bits, dtype)
    fn = binding.gemm_abt if layout == "abt" else binding.gemm_ab
    out = fn(A, B, D, options=options)
    torch.cuda.synchronize()
    return out


def parity(M, N, K, layout, dtype, dist="uniform", seed=0, options=None, lda=None, ldb=None):
    """The benchmark's tolerance against the rounded oracle output, and the strict
    1 ulp + 2^-16 sum|terms| bound against its unrounded sums."""
    A, B = inputs.operands(M, N, K, layout, dtype, dist, seed, lda=lda, ldb=ldb)
    got = from_device(run(A, B, layout, dtype, options))
    ref, ref64, sum_abs = oracle_with_bound(oracle, A, B, layout, dtype)
    what = f"{M}x{N}x{K} {layout} {dtype} {options}"
    out = check_close(got, ref, dtype, what, ref64)
    out.update(check_strict(got, ref64, sum_abs, dtype, what))
    return out


# ---- exact small-integer cases first: any layout/descriptor slip shows here --

def small_int_operands(M, N, K, layout, dtype, seed, lim=2):
    rng = np.random.default_rng(seed)
    Ai = rng.integers(-lim, lim + 1, size=(M, K)).astype(np.float32)
    Bi = rng.integers(-lim, lim + 1, size=(N, K) if layout == "abt" else (K, N)).astype(np.float32)
    if dtype == "f16":
        enc = lambda x: x.astype(np.float16).view(np.uint16)
    else:
        enc = inputs.f32_to_bf16_bits
    return np.ascontiguousarray(enc(Ai)), np.ascontiguousarray(enc(Bi))


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("layout", ["abt", "ab"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_exact_small_integers(variant, layout, dtype):
    # |D| <= 4 * 64 = 256: exact in FP32 and in both output types.
    M, N, K = 256, 448, 64
    A, B = small_int_operands(M, N, K, layout, dtype, seed=1)
    if k_major_only(variant, layout):
        with pytest.raises(binding.GemmError) as e:
            run(A, B, layout, dtype, variant)
        assert e.value.status == -8
        return
    got = from_device(run(A, B, layout, dtype, variant))
    ref = oracle.gemm(A, B, layout=layout, dtype=dtype)
    assert np.array_equal(got, ref)


RING_CASES = [(1, 224), (2, 224), (1, 256), (2, 256), (1, 64), (1, 32)]


@pytest.mark.parametrize("cg,bn", RING_CASES, ids=[f"cg{c}_n{b}" for c, b in RING_CASES])
@pytest.mark.parametrize("layout", ["abt", "ab"])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_exact_across_ring_wraps(cg, bn, layout, dtype):
    # Entries in {-1, 0, 1} and K = 1024: 16 k-blocks per tile on a 6-stage
    # ring, and three clusters walking several tiles each, so the ring position,
    # its phase bit and the TMEM buffer run on across tiles.  Every partial sum
    # is an integer of magnitude <= 1024, exact in FP32 in any order, so the
    # oracle's one rounding of the exact sum is the only correct output: a
    # k-block skipped, repeated or read from a stale stage changes it.
    if layout == "ab" and bn % 128 and bn != 64:
        pytest.skip("K-major B only")
    M, N, K = 640, 3 * bn - 40, 1024
    A, B = small_int_operands(M, N, K, layout, dtype, seed=cg * 1000 + bn, lim=1)
    opts = {"cta_group": cg, "block_n": bn, "max_clusters": 3}
    got = from_device(run(A, B, layout, dtype, opts))
    ref = oracle.gemm(A, B, layout=layout, dtype=dtype)
    assert np.array_equal(got, ref)


def test_identity_single_tile():
    # D = A . I^T = A on one 128 x 128 x 128 tile.
    M = N = K = 128
    A = inputs.matrix(5, 0, M, K, "f16", "uniform")
    eye = np.eye(K, dtype=np.float16).view(np.uint16)
    got = from_device(run(A, eye, "abt", "f16"))
    assert np.array_equal(got, A)


# ---- the five workloads ---------------------------------------------------------

def config_case(cfg):
    return inputs.operands(cfg.M, cfg.N, cfg.K, cfg.layout, cfg.dtype, cfg.dist, cfg.seed)


@pytest.mark.parametrize("cfg", configs.CONFIGS[:2], ids=lambda c: c.name)
def test_small_configs_full(cfg):
    A, B = config_case(cfg)
    got = from_device(run(A, B, cfg.layout, cfg.dtype))
    ref, ref64, sum_abs = oracle_with_bound(oracle, A, B, cfg.layout, cfg.dtype)
    check_close(got, ref, cfg.dtype, cfg.name, ref64)
    check_strict(got, ref64, sum_abs, cfg.dtype, cfg.name)


@pytest.mark.parametrize("cfg", [configs.CONFIGS[4], configs.CONFIGS[2]], ids=lambda c: c.name)
def test_large_configs_full(cfg):
    A, B = config_case(cfg)
    got = from_device(run(A, B, cfg.layout, cfg.dtype))
    ref, ref64, sum_abs = oracle_with_bound(oracle, A, B, cfg.layout, cfg.dtype)
    check_close(got, ref, cfg.dtype, cfg.name, ref64)
    check_strict(got, ref64, sum_abs, cfg.dtype, cfg.name)


def test_rect_bf16_ab_sampled_tiles():
    cfg = configs.CONFIGS[3]
    A, B = config_case(cfg)
    got = from_device(run(A, B, cfg.layout, cfg.dtype))
    plan = binding.gemm_plan(cfg.M, cfg.N, cfg.K, binding.GEMM_BF16, binding.LAYOUT_AB)
    bm, bn = plan["block_m"], plan["block_n"]
    group, order = plan["raster_group"], plan["raster_order"]
    tiles = sample_tiles(cfg.M, cfg.N, cfg.K, bm, bn, group, plan["num_clusters"], plan["stages"],
                         lambda t: binding.gemm_tile_origin(cfg.M, cfg.N, bm, bn, group, t, order))
    assert len(tiles) >= plan["num_clusters"]
    for (m0, n0) in tiles:
        m1, n1 = min(m0 + bm, cfg.M), min(n0 + bn, cfg.N)
        ref, ref64, sum_abs = oracle_with_bound(oracle, A, B, "ab", "bf16", rows=(m0, m1),
                                                cols=(n0, n1))
        check_close(got[m0:m1, n0:n1], ref, "bf16", f"tile ({m0},{n0})", ref64)
        # N(0, 0.02^2) inputs make the task's 1e-2 absolute term loose here
        # (|D| ~ 0.03); the strict bound still sees a single lost K = 16 slice
        check_strict(got[m0:m1, n0:n1], ref64, sum_abs, "bf16", f"tile ({m0},{n0})")
    # every output must have been written (no NaN/garbage outside the sample):
    # D = A.B with |entries| bounded by the operand norms
    vals = decode(got, "bf16")
    assert np.isfinite(vals).all() and np.abs(vals).max() < 1.0


# ---- shapes, strides and edge cases, every variant ---------------------------

SHAPES = [
    (128, 128, 64),     # one tile, one k-block
    (256, 256, 1024),   # 16 k-blocks: several ring wraps
    (300, 200, 200),    # ragged M, N and K
    (129, 520, 136),    # one row past a tile; K not a multiple of 64
    (1, 8, 8),          # smallest legal sizes
    (64, 96, 24),       # K < 64 (zero-filled tail of the only k-block)
    (520, 264, 4000),   # K tail of 32 after 62 full blocks
    (1000, 1000, 512),  # many tiles per cluster with few clusters capped below
    (520, 456, 320),    # 224-wide tiles: the second tile's last 32-column chunk is partial
]


@pytest.mark.parametrize("variant", VARIANTS, ids=VID)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout,dtype", [("abt", "f16"), ("ab", "bf16"), ("abt", "bf16"),
                                          ("ab", "f16")])
def test_shapes(variant, shape, layout, dtype):
    M, N, K = shape
    if k_major_only(variant, layout):
        pytest.skip("K-major B only")
    parity(M, N, K, layout, dtype, "uniform" if dtype == "f16" else "normal", seed=M + N + K,
           options=variant)


@pytest.mark.parametrize("max_clusters", [1, 3, 7])
def test_few_clusters_many_tiles(max_clusters):
    # Each cluster walks many tiles: the ring position and both TMEM
    # accumulators are reused across tiles many times.
    opts = {"cta_group": 2, "block_n": 256, "raster_group": 2, "max_clusters": max_clusters, "tail_split": 0}
    parity(1024, 1280, 320, "abt", "f16", seed=max_clusters, options=opts)


def test_long_k():
    parity(256, 512, 32768, "abt", "f16", seed=3)


@pytest.mark.parametrize("layout", ["abt", "ab"])
def test_strided_operands_and_guarded_output(layout):
    # Row strides above the row length; the padding holds NaN (any read of it
    # poisons the result).  D is a view inside a larger buffer filled with a
    # sentinel, which must survive outside D.
    M, N, K = 300, 200, 136
    A, B = inputs.operands(M, N, K, layout, "f16", "uniform", 9, lda=K + 24,
                           ldb=(K + 8) if layout == "abt" else (N + 56))
    sentinel = 0x5A5A
    ldd = N + 40
    buf = torch.full((M + 3, ldd), sentinel, dtype=torch.int16, device="cuda")
    D = buf.view(torch.float16)[1:M + 1, 8:8 + N]
    run(A, B, layout, "f16", D=D)
    host = buf.cpu().numpy().view(np.uint16)
    inside = np.zeros_like(host, dtype=bool)
    inside[1:M + 1, 8:8 + N] = True
    assert (host[~inside] == sentinel).all()
    ref = oracle.gemm(A, B, layout=layout, dtype="f16")
    check_close(host[1:M + 1, 8:8 + N], ref, "f16", "strided")


@pytest.mark.parametrize("cg", [1, 2])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_224_wide_tail_chunk_is_clipped(cg, dtype):
    # 224-wide tiles store their last 32 columns as a 32 x 32 TMA box.  N = 424
    # ends 8 columns into the second tile's last chunk and M = 300 inside a
    # 32-row box: the clipped store must write those 8 columns and nothing to
    # the right of D (a sentinel guard band) or below it.
    M, N, K = 300, 424, 192
    A, B = inputs.operands(M, N, K, "abt", dtype, "uniform" if dtype == "f16" else "normal", 47)
    sentinel = 0x5A5A
    ldd = 512
    buf = torch.full((M + 2, ldd), sentinel, dtype=torch.int16, device="cuda")
    D = buf.view(TORCH_DTYPE[dtype])[:M, :N]
    run(A, B, "abt", dtype, options={"cta_group": cg, "block_n": 224}, D=D)
    host = buf.cpu().numpy().view(np.uint16)
    assert (host[:, N:] == sentinel).all() and (host[M:, :] == sentinel).all()
    ref, ref64, sum_abs = oracle_with_bound(oracle, A, B, "abt", dtype)
    check_strict(host[:M, :N], ref64, sum_abs, dtype, "224-wide tail chunk")


def test_k_zero_writes_zeros():
    buf = torch.full((40, 56), 7.0, dtype=torch.float16, device="cuda")
    D = buf[:, :48]
    A = torch.empty((40, 0), dtype=torch.float16, device="cuda")
    B = torch.empty((48, 0), dtype=torch.float16, device="cuda")
    binding.gemm_abt(A, B, D)
    torch.cuda.synchronize()
    assert (buf[:, :48] == 0).all() and (buf[:, 48:] == 7.0).all()


def test_empty_output_is_a_no_op():
    A = torch.ones((0, 64), dtype=torch.float16, device="cuda")
    B = torch.ones((32, 64), dtype=torch.float16, device="cuda")
    D = binding.gemm_abt(A, B)
    assert D.shape == (0, 32)


def test_argument_errors_on_device_buffers():
    A = torch.zeros((128, 72), dtype=torch.float16, device="cuda")
    B = torch.zeros((128, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(binding.GemmError) as e:
        binding.gemm_abt(A[:, 1:65], B)  # base pointer off by 2 bytes
    assert e.value.status == -4
    buf = torch.zeros(256 * 128, dtype=torch.float16, device="cuda")
    A2 = buf[:128 * 64].view(128, 64)
    D2 = buf[64 * 64:64 * 64 + 128 * 128].view(128, 128)  # overlaps A2
    with pytest.raises(binding.GemmError) as e:
        binding.gemm_abt(A2, B, D2)
    assert e.value.status == -5
    with pytest.raises(binding.GemmError) as e:
        binding.gemm_abt(A[:, :64].float(), B.float())
    assert e.value.status == -2


def test_deterministic_and_stream_ordered():
    A, B = inputs.operands(512, 768, 1024, "abt", "f16", "uniform", 11)
    dA, dB = to_device(A, "f16"), to_device(B, "f16")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d1 = binding.gemm_abt(dA, dB)
        d2 = binding.gemm_abt(dA, dB)
    s.synchronize()
    assert torch.equal(d1.view(torch.int16), d2.view(torch.int16))


def test_wait_timeout_is_reported_and_context_survives():
    assert binding.gemm_device_status(clear=True) == 0
    binding.gemm_selftest_wait_timeout(20_000_000)  # 20 ms
    assert binding.gemm_device_status(clear=True) == 0x501
    assert binding.gemm_device_status(clear=True) == 0
    parity(256, 256, 256, "abt", "f16", seed=5)


@pytest.mark.parametrize("opts", [None, {"cta_group": 1}, {"cta_group": 2, "max_clusters": 3},
                                  {"cta_group": 2, "consumers": 2},
                                  {"cta_group": 1, "block_n": 128, "cluster_ksplit": 4}],
                         ids=["default", "cg1", "cg2_3clusters", "cg2_2cons", "cg1_ks4"])
def test_gemm_kernel_abort_path(opts):
    # The GEMM kernel itself with a 100 ns limit on every barrier wait: the
    # first operands take microseconds to arrive, so a wait gives up.  The
    # status word must read "timeout" with the role that gave up, every CTA
    # must leave (the call returns and the device synchronises), and the next
    # normal GEMM must be correct.
    assert binding.gemm_device_status(clear=True) == 0
    M, N, K = 1024, 1024, 1024
    if opts and opts.get("cluster_ksplit"):
        M, N, K = 256, 512, 2048  # 8 tiles: one 4-CTA cluster each
        assert binding.gemm_plan(M, N, K, 0, 0, opts)["cluster_ksplit"] == 4
    A, B = inputs.operands(M, N, K, "abt", "f16", "uniform", 31)
    dA, dB = to_device(A, "f16"), to_device(B, "f16")
    D = torch.empty((M, N), dtype=torch.float16, device="cuda")
    binding.gemm_selftest_gemm_timeout(dA, dB, D, 100, options=opts)
    st = binding.gemm_device_status(clear=True)
    assert st & 0xFF == 1 and (st >> 8) in (1, 2, 3, 4), hex(st)
    assert binding.gemm_device_status(clear=True) == 0
    parity(M, N, K, "abt", "f16", seed=31, options=opts)


# ---- split tail (last partial round split along K, FP32 partials in a workspace) --

SPLIT_CASES = [
    # (M, N, K, cta_group, max_clusters, tail_split): tail = tiles mod clusters > 0
    (512, 512, 1024, 2, 3, 2),      # 4 tiles on 3 clusters: 1 tail tile in 2 ranges
    (512, 512, 1024, 2, 3, 3),
    (512, 512, 1000, 2, 3, 16),     # split capped at 16 k-blocks; K tail of 40
    (768, 768, 512, 2, 4, 8),       # 9 tiles on 4 clusters: 8 ranges, 2 per cluster
    (300, 704, 640, 2, 4, 5),       # ragged tiles: 6 tiles on 4 clusters
    (640, 520, 200, 1, 7, 6),       # cta_group 1: 15 tiles on 7 clusters, split capped at 4 k-blocks
    (1024, 1024, 2048, 2, 7, 3),    # 16 tiles on 7 clusters: tail 2 -> split 3
]


@pytest.mark.parametrize("case", SPLIT_CASES, ids=lambda c: "_".join(map(str, c)))
@pytest.mark.parametrize("layout,dtype", [("abt", "f16"), ("ab", "bf16")])
def test_split_tail(case, layout, dtype):
    M, N, K, cg, clusters, split = case
    opts = {"cta_group": cg, "block_n": 256, "max_clusters": clusters, "tail_split": split}
    plan = binding.gemm_plan(M, N, K, 0 if dtype == "f16" else 1, 0 if layout == "abt" else 1,
                             opts)
    assert plan["num_tiles"] % plan["num_clusters"] != 0
    assert plan["tail_split"] >= 2
    parity(M, N, K, layout, dtype, "uniform" if dtype == "f16" else "normal", seed=K,
           options=opts)


NO_CLUSTER_SPLIT = {"cluster_ksplit": 1}


def test_automatic_k_split_of_single_round_problems():
    # Tiles that fit one round with clusters to spare share their K loop over the
    # idle clusters when a workspace is given: at least 64 k-blocks per range
    # (here with the in-cluster split turned off, which takes precedence).
    p = binding.gemm_plan(512, 512, 16384, 0, 0, NO_CLUSTER_SPLIT)  # 16 1-CTA tiles, 256 k-blocks
    assert p["num_tiles"] == 16 and p["tail_split"] == 4 and p["num_clusters"] == 64
    assert binding.gemm_workspace_size(512, 512, 16384, 0, 0, NO_CLUSTER_SPLIT) > 0
    q = binding.gemm_plan(256, 256, 1024, 0, 0, NO_CLUSTER_SPLIT)  # 16 k-blocks: never split
    assert q["tail_split"] == 1
    r = binding.gemm_plan(512, 512, 16384, 0, 0, {"tail_split": 1, "cluster_ksplit": 1})
    assert r["tail_split"] == 1 and r["num_clusters"] == 16


@pytest.mark.parametrize("shape,layout,dtype", [
    ((512, 512, 16384), "abt", "f16"),    # 4 ranges of 64 k-blocks
    ((384, 640, 12000), "ab", "bf16"),    # ragged tiles, K tail of 32
    ((256, 512, 32768), "abt", "f16"),    # 8 ranges: the fix-up reads partials from L2
])
def test_automatic_k_split_parity(shape, layout, dtype):
    M, N, K = shape
    plan = binding.gemm_plan(M, N, K, 0 if dtype == "f16" else 1, 0 if layout == "abt" else 1,
                             NO_CLUSTER_SPLIT)
    assert plan["tail_split"] >= 2
    parity(M, N, K, layout, dtype, "uniform" if dtype == "f16" else "normal", seed=K + 7,
           options=NO_CLUSTER_SPLIT)


def test_narrow_tile_options():
    # 32- and 64-wide tiles are 1-CTA tiles; 32 takes K-major B only.
    p = binding.gemm_plan(256, 256, 1024, 0, 0, {"block_n": 32})
    assert (p["cta_group"], p["block_m"], p["block_n"], p["num_tiles"]) == (1, 128, 32, 16)
    assert binding.gemm_plan(256, 256, 1024, 0, 1, {"block_n": 64})["block_n"] == 64
    for opts, layout in (({"block_n": 64, "cta_group": 2}, 0), ({"block_n": 32}, 1),
                         ({"block_n": 96}, 0)):
        with pytest.raises(binding.GemmError) as e:
            binding.gemm_plan(256, 256, 1024, 0, layout, opts)
        assert e.value.status == -8


def test_automatic_narrow_tiles_for_shallow_single_round_problems():
    # 16 k-blocks on four 128 x 128 tiles: sixteen 32-wide tiles still fit one round.
    p = binding.gemm_plan(256, 256, 1024, 0, 0)
    assert (p["cta_group"], p["block_n"], p["num_tiles"], p["cluster_ksplit"]) == (1, 32, 16, 1)
    assert p["stages"] % 2 == 0  # 1-CTA tiles of at most 128 columns pair their stages
    # B K x N: 32-wide tiles take B N x K only, so 64
    assert binding.gemm_plan(256, 256, 1024, 0, 1)["block_n"] == 64
    # 32-wide tiles would take two rounds here: 64
    q = binding.gemm_plan(1024, 1024, 2048, 0, 0)
    assert (q["block_n"], q["num_tiles"]) == (64, 128)
    # one k-block, or 64 and more: unchanged
    assert binding.gemm_plan(128, 128, 64, 0, 0)["block_n"] == 128
    assert binding.gemm_plan(256, 256, 4096, 0, 0)["block_n"] == 128
    # an explicit width is kept
    assert binding.gemm_plan(256, 256, 1024, 0, 0, {"block_n": 128})["block_n"] == 128


@pytest.mark.parametrize("shape,layout,dtype", [
    ((256, 256, 1024), "abt", "f16"),    # the 16-k-block workload: 32-wide tiles
    ((300, 520, 1000), "abt", "bf16"),   # ragged rows, columns and K on 32-wide tiles
    ((384, 640, 2000), "ab", "f16"),     # MN-major B: 64-wide tiles
    ((1000, 1000, 2048), "abt", "f16"),  # 64-wide tiles, a ragged edge
])
def test_automatic_narrow_tile_parity(shape, layout, dtype):
    M, N, K = shape
    plan = binding.gemm_plan(M, N, K, 0 if dtype == "f16" else 1, 0 if layout == "abt" else 1)
    assert plan["block_n"] in (32, 64)
    parity(M, N, K, layout, dtype, "uniform" if dtype == "f16" else "normal", seed=K + 5)


def test_in_cluster_k_split_plans():
    # Problems whose 1-CTA tiles fit one round of clusters of 4 (or 2) CTAs
    # split each tile's K loop inside its cluster, keeping >= 16 k-blocks per
    # range, unless the workspace split would run more ranges per tile.
    p = binding.gemm_plan(256, 256, 4096, 0, 0)        # 4 tiles x 64 k-blocks
    assert (p["cta_group"], p["block_n"], p["cluster_ksplit"]) == (1, 128, 4)
    assert p["num_clusters"] == p["num_tiles"] == 4 and p["tail_split"] == 1
    q = binding.gemm_plan(256, 4096, 4096, 0, 0)       # clusters of 4 do not fit
    assert q["cluster_ksplit"] == 2
    assert binding.gemm_plan(1024, 1024, 8192, 0, 0)["cluster_ksplit"] == 2
    assert binding.gemm_plan(512, 512, 16384, 0, 0)["cluster_ksplit"] == 4
    # 16 k-blocks: 8 per range would not pay for the exchange
    assert binding.gemm_plan(256, 256, 1024, 0, 0)["cluster_ksplit"] == 1
    # the workspace split runs 8 ranges per tile here, more than 4
    r = binding.gemm_plan(256, 512, 32768, 0, 0)
    assert r["cluster_ksplit"] == 1 and r["tail_split"] == 8
    assert binding.gemm_plan(128, 128, 64, 0, 0)["cluster_ksplit"] == 1  # one k-block
    assert binding.gemm_plan(128, 128, 64, 0, 0, {"cluster_ksplit": 2})["cluster_ksplit"] == 1
    assert binding.gemm_plan(4096, 4096, 4096, 0, 0)["cluster_ksplit"] == 1
    assert binding.gemm_plan(256, 256, 1024, 0, 0, {"cluster_ksplit": 2})["cluster_ksplit"] == 2
    assert binding.gemm_plan(256, 256, 4096, 0, 0, NO_CLUSTER_SPLIT)["cluster_ksplit"] == 1
    # needs no workspace
    assert binding.gemm_workspace_size(256, 256, 4096, 0, 0) == 0


@pytest.mark.parametrize("ks", [2, 4])
@pytest.mark.parametrize("shape,layout,dtype", [
    ((256, 256, 1024), "abt", "f16"),     # the 16-k-block case
    ((300, 520, 2000), "abt", "bf16"),    # ragged tiles, K not a multiple of 64
    ((384, 640, 4096), "ab", "f16"),      # MN-major B
    ((128, 1024, 1040), "ab", "bf16"),    # odd k-blocks per range
    ((200, 136, 5000), "abt", "f16"),     # CTAs whose columns lie wholly past N
])
def test_in_cluster_k_split_parity(ks, shape, layout, dtype):
    M, N, K = shape
    opts = {"cta_group": 1, "block_n": 128, "cluster_ksplit": ks}
    plan = binding.gemm_plan(M, N, K, 0 if dtype == "f16" else 1, 0 if layout == "abt" else 1,
                             opts)
    assert plan["cluster_ksplit"] == ks
    parity(M, N, K, layout, dtype, "uniform" if dtype == "f16" else "normal", seed=K + ks,
           options=opts)


def test_in_cluster_k_split_exact_and_deterministic():
    # Small integers: every partial and the CTA-order sum are exact in FP32.
    M, N, K = 256, 512, 2048
    A, B = small_int_operands(M, N, K, "abt", "f16", seed=9, lim=1)
    for opts in ({"cta_group": 1, "block_n": 128, "cluster_ksplit": 4},
                 {"cta_group": 1, "block_n": 256, "cluster_ksplit": 2}):
        assert binding.gemm_plan(M, N, K, 0, 0, opts)["cluster_ksplit"] == opts["cluster_ksplit"]
        got = from_device(run(A, B, "abt", "f16", opts))
        assert np.array_equal(got, oracle.gemm(A, B, layout="abt", dtype="f16"))
    Af, Bf = inputs.operands(M, N, K, "abt", "f16", "uniform", 10)
    dA, dB = to_device(Af, "f16"), to_device(Bf, "f16")
    opts = {"cta_group": 1, "block_n": 128, "cluster_ksplit": 4}
    d1 = binding.gemm_abt(dA, dB, options=opts)
    d2 = binding.gemm_abt(dA, dB, options=opts)
    torch.cuda.synchronize()
    assert torch.equal(d1.view(torch.int16), d2.view(torch.int16))


def test_split_tail_deterministic_and_workspace_reused():
    M, N, K = 1024, 1024, 2048
    opts = {"cta_group": 2, "block_n": 256, "max_clusters": 7, "tail_split": 3}
    A, B = inputs.operands(M, N, K, "abt", "f16", "uniform", 77)
    dA, dB = to_device(A, "f16"), to_device(B, "f16")
    need = binding.gemm_workspace_size(M, N, K, 0, 0, opts)
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    outs = [binding.gemm_abt(dA, dB, options=opts, workspace=ws) for _ in range(3)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    ref = oracle.gemm(A, B, layout="abt", dtype="f16")
    check_close(from_device(outs[0]), ref, "f16", "split tail")
    # without a workspace: the plain schedule, also within tolerance
    plain = binding.gemm_abt(dA, dB, options=opts, workspace=None)
    torch.cuda.synchronize()
    check_close(from_device(plain), ref, "f16", "no workspace")


def test_workspace_errors():
    M, N, K = 1024, 1024, 2048
    opts = {"cta_group": 2, "block_n": 256, "max_clusters": 7, "tail_split": 3}
    need = binding.gemm_workspace_size(M, N, K, 0, 0, opts)
    A = torch.zeros((M, K), dtype=torch.float16, device="cuda")
    B = torch.zeros((N, K), dtype=torch.float16, device="cuda")
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.GemmError) as e:
        binding.gemm_abt(A, B, options=opts, workspace=small)
    assert e.value.status == -10
    big = torch.zeros(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.GemmError) as e:
        binding.gemm_abt(A, B, options=opts, workspace=big[8:])  # not 256-byte aligned
    assert e.value.status == -10


def test_default_plan_is_a_balanced_grid():
    # Automatic plans spread the rounds over the fewest clusters that keep the
    # round count: e.g. 3000 x 5000 with 224-wide tiles has 12 x 23 = 276 tiles;
    # with 76 co-resident clusters that is 4 rounds, run on ceil(276 / 4) = 69
    # clusters.
    for M, N, K in [(4096, 4096, 4096), (3000, 5000, 4000), (8192, 17408, 5120)]:
        plan = binding.gemm_plan(M, N, K, 0, 0)
        full = binding.gemm_plan(M, N, K, 0, 0, {"block_n": plan["block_n"], "tail_split": 16})
        C = full["num_clusters"]
        rounds = -(-plan["num_tiles"] // C)
        assert plan["tail_split"] == 1
        assert plan["num_clusters"] == -(-plan["num_tiles"] // rounds)


def test_automatic_width_minimises_rounds_times_width():
    # 76 two-CTA clusters.  4096 x 4096: 256-wide tiles take 4 rounds of 256
    # columns, 224-wide tiles 4 rounds of 224, so 224 wins.  8192 x 8192: 14
    # rounds x 256 against 16 x 224, a tie that the larger tile takes.
    # 2048 x 2048: 64 tiles of 256 fit one round, 224 would need two.  The
    # MN-major A.B layout always uses a multiple of 128.
    assert binding.gemm_plan(4096, 4096, 4096, 0, 0)["block_n"] == 224
    assert binding.gemm_plan(8192, 8192, 8192, 1, 0)["block_n"] == 256
    assert binding.gemm_plan(2048, 2048, 8192, 0, 0)["block_n"] == 256
    assert binding.gemm_plan(8192, 17408, 5120, 1, 1)["block_n"] in (128, 256)


# ---- seeded random cases: shapes, strides, layouts, dtypes and plan options --

def _fuzz_cases(n=48, seed=2026):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        layout = "abt" if rng.random() < 0.6 else "ab"
        dtype = "f16" if rng.random() < 0.5 else "bf16"
        M = int(rng.integers(1, 700))
        N = int(rng.integers(1, 90)) * 8
        K = int(rng.integers(1, 100)) * 8
        cg = int(rng.choice([0, 1, 2]))
        widths = [0, 128, 256] + ([192, 224] if layout == "abt" else [])
        bn = int(rng.choice(widths))
        opts = {"cta_group": cg, "block_n": bn, "raster_group": int(rng.choice([0, 1, 3])),
                "max_clusters": int(rng.choice([0, 1, 2, 5])),
                "tail_split": int(rng.choice([0, 0, 2, 3]))}
        if cg == 2 and bn in (0, 256) and rng.random() < 0.4:
            opts["consumers"] = 2
        elif cg in (0, 2) and bn in (0, 256) and rng.random() < 0.4:
            pass  # (a retired option was drawn here; the draw keeps the case list unchanged)
        pad = [int(rng.choice([0, 8, 24])) for _ in range(2)]
        cases.append((i, layout, dtype, M, N, K, opts, pad))
    return cases


@pytest.mark.parametrize("case", _fuzz_cases(), ids=lambda c: f"fuzz{c[0]}")
def test_random_cases(case):
    _, layout, dtype, M, N, K, opts, pad = case
    lda = K + pad[0]
    ldb = (K if layout == "abt" else N) + pad[1]
    parity(M, N, K, layout, dtype, "uniform" if dtype == "f16" else "normal", seed=M * 7 + N,
           options=opts, lda=lda, ldb=ldb)


def test_two_consumers_many_tiles_per_cluster():
    # 512 x 256 tiles, few clusters: the single TMEM slot is reused by every
    # tile of a cluster, so each tile's MMAs wait for the previous epilogue.
    for layout, dtype in (("abt", "f16"), ("ab", "bf16")):
        opts = {"cta_group": 2, "consumers": 2, "max_clusters": 3}
        parity(1300, 1104, 640, layout, dtype, seed=13, options=opts)


def test_two_consumer_option_limits():
    A = torch.zeros((512, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    for bad in ({"consumers": 2, "cta_group": 1}, {"consumers": 2, "block_n": 128}):
        with pytest.raises(binding.GemmError) as e:
            binding.gemm_abt(A, B, options=bad)
        assert e.value.status == -8


RASTER_CASES = [
    {"raster_order": 2, "raster_group": 3, "max_clusters": 5},
    {"raster_order": 2, "raster_group": 16},
    {"raster_order": 1, "raster_group": 1, "max_clusters": 7},
    {"raster_order": 2, "raster_group": 2, "cta_group": 1, "max_clusters": 5},
    {"l2_hints": 3},            # A evict_last
    {"l2_hints": 5},            # B evict_first
    {"l2_hints": 9},            # D evict_first
    {"l2_hints": 15, "raster_order": 2, "raster_group": 4, "cta_group": 1},
    {"l2_hints": 7, "raster_order": 2, "raster_group": 2, "tail_split": 3, "max_clusters": 7},
]


@pytest.mark.parametrize("opts", RASTER_CASES, ids=[str(i) for i in range(len(RASTER_CASES))])
@pytest.mark.parametrize("layout,dtype", [("abt", "f16"), ("ab", "bf16")])
def test_raster_orders_and_l2_hints(opts, layout, dtype):
    # Every raster order and group writes every tile once, whatever the cache
    # priorities: a ragged grid of several tiles per cluster.
    plan = binding.gemm_plan(1100, 1704, 704, 0 if dtype == "f16" else 1,
                             0 if layout == "abt" else 1, opts)
    assert plan["raster_order"] == opts.get("raster_order", plan["raster_order"])
    parity(1100, 1704, 704, layout, dtype, "uniform" if dtype == "f16" else "normal", seed=41,
           options=opts)


def test_automatic_raster_follows_the_reuse_window():
    # 8192 x 17408 x 5120 A.B: A (84 MB) is the smaller operand, and a band of
    # 16 M tiles (42 MB) fits the band budget, so M groups of 16 read A once
    # and B twice.  The transposed problem keeps a band of B instead.
    # Operands that fit in L2 together keep the G = 16 M-group order.
    p = binding.gemm_plan(8192, 17408, 5120, binding.GEMM_BF16, binding.LAYOUT_AB)
    assert (p["raster_order"], p["raster_group"]) == (1, 16)
    q = binding.gemm_plan(17408, 8192, 5120, binding.GEMM_BF16, binding.LAYOUT_AB)
    assert q["raster_order"] == 2 and q["raster_group"] == 16
    r = binding.gemm_plan(4096, 4096, 4096, binding.GEMM_F16, binding.LAYOUT_ABT)
    assert (r["raster_order"], r["raster_group"]) == (1, 16)
    assert r["l2_hints"] == 1  # no automatic hints
    # options override each part of the choice
    o = binding.gemm_plan(8192, 17408, 5120, binding.GEMM_BF16, binding.LAYOUT_AB,
                          {"raster_order": 2})
    assert o["raster_order"] == 2
    o = binding.gemm_plan(8192, 17408, 5120, binding.GEMM_BF16, binding.LAYOUT_AB,
                          {"raster_group": 5, "l2_hints": 13})
    assert (o["raster_order"], o["raster_group"], o["l2_hints"]) == (1, 5, 13)


def test_transposed_rect_n_groups_parity():
    # A problem whose automatic plan takes N groups, checked on sampled tiles.
    M, N, K = 2304, 1536, 4096
    opts = {"raster_order": 2, "raster_group": 3, "max_clusters": 5}
    parity(M, N, K, "ab", "bf16", "normal", seed=53, options=opts)


def test_raster_option_limits():
    A = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    for bad in ({"raster_order": 3}, {"l2_hints": 2}, {"l2_hints": 17}, {"raster_order": -1}):
        with pytest.raises(binding.GemmError) as e:
            binding.gemm_abt(A, B, options=bad)
        assert e.value.status == -8


def test_clock_probe_records_start_and_end():
    # gemm_run_clock_probe runs the same GEMM and records the first CTA's
    # clock counter and global timer at its start and end.
    M, N, K = 1024, 1024, 2048
    A, B = inputs.operands(M, N, K, "abt", "f16", "uniform", 43)
    dA, dB = to_device(A, "f16"), to_device(B, "f16")
    D = torch.empty((M, N), dtype=torch.float16, device="cuda")
    probe = torch.zeros(4, dtype=torch.int64, device="cuda")
    binding.gemm_run_clock_probe(dA, dB, D, probe)
    torch.cuda.synchronize()
    c0, t0, c1, t1 = probe.cpu().tolist()
    assert c1 > c0 > 0 and t1 > t0 > 0
    mhz = (c1 - c0) / (t1 - t0) * 1e3
    assert 300 < mhz < 3000, mhz
    ref, ref64, sum_abs = oracle_with_bound(oracle, A, B, "abt", "f16")
    check_strict(from_device(D), ref64, sum_abs, "f16", "clock probe")


def test_multicast_option_is_rejected():
    # No TMA load is multicast: the option accepts 0 or 1 only.
    A = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((256, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(binding.GemmError) as e:
        binding.gemm_abt(A, B, options={"multicast": 2})
    assert e.value.status == -8


def test_cuda_graph_capture_and_replay():
    # The launch is one cudaLaunchKernelEx on the caller's stream with the tile
    # descriptors as parameters, so a CUDA graph can capture it: a replay
    # recomputes D from whatever the captured buffers hold at replay time.
    M, N, K = 1024, 1536, 2048
    A1, B1 = inputs.operands(M, N, K, "abt", "f16", "uniform", 51)
    A2, B2 = inputs.operands(M, N, K, "abt", "f16", "uniform", 52)
    dA, dB = to_device(A1, "f16"), to_device(B1, "f16")
    D = torch.empty((M, N), dtype=torch.float16, device="cuda")
    binding.gemm_abt(dA, dB, D)  # first call outside the capture: plan and attributes cached
    torch.cuda.synchronize()
    D.fill_(7.0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        binding.gemm_abt(dA, dB, D)
    g.replay()
    torch.cuda.synchronize()
    check_close(from_device(D), oracle.gemm(A1, B1, layout="abt", dtype="f16"), "f16", "replay 1")
    dA.copy_(to_device(A2, "f16"))
    dB.copy_(to_device(B2, "f16"))
    g.replay()
    torch.cuda.synchronize()
    check_close(from_device(D), oracle.gemm(A2, B2, layout="abt", dtype="f16"), "f16", "replay 2")
    assert binding.gemm_device_status(clear=True) == 0
