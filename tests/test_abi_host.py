"""The C ABI without a GPU: exported symbols, argument checks, scheduler map.

Argument validation runs before any CUDA call, so these checks need no GPU.
The scheduler tests pin the tile counts the pages print.
"""
import ctypes
import re

import pytest

from dense_gemm_engineering_gb300 import binding, build

HEADER = build.INCLUDE + "/gemm.h"


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(gemm_\w+)\s*\(", text, flags=re.M)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in binding.STATUS_NAMES.items():
        assert binding.gemm_status_string(code)
    assert binding.gemm_status_string(12345) == "unknown status"


P = 0x10000  # fake, 16-byte aligned "device" addresses: never dereferenced
Q = 0x40000000
R = 0x80000000


def call(A=P, B=Q, D=R, M=128, N=128, K=64, lda=64, ldb=64, ldd=128, dtype=0, layout=0, opts=None):
    return binding.gemm_run_ptr(A, B, D, M, N, K, lda, ldb, ldd, dtype, layout, opts, 0)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=2), -2),
    (dict(dtype=-1), -2),
    (dict(M=-1), -3),
    (dict(K=-5), -3),
    (dict(N=2 ** 31), -3),
    (dict(A=0), -1),
    (dict(B=0), -1),
    (dict(D=0), -1),
    (dict(lda=32), -3),          # lda < K
    (dict(ldd=64), -3),          # ldd < N
    (dict(layout=1, ldb=64), -3),  # A.B: ldb < N
    (dict(A=P + 8), -4),
    (dict(D=R + 2), -4),
    (dict(lda=68, K=64), -4),    # not a multiple of 8
    (dict(ldd=130), -4),
    (dict(D=P + 64), -5),        # D overlaps A
    (dict(D=Q), -5),             # D overlaps B
    (dict(layout=2), -8),
    (dict(opts={"cta_group": 3, "block_n": 0, "raster_group": 0, "max_clusters": 0, "tail_split": 0}), -8),
    (dict(opts={"cta_group": 0, "block_n": 160, "raster_group": 0, "max_clusters": 0, "tail_split": 0}), -8),
    (dict(opts={"cta_group": 0, "block_n": 0, "raster_group": 0, "max_clusters": 0, "tail_split": 17}), -8),
    (dict(opts={"consumers": 3}), -8),
    (dict(opts={"multicast": 3}), -8),
    (dict(opts={"multicast": 2}), -8),  # no multicast load exists
])
def test_argument_errors(lib, kw, status):
    assert call(**kw) == status


@pytest.mark.parametrize("kw", [dict(M=0), dict(N=0), dict(M=0, A=0, B=0, D=0)])
def test_empty_output_is_a_no_op(lib, kw):
    assert call(**kw) == 0


def test_k_zero_needs_no_inputs_but_validates_output(lib):
    assert call(K=0, A=0, B=0, D=0) == -1
    assert call(K=0, A=0, B=0, D=R + 2) == -4


# ---- the persistent scheduler's task -> tile map ---------------------------

def cover(M, N, bm, bn, group, order=1):
    tiles = -(-M // bm) * -(-N // bn)
    seen = [binding.gemm_tile_origin(M, N, bm, bn, group, t, order) for t in range(tiles)]
    return tiles, seen


@pytest.mark.parametrize("order", [1, 2], ids=["m_groups", "n_groups"])
@pytest.mark.parametrize("M,N,bm,bn,group", [
    (4096, 4096, 128, 128, 16),   # "TIRx GEMM on Blackwell", V3: 32 x 32 = 1,024 tiles
    (4096, 4096, 256, 256, 16),
    (3000, 5000, 256, 256, 16),   # ragged: last group and last tiles partial
    (3000, 5000, 128, 256, 7),
    (8192, 17408, 256, 256, 16),
    (8192, 17408, 256, 256, 5),   # N groups: 68 N tiles = 13 groups of 5 and one of 3
    (300, 100, 128, 128, 1),
])
def test_every_tile_exactly_once(lib, M, N, bm, bn, group, order):
    tiles, seen = cover(M, N, bm, bn, group, order)
    expect = {(m, n) for m in range(0, M, bm) for n in range(0, N, bn)}
    assert len(seen) == tiles == len(expect)
    assert set(seen) == expect


def test_n_group_order_is_the_m_order_transposed(lib):
    # Groups of N tiles walk M with the group's N tiles innermost: the map of
    # an M x N grid in N order is the map of the N x M grid in M order with
    # the two coordinates exchanged (and it differs from the M order).
    M, N, bm, bn, group = 3000, 5000, 256, 128, 6
    _, by_n = cover(M, N, bm, bn, group, 2)
    _, by_m_t = cover(N, M, bn, bm, group, 1)
    assert by_n == [(m, n) for (n, m) in by_m_t]
    _, by_m = cover(M, N, bm, bn, group, 1)
    assert by_n != by_m
    # the first tasks of an N group: the group's N tiles for M tile 0, then M tile 1
    assert by_n[:group + 1] == [(0, k * bn) for k in range(group)] + [(bm, 0)]
    with pytest.raises(binding.GemmError) as e:
        binding.gemm_tile_origin(M, N, bm, bn, group, 0, 3)
    assert e.value.status == -8


def test_v3_tile_count(lib):
    # "TIRx GEMM on Blackwell", V3: 4096 x 4096 with 128 x 128 tiles -> 32 x 32 = 1,024.
    tiles, _ = cover(4096, 4096, 128, 128, 16)
    assert tiles == 1024
    with pytest.raises(binding.GemmError):
        binding.gemm_tile_origin(4096, 4096, 128, 128, 16, 1024)
    # V6: 148 persistent CTAs each take about 1024 / 148 = 6.9 tiles.
    per_cta = [len(range(c, tiles, 148)) for c in range(148)]
    assert sum(per_cta) == 1024 and min(per_cta) == 6 and max(per_cta) == 7
    assert round(1024 / 148, 1) == 6.9


def test_tilefoundry_group16_order(lib):
    # "Choosing schedules and instructions for a backend", sections 1 and 3:
    # 8192 x 17408 with 128 x 256 tiles is a 64 x 68 grid of 4352 tiles; with
    # 132 resident CTAs a one-tile-per-CTA launch needs 33 waves.  The G = 16
    # order maps task -> g = task // (68*16), bn = (task // 16) % 68,
    # mi = task % 16, m = (g*16 + mi) * 128, n = bn * 256.
    M, N, BM, BN, G, GN = 8192, 17408, 128, 256, 16, 68
    tiles, seen = cover(M, N, BM, BN, G)
    assert tiles == 4352 == 64 * 68
    assert -(-4352 // 132) == 33
    for task in list(range(0, 4352, 37)) + [4351]:
        g, bn, mi = task // (GN * G), (task // G) % GN, task % G
        assert seen[task] == ((g * G + mi) * BM, bn * BN)


def test_smem_carve_up_is_disjoint():
    # The kernel's shared-memory plan (ring of A slots, ring of B slots,
    # epilogue staging, barriers) mirrors the TileFoundry tutorial's disjoint
    # intervals (section 6: [0, 98304), [98304, 147456), [147456, 212992)).
    for cg, bn, stages in ((2, 256, 6), (1, 256, 4), (2, 128, 8), (1, 128, 6)):
        a = 128 * 64 * 2
        b = (bn // cg) * 64 * 2
        spans = [(0, stages * a), (stages * a, stages * (a + b)),
                 (stages * (a + b), stages * (a + b) + 4 * 2 * 32 * 128)]
        for (s0, e0), (s1, e1) in zip(spans, spans[1:]):
            assert e0 == s1 and s0 < e0
        assert spans[-1][1] + (2 * stages + 4) * 8 + 8 + 1024 <= 232448


def test_block_scaled_smem_carve_up_is_disjoint_and_aligned():
    # Block-scaled FP8, 2-CTA 224-wide tiles, 6 stages: A and B rings (128-byte
    # K rows), A-scale atoms, B-scale blocks, one epilogue buffer per warp
    # (1 KiB aligned: it is 128-byte swizzled), barriers; within 227 KiB.
    stages, a, b = 6, 128 * 128, 112 * 128
    off_sfa = stages * (a + b)
    off_sfb = off_sfa + stages * 512
    off_epi = (off_sfb + stages * 4096 + 1023) // 1024 * 1024
    off_bar = off_epi + 4 * 4096
    spans = [(0, stages * a), (stages * a, off_sfa), (off_sfa, off_sfb),
             (off_sfb, off_sfb + stages * 4096), (off_epi, off_bar)]
    for (s0, e0), (s1, e1) in zip(spans, spans[1:]):
        assert e0 <= s1 and s0 < e0
    assert off_sfa % 512 == 0 and off_sfb % 512 == 0 and off_epi % 1024 == 0
    assert off_bar + (2 * stages + 4 + 4) * 8 + 8 + 1024 <= 232448


def test_tile_map_limits_and_large_grids(lib):
    # The scheduler's index arithmetic is 32-bit: 2^31 tiles or more is a shape
    # error; just below the limit the map still covers the far corner.
    with pytest.raises(binding.GemmError) as e:
        binding.gemm_tile_origin(1 << 30, 1 << 30, 128, 128, 16, 0)  # 2^46 tiles
    assert e.value.status == -3
    M, N, bm, bn, group = 46340 * 128, 46340 * 128, 128, 128, 16  # 2,147,395,600 tiles < 2^31
    tiles = (M // bm) * (N // bn)
    assert tiles < 2**31
    assert binding.gemm_tile_origin(M, N, bm, bn, group, tiles - 1) == (M - bm, N - bn)
    # the first task of the last (full) group and the last task of the grid
    per_group = group * (N // bn)
    last_group_first = (tiles // per_group - 1) * per_group
    m0, n0 = binding.gemm_tile_origin(M, N, bm, bn, group, last_group_first)
    assert n0 == 0 and m0 == ((M // bm) // group - 1) * group * bm


def call8(A=P, B=Q, D=R, M=128, N=128, K=128, lda=128, ldb=128, ldd=128, fmt=2, out=1, alpha=1.0,
          opts=None):
    o = binding._options(opts)
    return binding.load().gemm_fp8_run(A, B, D, M, N, K, lda, ldb, ldd, fmt, out, alpha, o, None)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt=0), -2),            # a 16-bit input type
    (dict(fmt=1), -2),
    (dict(fmt=4), -2),
    (dict(out=2), -2),            # FP8 output is not offered
    (dict(M=-1), -3),
    (dict(lda=64), -3),           # lda < K
    (dict(lda=136), -4),          # byte rows: ld must be a multiple of 16
    (dict(ldb=152, K=128), -4),
    (dict(A=P + 8), -4),
    (dict(ldd=130), -4),
    (dict(D=P + 64), -5),         # D overlaps A (A is 128 x 128 bytes = 16 KiB)
    (dict(A=0), -1),
    (dict(opts={"consumers": 3}), -8),
])
def test_fp8_argument_errors(lib, kw, status):
    assert call8(**kw) == status


def test_fp8_types_are_rejected_by_the_16bit_entry_points(lib):
    assert call(dtype=2) == -2 and call(dtype=3) == -2
    # an FP8 plan exists for A.Bt only
    n = binding.ctypes.c_size_t()
    st = binding.load().gemm_workspace_size(128, 128, 128, 2, 1, None, binding.ctypes.byref(n))
    assert st == -8


def test_fp8_empty_output_is_a_no_op(lib):
    assert call8(M=0) == 0 and call8(N=0) == 0 and call8(M=0, A=0, B=0, D=0) == 0


def call_mx(A=P, B=Q, SA=P, SB=Q, D=R, M=128, N=128, K=128, lda=128, ldb=128, ldd=128, fmt=2,
            out=1, alpha=1.0, opts=None):
    o = binding._options(opts)
    return binding.load().gemm_mx_run(A, B, SA, SB, D, M, N, K, lda, ldb, ldd, fmt, out, alpha, o,
                                      None)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt=0), -2),            # a 16-bit input type
    (dict(fmt=1), -2),
    (dict(out=3), -2),
    (dict(M=-1), -3),
    (dict(lda=64), -3),
    (dict(lda=136), -4),
    (dict(A=P + 8), -4),
    (dict(D=P + 64), -5),         # D overlaps A
    (dict(A=0), -1),
    (dict(SA=0), -1),             # the scales are operands too
    (dict(SB=0), -1),
    (dict(SA=P + 4), -4),
    (dict(SB=Q + 8), -4),
])
def test_mx_argument_errors(lib, kw, status):
    assert call_mx(**kw) == status


def test_mx_empty_output_and_empty_k(lib):
    assert call_mx(M=0) == 0 and call_mx(N=0, SA=0, SB=0) == 0


def test_mx_scales_size(lib):
    n = binding.ctypes.c_size_t()
    for rows, K, want in [(0, 128, 0), (1, 1, 512), (128, 128, 512), (129, 128, 1024),
                          (300, 1000, 3 * 8 * 512), (8192, 8192, 64 * 64 * 512)]:
        assert binding.load().gemm_mx_scales_size(rows, K, binding.ctypes.byref(n)) == 0
        assert n.value == want == binding.mx_scales_size(rows, K)
    assert binding.load().gemm_mx_scales_size(-1, 8, binding.ctypes.byref(n)) == -3
    assert binding.load().gemm_mx_scales_size(8, 8, None) == -1


def test_mx_pack_argument_errors(lib):
    pack = binding.load().gemm_mx_pack_scales
    assert pack(P, -1, 64, 2, Q, None) == -3
    assert pack(P, 4, 64, 1, Q, None) == -3     # ld < ceil(K / 32)
    assert pack(0, 4, 64, 2, Q, None) == -1
    assert pack(P, 4, 64, 2, Q + 4, None) == -4
    assert pack(P + 4, 4, 64, 2, P, None) == -5   # dst overlaps src
    assert pack(P, 0, 64, 2, 0, None) == 0        # nothing to write


def test_mx_scales_b_size_and_pack_errors(lib):
    n = binding.ctypes.c_size_t()
    for N, K, want in [(0, 128, 0), (1, 1, 4096), (224, 128, 4096), (225, 129, 2 * 2 * 4096),
                       (8192, 8192, 37 * 64 * 4096)]:
        assert binding.load().gemm_mx_scales_b_size(N, K, binding.ctypes.byref(n)) == 0
        assert n.value == want == binding.mx_scales_b_size(N, K)
    pack = binding.load().gemm_mx_pack_scales_b
    assert pack(P, -1, 64, 2, Q, None) == -3
    assert pack(P, 4, 64, 1, Q, None) == -3
    assert pack(0, 4, 64, 2, Q, None) == -1
    assert pack(P, 4, 64, 2, Q + 4, None) == -4
    assert pack(P + 4, 4, 64, 2, P, None) == -5


def test_binding_offers_every_c_entry_point_by_name():
    # every function include/gemm.h declares has a Python callable of the same name
    missing = [name for name in binding.EXPORTS if not callable(getattr(binding, name, None))]
    assert not missing, missing
