"""Pins for the CPU oracle, independent of the oracle's own code.

Each check compares the oracle with something other than itself: products
worked out by hand (tests/golden/hand_products.txt), identity and permutation
operands, the transpose invariant (A.Bt)t = B.At, closed forms, exact integer
products from numpy's int64 matmul, torch.mm in float64, and numpy's / torch's
own 16-bit conversions for the rounding rule.

The checks are plain functions of an oracle object so that
tests/test_oracle_mutants.py can run them against copies of the oracle with
planted mistakes and show that each mistake is caught.
"""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_engineering_gb300 import inputs
from golden_io import hand_products


def enc(values, dtype):
    """Exact decimal values -> 16-bit patterns through numpy / torch (not the oracle)."""
    v = np.asarray(values, dtype=np.float64)
    if dtype == "f16":
        h = v.astype(np.float16)
        assert np.array_equal(h.astype(np.float64), v, equal_nan=True), "not representable"
        return h.view(np.uint16)
    t = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(t.to(torch.float64).numpy(), v), "not representable"
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def dec(bits, dtype):
    """16-bit patterns -> float64 through numpy / torch (not the oracle)."""
    b = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return b.view(np.float16).astype(np.float64)
    return torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()


CASES = hand_products()


def pin_hand_products_abt(orc):
    for case in CASES:
        dt = case["dtype"]
        A, B = enc(case["A"], dt), enc(case["B"], dt)
        D = orc.gemm(A, B, layout="abt", dtype=dt)
        assert np.array_equal(D, case["bits"]), (case["name"], D, case["bits"])
        assert np.array_equal(dec(D, dt), case["D"]), case["name"]


def pin_hand_products_ab(orc):
    for case in CASES:
        dt = case["dtype"]
        A = enc(case["A"], dt)
        Bkn = np.ascontiguousarray(enc(case["B"], dt).T)  # K x N storage
        D = orc.gemm(A, Bkn, layout="ab", dtype=dt)
        assert np.array_equal(D, case["bits"]), case["name"]


def pin_identity(orc):
    for dtype in ("f16", "bf16"):
        A = inputs.matrix(11, 0, 7, 16, dtype, "uniform")
        eye = enc(np.eye(16), dtype)
        assert np.array_equal(orc.gemm(A, eye, layout="abt", dtype=dtype), A)
        assert np.array_equal(orc.gemm(A, eye, layout="ab", dtype=dtype), A)


def pin_permutation(orc):
    rng = np.random.default_rng(5)
    K = 24
    perm = rng.permutation(K)
    P = np.zeros((K, K))
    P[np.arange(K), perm] = 1.0  # row j of P picks column perm[j] of A
    for dtype in ("f16", "bf16"):
        A = inputs.matrix(12, 0, 9, K, dtype, "uniform")
        D = orc.gemm(A, enc(P, dtype), layout="abt", dtype=dtype)
        assert np.array_equal(D, A[:, perm])
        # A.P with P stored K x N: column j of D is column argsort(perm)[j] of A
        D2 = orc.gemm(A, enc(P, dtype), layout="ab", dtype=dtype)
        assert np.array_equal(D2, A[:, np.argsort(perm)])


def pin_transpose_invariant(orc):
    for dtype in ("f16", "bf16"):
        A, B = inputs.operands(13, 21, 37, "abt", dtype, "uniform", seed=7)
        D1 = orc.gemm(A, B, layout="abt", dtype=dtype)
        D2 = orc.gemm(B, A, layout="abt", dtype=dtype)
        assert np.array_equal(D1.T, D2)
        # the A.B form on the transposed B gives the same bits
        D3 = orc.gemm(A, np.ascontiguousarray(B.T), layout="ab", dtype=dtype)
        assert np.array_equal(D1, D3)


def pin_all_ones_closed_form(orc):
    # D[i,j] = sum_k B[j,k].  Values are multiples of 2^-24 (binary16) or
    # 2^-30 (bfloat16 of the uniform draws) with |v| <= 1, so every summation
    # order is exact in binary64; numpy then rounds to binary16.
    K = 300
    for dtype in ("f16", "bf16"):
        B = inputs.matrix(3, 1, 17, K, dtype, "uniform")
        ones = enc(np.ones((5, K)), dtype)
        D, D64 = orc.gemm(ones, B, layout="abt", dtype=dtype, want_f64=True)
        s = dec(B, dtype).sum(axis=1)
        assert np.array_equal(D64, np.broadcast_to(s, (5, 17)))
        if dtype == "f16":
            assert np.array_equal(D, np.broadcast_to(s.astype(np.float16).view(np.uint16), (5, 17)))


def pin_small_integers_exact(orc):
    # |D| <= lim^2 * K stays within the exactly representable integers
    # (2048 for binary16, 256 for bfloat16), so D must equal numpy's int64 product.
    rng = np.random.default_rng(9)
    M, N, K = 19, 23, 64
    for dtype, lim in (("f16", 4), ("bf16", 2)):
        Ai = rng.integers(-lim, lim + 1, size=(M, K))
        Bi = rng.integers(-lim, lim + 1, size=(N, K))
        ref = (Ai @ Bi.T).astype(np.float64)
        for layout in ("abt", "ab"):
            Bstore = Bi if layout == "abt" else np.ascontiguousarray(Bi.T)
            D = orc.gemm(enc(Ai, dtype), enc(Bstore, dtype), layout=layout, dtype=dtype)
            assert np.array_equal(dec(D, dtype), ref), (dtype, layout)


def pin_against_torch_float64(orc):
    for dtype in ("f16", "bf16"):
        for layout in ("abt", "ab"):
            A, B = inputs.operands(33, 29, 200, layout, dtype, "uniform", seed=21)
            D, D64 = orc.gemm(A, B, layout=layout, dtype=dtype, want_f64=True)
            Bt = torch.from_numpy(dec(B, dtype))
            Bt = Bt.T if layout == "abt" else Bt
            ref = (torch.from_numpy(dec(A, dtype)) @ Bt).numpy()
            np.testing.assert_allclose(D64, ref, rtol=1e-13, atol=1e-15)
            if dtype == "f16":
                assert np.array_equal(D, ref.astype(np.float16).view(np.uint16))


def pin_strided_operands_ignore_padding(orc):
    # Row strides larger than K; the padding holds NaN, which would poison any
    # sum that read it.
    A = inputs.matrix(40, 0, 10, 30, "f16", "uniform", ld=40)
    B = inputs.matrix(40, 1, 12, 30, "f16", "uniform", ld=48)
    D = orc.gemm(A, B, layout="abt", dtype="f16")
    Dc = orc.gemm(np.ascontiguousarray(A), np.ascontiguousarray(B), layout="abt", dtype="f16")
    assert np.array_equal(D, Dc)
    assert np.isfinite(dec(D, "f16")).all()


def pin_sub_block_matches_full(orc):
    A, B = inputs.operands(40, 50, 33, "ab", "bf16", "normal", seed=3)
    full = orc.gemm(A, B, layout="ab", dtype="bf16")
    part = orc.gemm(A, B, layout="ab", dtype="bf16", rows=(7, 31), cols=(13, 47))
    assert np.array_equal(part, full[7:31, 13:47])


def pin_empty_k_gives_zero(orc):
    A = np.zeros((3, 0), dtype=np.uint16)
    B = np.zeros((4, 0), dtype=np.uint16)
    D = orc.gemm(A, B, layout="abt", dtype="f16")
    assert D.shape == (3, 4) and not D.any()


# ---- the rounding rule, against independent conversions --------------------

def pin_f16_decode_matches_numpy(orc):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.to_double(allbits, "f16")
    ref = allbits.view(np.float16).astype(np.float64)
    assert np.array_equal(got, ref, equal_nan=True)


def pin_bf16_decode_matches_torch(orc):
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.to_double(allbits, "bf16")
    assert np.array_equal(got, dec(allbits, "bf16"), equal_nan=True)


def pin_f16_rounding_matches_numpy(orc):
    # numpy rounds binary64 -> binary16 directly (one rounding step).
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, size=20000),
        (np.arange(-3000, 3000) + 0.5) * 2.0 ** -10,  # exact ties around 1..3
        (np.arange(0, 2000) + 0.5) * 2.0 ** -24,  # ties in the subnormal range
        np.array([65504.0, 65519.999, 65520.0, -65520.0, 1e6, 0.0, -0.0, 2.0 ** -25]),
    ])
    got = orc.from_double(x, "f16")
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def pin_bf16_rounding_matches_torch_on_binary32_values(orc):
    # For values that are exact binary32 numbers, rounding binary64 -> bfloat16
    # equals torch's binary32 -> bfloat16 rounding (nearest, ties to even).
    rng = np.random.default_rng(2)
    x32 = np.concatenate([
        (rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, size=20000)),
        (np.arange(-3000, 3000) + 0.5) * 2.0 ** -7,  # exact ties
    ]).astype(np.float32)
    got = orc.from_double(x32.astype(np.float64), "bf16")
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ---- FP8 (E4M3 / E5M2) inputs -------------------------------------------------

def fp8_torch_values(codes, fmt):
    """FP8 patterns -> float64 through torch's own float8 types (not the oracle)."""
    t = torch.from_numpy(np.asarray(codes, dtype=np.uint8).copy())
    dt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return t.view(dt).to(torch.float64).numpy()


def pin_fp8_decode_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    for fmt in ("e4m3", "e5m2"):
        got = orc.fp8_to_double(codes, fmt)
        ref = fp8_torch_values(codes, fmt)
        assert np.array_equal(np.isnan(got), np.isnan(ref)), fmt
        ok = ~np.isnan(ref)
        assert np.array_equal(got[ok], ref[ok]), fmt


def pin_fp8_decode_hand_values(orc):
    # OCP 8-bit floating point: E4M3 bias 7 (no infinities, S.1111.111 = NaN),
    # E5M2 bias 15 (IEEE style); values worked out by hand.
    e4m3 = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5,
            0x38: 1.0, 0x3F: 1.875, 0x40: 2.0, 0x48: 4.0, 0x77: 240.0, 0x7E: 448.0,
            0xB8: -1.0, 0xFE: -448.0}
    e5m2 = {0x00: 0.0, 0x01: 2.0 ** -16, 0x03: 3 * 2.0 ** -16, 0x04: 2.0 ** -14,
            0x3C: 1.0, 0x3D: 1.25, 0x40: 2.0, 0x7B: 57344.0, 0xBC: -1.0}
    for fmt, table in (("e4m3", e4m3), ("e5m2", e5m2)):
        codes = np.array(list(table), dtype=np.uint8)
        assert np.array_equal(orc.fp8_to_double(codes, fmt), np.array(list(table.values()))), fmt
    assert np.isnan(orc.fp8_to_double(np.array([0x7F, 0xFF], np.uint8), "e4m3")).all()
    assert np.isinf(orc.fp8_to_double(np.array([0x7C], np.uint8), "e5m2")).all()
    assert np.isnan(orc.fp8_to_double(np.array([0x7D, 0x7E, 0x7F], np.uint8), "e5m2")).all()


def pin_fp8_hand_product(orc):
    # A = [1, 2, -0.5], B rows [4, 0.25, 2] and [1, 1, 1]:  D = [3.5, 2.5]
    A = np.array([[0x38, 0x40, 0xB0]], dtype=np.uint8)
    B = np.array([[0x48, 0x28, 0x40], [0x38, 0x38, 0x38]], dtype=np.uint8)
    _, d64 = orc.gemm_fp8(A, B, fmt="e4m3", out_dtype="f16", want_f64=True)
    assert np.array_equal(d64, [[3.5, 2.5]])
    d16 = orc.gemm_fp8(A, B, fmt="e4m3", out_dtype="bf16", alpha=2.0)
    assert np.array_equal(dec(d16, "bf16"), [[7.0, 5.0]])


def pin_fp8_gemm_matches_16bit_path(orc):
    # Every E4M3 and E5M2 value is exact in binary16, so the FP8 GEMM must equal
    # the 16-bit GEMM of the same values (converted here by torch and numpy).
    for fmt in ("e4m3", "e5m2"):
        A, B = inputs.operands(19, 23, 77, "abt", fmt, "uniform", 5)
        A16 = fp8_torch_values(A, fmt).astype(np.float16).view(np.uint16)
        B16 = fp8_torch_values(B, fmt).astype(np.float16).view(np.uint16)
        got, g64 = orc.gemm_fp8(A, B, fmt=fmt, out_dtype="f16", want_f64=True)
        ref, r64 = orc.gemm(A16, B16, layout="abt", dtype="f16", want_f64=True)
        assert np.array_equal(g64, r64) and np.array_equal(got, ref), fmt


def pin_fp8_against_torch_float64(orc):
    for fmt in ("e4m3", "e5m2"):
        A, B = inputs.operands(13, 9, 150, "abt", fmt, "normal", 6)
        a, b = fp8_torch_values(A, fmt), fp8_torch_values(B, fmt)
        ref = (torch.from_numpy(a) @ torch.from_numpy(b).T).numpy() * np.float64(np.float32(0.375))
        _, got = orc.gemm_fp8(A, B, fmt=fmt, out_dtype="bf16", alpha=0.375, want_f64=True)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-300), fmt


def pin_fp8_alpha_applied_once(orc):
    A, B = inputs.operands(7, 11, 64, "abt", "e4m3", "uniform", 8)
    _, one = orc.gemm_fp8(A, B, fmt="e4m3", out_dtype="bf16", want_f64=True)
    for alpha in (0.5, 3.0, 0.1):
        _, got = orc.gemm_fp8(A, B, fmt="e4m3", out_dtype="bf16", alpha=alpha, want_f64=True)
        assert np.array_equal(got, np.float64(np.float32(alpha)) * one), alpha


def pin_fp8_transpose_invariant(orc):
    A, B = inputs.operands(12, 17, 40, "abt", "e5m2", "uniform", 9)
    d1 = orc.gemm_fp8(A, B, fmt="e5m2", out_dtype="bf16")
    d2 = orc.gemm_fp8(B, A, fmt="e5m2", out_dtype="bf16")
    assert np.array_equal(d1.T, d2)


def pin_ue8m0_decode_hand_values(orc):
    # UE8M0 (OCP Microscaling): 8 exponent bits, bias 127, no sign or fraction;
    # 255 is NaN.
    codes = np.array([0, 1, 120, 126, 127, 128, 130, 254], dtype=np.uint8)
    want = [2.0 ** -127, 2.0 ** -126, 2.0 ** -7, 0.5, 1.0, 2.0, 8.0, 2.0 ** 127]
    assert np.array_equal(orc.ue8m0_to_double(codes), want)
    assert np.isnan(orc.ue8m0_to_double(np.array([255], np.uint8))).all()


def pin_mx_hand_product(orc):
    # K = 33: group 0 = 32 ones, group 1 = one element.  A = [1 x32, 2],
    # B = [1 x33]; SA = [128, 126] (x2, x0.5), SB = [127, 129] (x1, x4):
    # D = 32 * 2 * 1 + 2 * 0.5 * 4 = 68.
    A = np.array([[0x38] * 32 + [0x40]], dtype=np.uint8)
    B = np.array([[0x38] * 33], dtype=np.uint8)
    SA = np.array([[128, 126]], dtype=np.uint8)
    SB = np.array([[127, 129]], dtype=np.uint8)
    _, d64 = orc.gemm_mx(A, B, SA, SB, fmt="e4m3", out_dtype="f16", want_f64=True)
    assert np.array_equal(d64, [[68.0]])
    d16 = orc.gemm_mx(A, B, SA, SB, fmt="e4m3", out_dtype="bf16", alpha=0.25)
    assert np.array_equal(dec(d16, "bf16"), [[17.0]])


def pin_mx_unit_scales_equal_fp8(orc):
    # Every scale 2^0: the block-scaled product is the plain FP8 product.
    for fmt in ("e4m3", "e5m2"):
        A, B = inputs.operands(9, 14, 77, "abt", fmt, "uniform", 12)
        ones = lambda r: np.full((r, 3), 127, dtype=np.uint8)
        got, g64 = orc.gemm_mx(A, B, ones(9), ones(14), fmt=fmt, out_dtype="bf16", alpha=0.75,
                               want_f64=True)
        ref, r64 = orc.gemm_fp8(A, B, fmt=fmt, out_dtype="bf16", alpha=0.75, want_f64=True)
        assert np.array_equal(g64, r64) and np.array_equal(got, ref), fmt


def pin_mx_uniform_scales_scale_the_result(orc):
    # SA = 127 + a and SB = 127 + b everywhere: D = 2^(a + b) * (A . Bt), exactly.
    A, B = inputs.operands(11, 8, 96, "abt", "e4m3", "normal", 13)
    _, base = orc.gemm_fp8(A, B, fmt="e4m3", out_dtype="bf16", want_f64=True)
    for a, b in ((3, -5), (-2, 0), (6, 1)):
        SA = np.full((11, 3), 127 + a, dtype=np.uint8)
        SB = np.full((8, 3), 127 + b, dtype=np.uint8)
        _, got = orc.gemm_mx(A, B, SA, SB, fmt="e4m3", out_dtype="bf16", want_f64=True)
        assert np.array_equal(got, base * 2.0 ** (a + b)), (a, b)


def pin_mx_groups_closed_form(orc):
    # Small-integer FP8 values and a different scale per (row, group): the sum
    # splits into one exact product per 32-column group,
    #   D = sum_g 2^(SA[:,g] - 127) 2^(SB[:,g] - 127)^T * (A_g . B_g^T),
    # computed with numpy's float64 matmul (all partial sums exact here).
    # K = 100: groups of 32, 32, 32 and 4 columns.
    rng = np.random.default_rng(14)
    M, N, K = 6, 5, 100
    for fmt in ("e4m3", "e5m2"):
        a = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
        b = rng.integers(-3, 4, size=(N, K)).astype(np.float32)
        A, B = inputs.f32_to_fp8_bits(a, fmt), inputs.f32_to_fp8_bits(b, fmt)
        SA = rng.integers(121, 134, size=(M, 4)).astype(np.uint8)
        SB = rng.integers(121, 134, size=(N, 4)).astype(np.uint8)
        want = np.zeros((M, N))
        for g in range(4):
            cols = slice(32 * g, min(32 * g + 32, K))
            sa = np.ldexp(1.0, SA[:, g].astype(int) - 127)
            sb = np.ldexp(1.0, SB[:, g].astype(int) - 127)
            want += np.outer(sa, sb) * (a[:, cols].astype(np.float64) @ b[:, cols].astype(np.float64).T)
        _, got = orc.gemm_mx(A, B, SA, SB, fmt=fmt, out_dtype="bf16", want_f64=True)
        assert np.array_equal(got, want), fmt


def pin_mx_strided_scales_ignore_padding(orc):
    # Scale rows with padding (255 = NaN there) and operands with NaN padding:
    # nothing outside the logical shapes may be read.
    A, B, SA, SB = inputs.mx_operands(7, 9, 70, "e5m2", "uniform", 15, lda=96, ldb=80)
    SA2 = inputs.mx_scales(15, 2, 7, 70, ld=8)
    SB2 = inputs.mx_scales(15, 3, 9, 70, ld=5)
    assert np.array_equal(SA2, SA) and np.array_equal(SB2, SB)
    got = orc.gemm_mx(A, B, SA2, SB2, fmt="e5m2", out_dtype="bf16")
    ref = orc.gemm_mx(np.ascontiguousarray(A), np.ascontiguousarray(B), np.ascontiguousarray(SA),
                      np.ascontiguousarray(SB), fmt="e5m2", out_dtype="bf16")
    assert np.array_equal(got, ref) and not np.isnan(dec(got, "bf16")).any()


def pin_mx_nan_scale_poisons_its_row(orc):
    A, B, SA, SB = inputs.mx_operands(4, 3, 64, "e4m3", "uniform", 16)
    SA = SA.copy()
    SA[2, 1] = 255
    _, d64 = orc.gemm_mx(A, B, SA, SB, fmt="e4m3", out_dtype="bf16", want_f64=True)
    assert np.isnan(d64[2]).all() and not np.isnan(np.delete(d64, 2, axis=0)).any()


def pin_mx_transpose_invariant(orc):
    A, B, SA, SB = inputs.mx_operands(10, 13, 90, "e4m3", "normal", 17)
    d1 = orc.gemm_mx(A, B, SA, SB, fmt="e4m3", out_dtype="f16")
    d2 = orc.gemm_mx(B, A, SB, SA, fmt="e4m3", out_dtype="f16")
    assert np.array_equal(d1.T, d2)


PINS = {name: fn for name, fn in sorted(globals().items()) if name.startswith("pin_")}


@pytest.mark.parametrize("name", sorted(PINS))
def test_pin(name):
    PINS[name](oracle.get())
