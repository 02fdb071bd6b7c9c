"""The seeded input generator: published SplitMix64 outputs, determinism, ranges."""
import numpy as np

from dense_gemm_engineering_gb300 import inputs


def test_splitmix64_published_vector():
    # First outputs of SplitMix64 from state 0, as printed with Vigna's
    # reference implementation (splitmix64.c).
    got = inputs.splitmix64_sequence(0, 3)
    assert [int(x) for x in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_based_chunks_agree():
    a = inputs.draws(5, 1, 0, 1000)
    b = np.concatenate([inputs.draws(5, 1, 0, 300), inputs.draws(5, 1, 300, 700)])
    assert np.array_equal(a, b)


def test_streams_and_seeds_differ():
    assert not np.array_equal(inputs.draws(1, 0, 0, 64), inputs.draws(1, 1, 0, 64))
    assert not np.array_equal(inputs.draws(1, 0, 0, 64), inputs.draws(2, 0, 0, 64))


def test_uniform_range_and_exactness():
    v = inputs.values_f32(0, 0, 0, 100000, "uniform")
    assert v.min() >= -1.0 and v.max() < 1.0
    # every value is a multiple of 2^-23
    assert np.array_equal(np.round(v.astype(np.float64) * 2 ** 23), v.astype(np.float64) * 2 ** 23)
    assert abs(float(v.mean())) < 0.01


def test_normal_moments():
    v = inputs.values_f32(3, 1, 0, 200000, "normal").astype(np.float64)
    assert abs(v.mean()) < 3e-4
    assert abs(v.std() - 0.02) < 3e-4


def test_bf16_rounding_ties_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 1.0 + 2 ** -8 + 2 ** -20],
                 dtype=np.float32)
    assert [hex(v) for v in inputs.f32_to_bf16_bits(x)] == ["0x3f80", "0x3f82", "0xbf80", "0x3f81"]


def test_matrix_padding_is_nan_and_view_matches():
    m = inputs.matrix(7, 0, 5, 9, "f16", "uniform", ld=16)
    assert m.shape == (5, 9) and m.strides == (32, 2)
    base = m.base if m.base is not None else m
    full = np.asarray(base).reshape(5, 16)
    assert (full[:, 9:] == inputs.NAN_BITS["f16"]).all()
    assert np.array_equal(m, inputs.matrix(7, 0, 5, 9, "f16", "uniform"))
