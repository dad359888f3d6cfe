"""The seeded input generator: determinism, distribution, rounding, row stress."""
import numpy as np

from exact_tiled_attention_forward_gb300 import inputs as I


def test_splitmix64_published_first_outputs():
    # SplitMix64 seeded with 0: the first outputs are mix(k * GAMMA), k = 1, 2, 3
    # (published sequence of the reference generator by Vigna).
    z = I._mix64(np.arange(1, 4, dtype=np.uint64) * I.GAMMA)
    assert [int(x) for x in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_prefix_consistent():
    a = I.normal_bf16(0, I.STREAM_K, (3, 1000))
    b = I.normal_bf16(0, I.STREAM_K, (3, 1000))
    assert np.array_equal(a, b)
    c = I.normal_bf16(0, I.STREAM_K, (3001,))
    assert np.array_equal(a.ravel(), c[:3000])
    assert not np.array_equal(a, I.normal_bf16(1, I.STREAM_K, (3, 1000)))
    assert not np.array_equal(a, I.normal_bf16(0, I.STREAM_V, (3, 1000)))


def test_standard_normal_moments():
    x = I.normal_f64(0, I.STREAM_Q, 1 << 20)
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1) < 5e-3
    assert abs((x > 1.0).mean() - 0.158655) < 2e-3


def test_bf16_rounding_is_nearest_even():
    vals = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 0.0, 3.0e-3])
    bits = I.f64_to_bf16_bits(vals)
    back = I.bf16_bits_to_f32(bits).astype(np.float64)
    # ties go to even: 1 + 2^-8 -> 1.0, 1 + 3*2^-8 -> 1 + 2^-6
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == 1.0 + 2**-6
    assert back[3] == 1.0 and back[4] == -2.5 and back[5] == 0.0
    assert abs(back[6] - 3.0e-3) <= 3.0e-3 * 2**-8


def test_k_row_stress():
    a = I.make_inputs(2, 4, 2, 16, 1000, 8, seed=0, k_row_frac=0.01)
    base = I.make_inputs(2, 4, 2, 16, 1000, 8, seed=0)
    rows = I.scaled_rows(0, 4, 1000, 0.01)
    assert rows.shape == (4, 10)
    kf = I.bf16_bits_to_f32(a.k).reshape(4, 1000, 8)
    bf = I.bf16_bits_to_f32(base.k).reshape(4, 1000, 8)
    for bh in range(4):
        mask = np.zeros(1000, bool)
        mask[rows[bh]] = True
        assert np.array_equal(kf[bh, mask], bf[bh, mask] * 8)   # exact in bf16
        assert np.array_equal(kf[bh, ~mask], bf[bh, ~mask])
    assert np.array_equal(a.q, base.q) and np.array_equal(a.v, base.v)


def test_f16_rounding_is_ieee_nearest_even():
    # binary16: 10 fraction bits; ties go to the even neighbour, past the largest
    # finite value (65504) the halfway point 65520 rounds to infinity, and the
    # subnormal grid is 2^-24
    x = np.array([1 + 2.0**-11, 1 + 3 * 2.0**-11, 1 + 2.0**-11 + 2.0**-30, 65504.0, 65519.99,
                  65520.0, 2.0**-25, 3 * 2.0**-26, -2.0**-25, 2.0**-14 - 2.0**-25])
    want = np.array([1.0, 1 + 2.0**-9, 1 + 2.0**-10, 65504.0, 65504.0, np.inf, 0.0, 2.0**-24,
                     -0.0, 2.0**-14])
    with np.errstate(over="ignore"):      # 65520 overflows on purpose
        got = I.f64_to_f16(x).astype(np.float64)
    assert np.array_equal(got, want)
    assert np.signbit(got[8])


def test_f16_inputs_follow_the_same_stream():
    # the FP16 draw is the same deviates as the BF16 one, rounded to binary16
    z = I.normal_f64(4, I.STREAM_V, 4096)
    assert np.array_equal(I.normal_f16(4, I.STREAM_V, (4096,)), z.astype(np.float16))
    a = I.make_inputs(1, 2, 1, 40, 300, 64, seed=4, k_row_frac=0.02, dtype="f16")
    b = I.make_inputs(1, 2, 1, 40, 300, 64, seed=4, k_row_frac=0.02, dtype="bf16")
    assert a.dtype == "f16" and a.q.dtype == np.float16 and b.q.dtype == np.uint16
    # the scaled K rows are the same rows, and x8 is exact in binary16
    plain = I.make_inputs(1, 2, 1, 40, 300, 64, seed=4, dtype="f16")
    rows = I.scaled_rows(4, 1, 300, 0.02)[0]
    assert np.array_equal(a.k[0, 0, rows].astype(np.float64), plain.k[0, 0, rows].astype(np.float64) * 8)
    others = np.setdiff1d(np.arange(300), rows)
    assert np.array_equal(a.k[0, 0, others], plain.k[0, 0, others])
    # both roundings of one deviate are within their half-ulps of each other
    qf = a.q.astype(np.float64)
    qb = I.bf16_bits_to_f32(b.q).astype(np.float64)
    assert np.all(np.abs(qf - qb) <= np.abs(qf) * (2.0**-8 + 2.0**-11) + 2.0**-24)
