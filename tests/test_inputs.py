"""The seeded input generator: determinism, counter addressing, bf16 rounding."""
from fractions import Fraction

import numpy as np

from scaled_dot_product_18_b300 import inputs as I


def test_deterministic_and_streams_differ():
    a = I.make_tensor_bits(3, I.STREAM_Q, (2, 3, 5, 8))
    b = I.make_tensor_bits(3, I.STREAM_Q, (2, 3, 5, 8))
    c = I.make_tensor_bits(3, I.STREAM_K, (2, 3, 5, 8))
    d = I.make_tensor_bits(4, I.STREAM_Q, (2, 3, 5, 8))
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)


def test_counter_addressing_matches_bulk_draw():
    bulk = I.normals_f64(7, 1, 3_000_001)  # several thread blocks, odd length
    for start, n in [(0, 5), (1, 4), (1_048_575, 3), (2_999_990, 11)]:
        assert np.array_equal(I.normals_f64(7, 1, n, start=start), bulk[start:start + n])
    bits = I.make_tensor_bits(7, 1, (3_000_001,))
    assert np.array_equal(bits, I.f64_to_bf16_bits(bulk))


def test_normal_moments():
    x = I.normals_f64(0, 0, 1 << 20)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1.0) < 5e-3
    assert abs((x ** 4).mean() - 3.0) < 0.05  # Gaussian kurtosis


def _nearest_bf16_exact(x: float) -> int:
    """Nearest bf16 (ties to even) by exact rational arithmetic, for positive normals."""
    fx = Fraction(x)
    e = fx.numerator.bit_length() - fx.denominator.bit_length()
    while Fraction(2) ** e > fx:
        e -= 1
    while Fraction(2) ** (e + 1) <= fx:
        e += 1
    ulp = Fraction(2) ** (e - 7)
    lo = (fx // ulp) * ulp
    hi = lo + ulp
    if fx - lo < hi - fx:
        r = lo
    elif fx - lo > hi - fx:
        r = hi
    else:
        r = lo if ((lo / ulp) % 2 == 0) else hi
    return int(np.float32(float(r)).view(np.uint32) >> 16)


def test_single_rounding_to_bf16():
    r = np.random.default_rng(0)
    xs = np.abs(r.standard_normal(2000)) * 3 + 1e-3
    # exact ties and near-ties between two bf16 values
    base = I.bf16_bits_to_f32(np.arange(0x3F80, 0x3F90, dtype=np.uint16)).astype(np.float64)
    ulp = 2.0 ** -7
    ties = np.concatenate([base + ulp / 2, base + ulp / 2 + 2.0 ** -40, base + ulp / 2 - 2.0 ** -40])
    xs = np.concatenate([xs, ties])
    got = I.f64_to_bf16_bits(xs)
    want = np.array([_nearest_bf16_exact(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, want)
    # the sign is carried through
    assert np.array_equal(I.f64_to_bf16_bits(-xs), want | np.uint16(0x8000))


def test_key_lens_in_range():
    kl = I.make_key_lens(0, 1000, 256, 512)
    assert kl.dtype == np.int32 and kl.min() >= 256 and kl.max() <= 512
    assert kl.min() < 270 and kl.max() > 500
    kl = I.make_key_lens(0, 500, 1, 100)
    assert kl.min() >= 1 and kl.max() <= 100


def test_workloads():
    w = I.WORKLOADS["c5_b1h32n16384d128_causal"]
    assert w.flops() == 4 * 32 * 16384 ** 2 * 128 / 2
    w3 = I.WORKLOADS["c3_b16h12n512d64_keylens_x1.5"]
    x = I.make_inputs(I.Workload("t", 1, 1, 4, 64, False, amplitude=1.5, seed=0))
    ref = I.f64_to_bf16_bits(1.5 * I.normals_f64(0, I.STREAM_Q, 256)).reshape(1, 1, 4, 64)
    assert np.array_equal(x.q, ref)
    assert w3.amplitude == 1.5 and w3.key_len_range == (256, 512)
