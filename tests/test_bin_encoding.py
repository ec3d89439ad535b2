"""The 16-bit chunk-bin encoding of the scoring kernels (bin_encode / bin_decode in common.cuh).

The kernels store each chunk bin b (a sum of 2^(t - R) >= 0 over one chunk) through its value
scaled by 2^-86: the scoring kernels form the scaled values directly, against the shifted
reference R + 86, and keep the upper 16 bits of the fp32 pattern, rounded half up at the 11th
significant bit.  Over [2^-40, 2^23) of R the scaled value is a normal float and the code holds its
exponent field (1 .. 63) and ten mantissa bits; smaller bins become fp32 subnormals or zero.  The
same integer steps replayed in numpy must keep the relative error within 2^-11 over
[2^-40, (1 - 2^-12) 2^23), the absolute error at about 2^-51 under 2^-40, and stay monotone: the
chunk-score tolerance 1e-3 relative rests on it.
"""
import numpy as np

SHIFT = 86


def scaled(b):
    """b * 2^-86 in fp32 (the value the kernels form), from a float64 b."""
    return (np.asarray(b, np.float64) * 2.0 ** -SHIFT).astype(np.float32)


def encode(v):
    """Code of a scaled fp32 value below 2^-63 (two integer ops in the kernels)."""
    u = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x1000) >> 13).astype(np.uint32)


def encode_sat(v):
    return np.minimum(encode(v), 0xFFFF).astype(np.uint32)


def decode(code):
    """The scaled value of a code; times 2^86 the bin relative to R."""
    code = np.asarray(code, np.uint32).astype(np.uint64)
    return (code << 13).astype(np.uint32).view(np.float32)


def unscaled(v):
    return np.asarray(v, np.float64) * 2.0 ** SHIFT


def test_relative_error_over_the_range():
    rng = np.random.default_rng(5)
    b = 2.0 ** rng.uniform(-39.99, 22.99, 1_000_000)
    codes = encode(scaled(b))
    assert codes.max() <= 0xFFFF
    rel = np.abs(unscaled(decode(codes)) / b - 1.0)
    assert rel.max() <= 2.0 ** -11 * (1 + 1e-6)


def test_zero_small_bins_and_top():
    assert encode(scaled(0.0)) == 0 and decode(np.uint32(0)) == 0.0
    # below 2^-40 of the reference: subnormal scaled values, absolute error at most 2^-51
    b = np.concatenate([2.0 ** np.random.default_rng(7).uniform(-60, -40, 100_000), [2.0 ** -41, 2.0 ** -52]])
    err = np.abs(unscaled(decode(encode(scaled(b)))) - b)
    assert err.max() <= 2.0 ** -51 * (1 + 1e-3)       # half the code spacing, plus the fp32 rounding
    # the largest bin the tensor-core kernel keeps, (1 - 2^-10) 2^23, stays in 16 bits, and so does
    # (1 - 2^-11) 2^23 (the top code); from (1 - 2^-12) 2^23 the rounding carries past them, which the
    # saturating encoder stops
    assert encode(scaled(2.0 ** 23 * (1 - 2.0 ** -10))).item() == 0xFFFE
    assert encode(scaled(2.0 ** 23 * (1 - 2.0 ** -11))).item() == 0xFFFF
    assert encode(scaled(2.0 ** 23 * (1 - 2.0 ** -12))).item() == 0x10000
    assert encode_sat(scaled(2.0 ** 30)).item() == 0xFFFF


def test_monotone_and_exact_on_short_mantissas():
    b = np.sort(2.0 ** np.random.default_rng(9).uniform(-45, 22.9, 200_000))
    y = unscaled(decode(encode(scaled(b))))
    assert np.all(np.diff(y) >= 0)
    z = (np.arange(1, 1024, dtype=np.float64) / 1024 + 1) * 2.0 ** -7       # 10-bit mantissas
    assert np.array_equal(unscaled(decode(encode(scaled(z)))), z)


def decode2(v):
    """The finalisation's decode of two bins packed in a 32-bit word (two integer ops a bin)."""
    v = np.asarray(v, np.uint32).astype(np.uint64)
    lo = ((v << 13) & 0x1FFFE000).astype(np.uint32).view(np.float32)
    hi = ((v >> 3) & 0x1FFFE000).astype(np.uint32).view(np.float32)
    return lo, hi


def test_pair_decode_matches_single_decode():
    v = np.random.default_rng(13).integers(0, 2 ** 32, 500_000, dtype=np.uint64).astype(np.uint32)
    lo, hi = decode2(v)
    for half, got in ((v & 0xFFFF, lo), (v >> 16, hi)):
        assert np.array_equal(decode(half).view(np.uint32), got.view(np.uint32))
