"""The 16-bit chunk-bin encoding of the scoring kernels (bin_encode / bin_decode in common.cuh).

The kernels store each chunk bin (a sum of 2^(t - R) >= 0 over one chunk) as an
unsigned 16-bit float: 6 exponent bits, 10 mantissa bits, exponent field 87 of
fp32 as code exponent 0, rounding half up at the 11th significant bit, code 0
= zero.  The same integer steps replayed in numpy must keep the relative error
within 2^-11 over [2^-40, 2^24), flush below 2^-40 and stay monotone: the
chunk-score tolerance 1e-3 relative rests on it.
"""
import numpy as np

BIAS = 87


def encode(b):
    u = np.asarray(b, np.float32).view(np.uint32).astype(np.int64)
    code = ((u + 0x1000) >> 13) - (BIAS << 10)
    return np.clip(code, 0, 0xFFFF).astype(np.uint32)


def decode(code):
    code = np.asarray(code, np.uint32).astype(np.uint64)
    bits = ((code + (BIAS << 10)) << 13).astype(np.uint32)
    return np.where(code == 0, np.float32(0), bits.view(np.float32))


def test_relative_error_over_the_range():
    rng = np.random.default_rng(5)
    x = (2.0 ** rng.uniform(-39.9, 23.99, 1_000_000)).astype(np.float32)
    y = decode(encode(x)).astype(np.float64)
    rel = np.abs(y / x.astype(np.float64) - 1.0)
    assert rel.max() <= 2.0 ** -11 * (1 + 1e-6)


def test_zero_flush_and_saturation():
    assert decode(encode(np.float32(0.0))) == 0.0
    assert decode(encode(np.float32(2.0 ** -41))) == 0.0
    top = decode(np.uint32(0xFFFF))
    assert 2.0 ** 23 < top < 2.0 ** 24
    assert decode(encode(np.float32(2.0 ** 30))) == top


def test_monotone_and_exact_on_short_mantissas():
    x = np.sort((2.0 ** np.random.default_rng(9).uniform(-39, 23, 200_000)).astype(np.float32))
    y = decode(encode(x))
    assert np.all(np.diff(y) >= 0)
    z = (np.arange(1, 1024, dtype=np.float32) / 1024 + 1) * np.float32(2.0 ** -7)     # 10-bit mantissas
    assert np.array_equal(decode(encode(z)), z)


def encode_bounded(b):
    """The tensor-core kernel's encoder for bins at most 2^23: bias folded into the rounding add,
    arithmetic shift, one clamp at zero."""
    u = np.asarray(b, np.float32).view(np.uint32).astype(np.int64)
    return np.maximum((u + (0x1000 - (BIAS << 23))) >> 13, 0).astype(np.uint32)     # numpy >> floors


def test_bounded_encoder_matches_up_to_2_23():
    rng = np.random.default_rng(11)
    x = np.concatenate([(2.0 ** rng.uniform(-45, 23, 1_000_000)).astype(np.float32),
                        np.float32([0.0, 2.0 ** -40, 2.0 ** -41, 2.0 ** 23, 2.0 ** 23 * 0.9999])])
    assert np.array_equal(encode_bounded(x), encode(x))
    assert encode_bounded(np.float32(2.0 ** 23)).item() < 0xFFFF


def decode2(v):
    """The finalisation's decode of two bins packed in a 32-bit word (code 0 reads as 2^-40)."""
    v = np.asarray(v, np.uint32).astype(np.uint64)
    lo = (((v << 13) & 0x1FFFE000) + (BIAS << 23)).astype(np.uint32).view(np.float32)
    hi = (((v >> 3) & 0x1FFFE000) + (BIAS << 23)).astype(np.uint32).view(np.float32)
    return lo, hi


def test_pair_decode_matches_single_decode():
    v = np.random.default_rng(13).integers(0, 2 ** 32, 500_000, dtype=np.uint64).astype(np.uint32)
    lo, hi = decode2(v)
    for half, got in ((v & 0xFFFF, lo), (v >> 16, hi)):
        want = decode(half)
        assert np.array_equal(np.where(half == 0, np.float32(2.0 ** -40), want), got)
