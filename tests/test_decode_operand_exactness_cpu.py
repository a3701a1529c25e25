"""The arithmetic facts the decode projection's tensor-core form rests on,
checked exhaustively on the CPU (numpy's float16 and float32 round to nearest
even, as the GPU's do):

* the A operand sc*q comes out exact from one fp16 fma on the pattern
  1024 + q (low nibble) or 1024 + 16q with sc/16 (high nibble), for every
  4-bit code and 6-bit scale;
* a token's int8 code x becomes the exact fp16 value through the pattern of
  (x + 128) under 0x64 less 1152, and the repeated 6-bit min through its
  byte under 0x64 less 1024;
* the integer sums stay below 2^24 (exact in fp32), and the one-token path's
  rounding of the whole integer equals the rounding of the sum of its two
  exact halves.
"""
import numpy as np

F16 = np.float16


def _fma16(a, b, c):
    """One fp16 rounding of the exact a*b + c (fp16 inputs: the product and
    the sum are exact in float64)."""
    return F16(np.float64(a) * np.float64(b) + np.float64(c))


def _half_from_bits(bits):
    return np.array([bits], dtype=np.uint16).view(np.float16)[0]


def test_pattern_1024_plus_byte():
    for b in range(256):
        assert float(_half_from_bits(0x6400 | b)) == 1024.0 + b


def test_scaled_code_operand_is_exact():
    for sc in range(64):
        s = F16(sc)
        n = F16(-1024.0 * sc)
        assert float(n) == -1024.0 * sc
        s16 = F16(sc / 16.0)
        assert float(s16) == sc / 16.0
        n16 = F16(-1024.0 * float(s16))
        assert float(n16) == -64.0 * sc
        for q in range(16):
            lo = _fma16(_half_from_bits(0x6400 | q), s, n)
            hi = _fma16(_half_from_bits(0x6400 | (q << 4)), s16, n16)
            assert float(lo) == q * sc, (q, sc)
            assert float(hi) == q * sc, (q, sc)


def test_token_code_and_min_operands_are_exact():
    for x in range(-127, 128):
        u = (x & 0xFF) ^ 0x80
        assert float(F16(np.float64(_half_from_bits(0x6400 | u)) - 1152.0)) == x
    for m in range(64):
        assert float(F16(np.float64(_half_from_bits(0x6400 | m)) - 1024.0)) == m


def test_integer_sums_stay_exact_in_fp32():
    # one k16 step of one sub-block, then one of a superblock's two halves
    # (8 sub-blocks): products sc*q*x, and the min's m*x
    step = 16 * (63 * 15) * 127
    half = 8 * step
    assert half < 2 ** 24
    assert 8 * 16 * 63 * 127 < 2 ** 24
    # the one-token path's integers: 16 * S over the 8 sub-block lanes fits int32
    assert 16 * 2 * half < 2 ** 31


def test_rounding_the_whole_equals_rounding_the_sum_of_exact_halves():
    rng = np.random.default_rng(3)
    limit = 8 * 16 * 945 * 127
    a = rng.integers(-limit, limit + 1, size=200000)
    b = rng.integers(-limit, limit + 1, size=200000)
    a[:4] = [limit, -limit, limit, 2 ** 24 - 1]
    b[:4] = [limit, -limit, limit - 1, 3]
    fa, fb = a.astype(np.float32), b.astype(np.float32)
    assert np.array_equal(fa.astype(np.int64), a) and np.array_equal(fb.astype(np.int64), b)
    whole = (a + b).astype(np.float32)
    assert np.array_equal(fa + fb, whole)
    # and scaling by 16 commutes with the rounding
    assert np.array_equal(((a + b) * 16).astype(np.float32), whole * np.float32(16))
