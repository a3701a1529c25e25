"""Pins for the oracle's int8 row quantisation, exact integer product, fp32 rescale and bf16 rounding."""
import numpy as np
import pytest

from oracle import quant


def check_quant_rows(fn):
    rng = np.random.default_rng(5)
    w = rng.normal(0, 1, size=(16, 300)).astype(np.float32)
    w[3] *= 1e-6
    q, s = fn(w)
    assert q.dtype == np.int8 and s.dtype == np.float32
    # scale is amax / 127 and the row maximum lands on +-127
    amax = np.abs(w).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(127)).astype(np.float32))
    idx = np.abs(w).argmax(axis=1)
    assert np.all(np.abs(q[np.arange(16), idx]) == 127)
    # reconstruction error at most half a step (plus fp32 rounding of w / s)
    err = np.abs(w.astype(np.float64) - s[:, None].astype(np.float64) * q)
    assert np.all(err <= s[:, None] * (0.5 + 1e-6))
    # brute force on a few rows: every code is the nearest of -127..127
    cand = np.arange(-127, 128, dtype=np.float64)
    for r in (0, 3, 9):
        for i in range(0, 300, 7):
            e = np.abs(cand * float(s[r]) - float(w[r, i]))
            assert e[int(q[r, i]) + 127] <= e.min() + 1e-6 * float(s[r])


def check_quant_ties_and_zero(fn):
    # amax = 127 -> s = 1 exactly: codes are the nearest-even integers
    w = np.array([[127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 1.5, 126.5]], np.float32)
    q, s = fn(w)
    assert s[0] == 1.0
    assert list(q[0]) == [127, 2, 4, -2, 0, 0, 2, 126]
    q, s = fn(np.zeros((2, 8), np.float32))
    assert np.all(q == 0) and np.all(s == 0)


@pytest.mark.parametrize("check", [check_quant_rows, check_quant_ties_and_zero])
def test_quant_pins(check):
    check(quant.quant_rows_i8)


def test_planted_truncation_is_caught():
    """Quantisation that truncates instead of rounding must fail a pin."""
    def trunc(w):
        q, s = quant.quant_rows_i8(w)
        r = np.trunc(w / np.where(s > 0, s, 1)[:, None])
        return np.clip(r, -127, 127).astype(np.int8), s
    with pytest.raises(AssertionError):
        check_quant_ties_and_zero(trunc)


def _brute_int_matmul(a, b):
    m, k = a.shape
    n = b.shape[0]
    out = np.zeros((m, n), np.int64)
    for i in range(m):
        for j in range(n):
            acc = 0
            for t in range(k):
                acc += int(a[i, t]) * int(b[j, t])
            out[i, j] = acc
    return out


def test_int_matmul_matches_python_integers():
    rng = np.random.default_rng(1)
    a = rng.integers(-127, 128, size=(5, 37)).astype(np.int8)
    b = rng.integers(-127, 128, size=(6, 37)).astype(np.int8)
    assert np.array_equal(quant.int_matmul_exact(a, b), _brute_int_matmul(a, b))


def test_int_matmul_exact_beyond_fp32_range():
    # all codes 127 over K = 4096: 4096 * 16129 = 66,064,384 > 2^24
    a = np.full((2, 4096), 127, np.int8)
    b = np.full((3, 4096), 127, np.int8)
    b[1] = -127
    b[2, ::2] = -127
    acc = quant.int_matmul_exact(a, b)
    assert acc[0, 0] == 66064384 and acc[0, 1] == -66064384 and acc[0, 2] == 0


def test_rescale_rounding():
    acc = np.array([[3, 2 ** 24 + 1, -(2 ** 24 + 3)]], np.int64)
    sa = np.array([0.5], np.float32)
    sb = np.array([0.25, 1.0, 1.0], np.float32)
    y = quant.rescale(acc, sa, sb)
    # 3 * 0.5 * 0.25 = 0.375; 2^24 + 1 -> 2^24 (tie to even); -(2^24 + 3) -> -(2^24 + 4)
    assert y[0, 0] == 0.375
    assert y[0, 1] == np.float32(2 ** 23)
    assert y[0, 2] == np.float32(-(2 ** 24 + 4) / 2)


def test_bf16_round_closed_forms():
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -20, -(1 + 2 ** -8), 3.0e38, 1.0], np.float32)
    r = quant.bf16_round(x)
    assert r[0] == 1.0                       # halfway -> even mantissa
    assert r[1] == 1 + 2 ** -6               # halfway -> even (mantissa 2)
    assert r[2] == 1 + 2 ** -7               # above halfway -> up
    assert r[3] == -1.0
    assert abs(float(r[4]) - 3.0e38) <= 2 ** -8 * 3.0e38     # within half a bf16 step
    assert r[5] == 1.0
    # every result has its low 16 bits clear
    assert np.all((r.view(np.uint32) & 0xFFFF) == 0)


# ------------------------------------------------- decode-step product (exact weights)

def test_matvec_exact_weights_brute_force():
    """Element by element against Python's exact rationals on a tiny case,
    with Q4_K-decoded weights (fp32 values, exact as fractions)."""
    from fractions import Fraction
    from oracle import q4k
    rng = np.random.default_rng(4)
    w = q4k.unpack_q4k(q4k.pack_q4k(rng.normal(0, 0.02, size=(3, 256)).astype(np.float32)), 3, 256)
    qa, sa = quant.quant_rows_i8(rng.normal(0, 1, size=(2, 256)).astype(np.float32))
    got = quant.matvec_exact_weights(qa, sa, w)
    for m in range(2):
        for n in range(3):
            exact = Fraction(float(sa[m])) * sum(Fraction(int(qa[m, k])) * Fraction(float(w[n, k])) for k in range(256))
            assert abs(Fraction(float(got[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)


def test_matvec_exact_weights_closed_form_and_bound():
    """Constant weight rows give s * c * sum(q); against the prefill's product
    (weights re-quantised to int8 rows) the difference is bounded by the
    weights' half-step: |y_exact - y_q8| <= s_x * sum|q_x| * s_w / 2 (+ fp32 rounding)."""
    rng = np.random.default_rng(8)
    qa, sa = quant.quant_rows_i8(rng.normal(0, 1, size=(4, 512)).astype(np.float32))
    w = np.full((2, 512), 0.375, np.float32)
    w[1] = -0.0625
    y = quant.matvec_exact_weights(qa, sa, w)
    for m in range(4):
        tot = int(qa[m].astype(np.int64).sum())
        assert y[m, 0] == float(sa[m]) * 0.375 * tot
        assert y[m, 1] == float(sa[m]) * -0.0625 * tot
    wr = rng.normal(0, 0.02, size=(64, 512)).astype(np.float32)
    qw, sw = quant.quant_rows_i8(wr)
    ye = quant.matvec_exact_weights(qa, sa, wr)
    yq = quant.gemm_q8(qa, sa, qw, sw).astype(np.float64)
    bound = sa[:, None].astype(np.float64) * np.abs(qa).astype(np.float64).sum(1)[:, None] * sw[None, :] / 2
    assert np.all(np.abs(ye - yq) <= bound * (1 + 1e-6) + 1e-6 * np.abs(ye))
    assert np.any(ye != yq)        # the two products really differ
