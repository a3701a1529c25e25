"""Pins for the oracle's causal grouped-query attention: closed forms,
element-by-element brute force, and the invariants of the definition."""
import math

import numpy as np
import pytest

from oracle import attention as OA


def test_first_query_returns_first_value():
    """The first position sees only key 0: its output is v_0 whatever q, k."""
    rng = np.random.default_rng(0)
    q, k, v = (rng.normal(size=(5, 4, 8)) for _ in range(3))
    k = k[:, :2]
    v = v[:, :2]
    o = OA.attention(q, k, v)
    for h in range(4):
        assert np.allclose(o[0, h], v[0, h // 2], atol=1e-14)


def test_equal_keys_give_running_mean():
    """All keys equal: every allowed score is the same, so o_i is the mean of
    v_0 .. v_i (a closed form)."""
    rng = np.random.default_rng(1)
    q = rng.normal(size=(6, 2, 4))
    k = np.tile(rng.normal(size=(1, 1, 4)), (6, 1, 1))
    v = rng.normal(size=(6, 1, 4))
    o = OA.attention(q, k, v)
    for i in range(6):
        assert np.allclose(o[i, 0], v[: i + 1, 0].mean(0), atol=1e-13)
        assert np.allclose(o[i, 1], v[: i + 1, 0].mean(0), atol=1e-13)


def test_brute_force_elementwise():
    """Scores, softmax and weighted sums written out with Python loops."""
    rng = np.random.default_rng(2)
    nq, nk, hq, hkv, d = 3, 5, 4, 2, 3
    q = rng.normal(size=(nq, hq, d))
    k = rng.normal(size=(nk, hkv, d))
    v = rng.normal(size=(nk, hkv, d))
    scale = 0.7
    o = OA.attention(q, k, v, scale)
    for i in range(nq):
        p_i = nk - nq + i
        for h in range(hq):
            g = h // (hq // hkv)
            s = [scale * sum(q[i, h, e] * k[j, g, e] for e in range(d)) for j in range(p_i + 1)]
            w = [math.exp(x) for x in s]
            tot = sum(w)
            for e in range(d):
                want = sum(w[j] * v[j, g, e] for j in range(p_i + 1)) / tot
                assert abs(o[i, h, e] - want) <= 1e-12 * max(1.0, abs(want))


def test_prefix_extend_equals_full_rows():
    """Queries that extend a held prefix equal the last rows of the full
    attention over the whole sequence (the causal definition)."""
    rng = np.random.default_rng(3)
    nk, hq, hkv, d = 40, 4, 1, 8
    q = rng.normal(size=(nk, hq, d))
    k = rng.normal(size=(nk, hkv, d))
    v = rng.normal(size=(nk, hkv, d))
    full = OA.attention(q, k, v)
    tail = OA.attention(q[25:], k, v)
    assert np.allclose(tail, full[25:], atol=1e-13)


def test_grouped_heads_equal_repeated_heads():
    """Grouped key/value heads act as if each were repeated for its query heads."""
    rng = np.random.default_rng(4)
    q = rng.normal(size=(7, 6, 4))
    k = rng.normal(size=(7, 2, 4))
    v = rng.normal(size=(7, 2, 4))
    o = OA.attention(q, k, v)
    o_rep = OA.attention(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1))
    assert np.allclose(o, o_rep, atol=1e-14)


def test_planted_mask_off_by_one_is_caught():
    """Letting a query see the next key must break the first-query pin."""
    def leaky(q, k, v, scale=None):
        return OA.attention(q[1:], k, v, scale)[[0] * q.shape[0]] if q.shape[0] > 1 else OA.attention(q, k, v, scale)
    rng = np.random.default_rng(5)
    q, k, v = (rng.normal(size=(5, 1, 8)) for _ in range(3))
    with pytest.raises(AssertionError):
        assert np.allclose(leaky(q, k, v)[0, 0], v[0, 0], atol=1e-14)
