"""Pins of the decode-step attention oracle (oracle.attention_decode): one
query per sequence, at position lens[b] - 1, over a KV cache.

Pinned against closed forms and a loop-only scalar restatement, not against
the oracle's own prefill attention: a single visible key returns its value
row; a zero query averages the visible value rows; cache entries past
lens[b] do not matter; ALiBi with zero slopes is plain attention and ALiBi
(-slope (i - j)) weights key j by e^{slope j} relative to plain scores."""
import math

import numpy as np
import pytest

import oracle

rng = np.random.default_rng(7)


def _case(B=3, H=4, Hk=2, S=40, d=16):
    q = rng.standard_normal((B, H, d))
    k = rng.standard_normal((B, Hk, S, d))
    v = rng.standard_normal((B, Hk, S, d))
    return q, k, v


def _loop_decode(q, k, v, lens, scale, slopes=None):
    """Scalar loops, math.exp, no NumPy arithmetic."""
    B, H, d = q.shape
    Hk = k.shape[1]
    out = [[[0.0] * d for _ in range(H)] for _ in range(B)]
    for b in range(B):
        n = int(lens[b])
        for h in range(H):
            g = h // (H // Hk)
            sc = []
            for j in range(n):
                t = sum(float(q[b, h, c]) * float(k[b, g, j, c]) for c in range(d)) * scale
                if slopes is not None:
                    t -= float(slopes[h]) * ((n - 1) - j)
                sc.append(t)
            m = max(sc)
            e = [math.exp(t - m) for t in sc]
            z = sum(e)
            for c in range(d):
                out[b][h][c] = sum(e[j] * float(v[b, g, j, c]) for j in range(n)) / z
    return np.array(out)


def test_single_key_returns_its_value_row():
    q, k, v = _case()
    o = oracle.attention_decode(q, k, v, lens=[1, 1, 1])
    for b in range(3):
        for h in range(4):
            np.testing.assert_array_equal(o[b, h], v[b, h // 2, 0])


def test_zero_query_averages_visible_values():
    q, k, v = _case()
    lens = [5, 17, 40]
    o = oracle.attention_decode(np.zeros_like(q), k, v, lens)
    for b, n in enumerate(lens):
        for h in range(4):
            np.testing.assert_allclose(o[b, h], v[b, h // 2, :n].mean(axis=0), rtol=0, atol=1e-14)


def test_entries_past_the_length_do_not_matter():
    q, k, v = _case()
    lens = [3, 20, 33]
    o = oracle.attention_decode(q, k, v, lens)
    k2, v2 = k.copy(), v.copy()
    for b, n in enumerate(lens):
        k2[b, :, n:] = 1e6
        v2[b, :, n:] = np.nan
    np.testing.assert_array_equal(oracle.attention_decode(q, k2, v2, lens), o)


def test_matches_scalar_loops():
    q, k, v = _case(B=2, H=4, Hk=1, S=9, d=5)
    lens = [4, 9]
    np.testing.assert_allclose(oracle.attention_decode(q, k, v, lens),
                               _loop_decode(q, k, v, lens, 5 ** -0.5), rtol=0, atol=1e-13)


def test_alibi_zero_slopes_and_key_weights():
    q, k, v = _case(B=2, H=4, Hk=4, S=12, d=8)
    lens = [7, 12]
    plain = oracle.attention_decode(q, k, v, lens)
    np.testing.assert_array_equal(oracle.attention_decode(q, k, v, lens, slopes=np.zeros(4)),
                                  plain)
    slopes = oracle.alibi_slopes(4)
    np.testing.assert_allclose(oracle.attention_decode(q, k, v, lens, slopes=slopes),
                               _loop_decode(q, k, v, lens, 8 ** -0.5, slopes), rtol=0, atol=1e-13)


def test_rejects_bad_lengths():
    q, k, v = _case()
    with pytest.raises(ValueError):
        oracle.attention_decode(q, k, v, lens=[0, 3, 3])
    with pytest.raises(ValueError):
        oracle.attention_decode(q, k, v, lens=[41, 3, 3])
