"""Oracle pins: partial NeoX split-half rotary.

"StableLM-2: partial RoPE ..." section 1 (span 16 of 64, NeoX split-half,
other dims pass through) and section 4 (full-RoPE negative control);
nnterp "stablelm" 03 Notes "Rotary turns a quarter of each head" (two halves
of 8; dims past 16 equal q_proj's output; rope_theta 10000).
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from workloads import BLOCK_CONFIGS, scaled


def _x(shape, seed=0):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


def test_span_zero_is_identity():
    x = _x((2, 3, 7, 64))
    np.testing.assert_array_equal(oracle.rope(x, np.arange(7), 0, 1e4), x)


def test_position_zero_is_identity():
    x = _x((1, 2, 1, 64))
    np.testing.assert_array_equal(oracle.rope(x, np.array([0]), 16, 1e4), x)


@pytest.mark.parametrize("r", [2, 16, 40, 64])
def test_dims_past_span_are_bitwise_untouched(r):
    x = _x((1, 2, 9, 160 if r == 40 else 64), seed=r)
    y = oracle.rope(x, np.arange(9), r, 1e4)
    np.testing.assert_array_equal(y[..., r:], x[..., r:])


@pytest.mark.parametrize("r", [16, 64, 128])
def test_rotation_preserves_pair_norms(r):
    x = _x((1, 1, 33, 128), seed=1)
    y = oracle.rope(x, np.arange(33) * 97, r, 5e5)
    h = r // 2
    np.testing.assert_allclose(y[..., :h] ** 2 + y[..., h:r] ** 2,
                               x[..., :h] ** 2 + x[..., h:r] ** 2, rtol=1e-12)


def test_closed_form_single_pair():
    """r = 2: theta_0 = 1, so (1, 0) at position p turns into (cos p, sin p)."""
    x = np.zeros((1, 1, 6, 4))
    x[..., 0] = 1.0
    y = oracle.rope(x, np.arange(6), 2, 10000.0)
    for p in range(6):
        assert y[0, 0, p, 0] == pytest.approx(math.cos(p), abs=1e-15)
        assert y[0, 0, p, 1] == pytest.approx(math.sin(p), abs=1e-15)
        assert y[0, 0, p, 2] == 0.0 and y[0, 0, p, 3] == 0.0


def test_frequency_uses_the_span_and_pairs_split_half():
    """Pairs are (j, j + r/2) (split-half, not interleaved) and theta_j = base^(-2j/r)."""
    r, base, p = 4, 100.0, 3
    x = np.zeros((1, 1, p + 1, 8))
    x[..., 1] = 1.0                      # second pair: (1, 1 + r/2 = 3)
    y = oracle.rope(x, np.arange(p + 1), r, base)[0, 0, p]
    ang = p * base ** (-2.0 * 1 / r)     # = p / 10
    assert y[1] == pytest.approx(math.cos(ang), abs=1e-15)
    assert y[3] == pytest.approx(math.sin(ang), abs=1e-15)
    assert y[0] == y[2] == 0.0 and np.all(y[4:] == 0.0)


def test_relative_position_invariance():
    """<R_m q, R_n k> depends only on m - n."""
    q = _x((1, 1, 1, 64), seed=2)
    k = _x((1, 1, 1, 64), seed=3)

    def score(m, n):
        qm = oracle.rope(np.repeat(q, m + 1, axis=2), np.arange(m + 1), 16, 1e4)[0, 0, m]
        kn = oracle.rope(np.repeat(k, n + 1, axis=2), np.arange(n + 1), 16, 1e4)[0, 0, n]
        return float(qm @ kn)

    assert score(9, 4) == pytest.approx(score(25, 20), rel=1e-12)
    assert score(3, 3) == pytest.approx(score(0, 0), rel=1e-12)


def test_rejects_odd_or_oversized_span():
    with pytest.raises(ValueError):
        oracle.rope(np.zeros((1, 1, 2, 8)), np.arange(2), 3, 1e4)
    with pytest.raises(ValueError):
        oracle.rope(np.zeros((1, 1, 2, 8)), np.arange(2), 10, 1e4)


def _row_cos(a, b):
    a = a.reshape(-1, a.shape[-1])
    b = b.reshape(-1, b.shape[-1])
    return (a * b).sum(-1) / np.linalg.norm(a, axis=-1) / np.linalg.norm(b, axis=-1)


def test_negative_control_full_span_diverges():
    """Rotating the whole head instead of the first 16 dims changes the block
    output ("StableLM-2 ..." section 4, full-RoPE control). Only divergence is
    pinned; the page's -0.62 was measured on real weights and logits."""
    cfg = scaled(BLOCK_CONFIGS["tiny_stablelm2"], seq=64, batch=1)
    x, w = workloads.block_inputs(cfg)
    # Large activations in q/k make the position signal visible at random init.
    w = dict(w)
    w["w_qkv"] = w["w_qkv"] * 8
    good = oracle.block_forward(cfg, x, w)["attn_out"]
    bad = oracle.block_forward(scaled(cfg, rotary_span=64), x, w)["attn_out"]
    assert _row_cos(good, bad).min() < 0.999
    same = oracle.block_forward(scaled(cfg, rotary_span=16), x, w)["attn_out"]
    np.testing.assert_array_equal(good, same)
