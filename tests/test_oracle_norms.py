"""Oracle pins: LayerNorm-with-bias, RMSNorm, activations.

LayerNorm with bias: "StableLM-2: partial RoPE and a first LayerNorm-with-bias
path" section 1, and nnterp "stablelm" Printout. RMSNorm: "OLMo-2: reordered
(post) normalization" section 1.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _rng(seed=0):
    return np.random.Generator(np.random.PCG64(seed))


def test_layer_norm_moments_before_affine():
    x = _rng().standard_normal((64, 200)) * 3.0 + 1.5
    eps = 1e-5
    n = oracle.layer_norm(x, np.ones(200), np.zeros(200), eps)
    var = x.var(axis=-1)
    assert np.abs(n.mean(axis=-1)).max() < 1e-12
    # population variance with eps inside the sqrt: var(n) = var / (var + eps)
    np.testing.assert_allclose(n.var(axis=-1), var / (var + eps), rtol=0, atol=1e-12)


def test_layer_norm_affine_is_elementwise():
    x = _rng(1).standard_normal((8, 32))
    g = _rng(2).standard_normal(32)
    b = _rng(3).standard_normal(32)
    n = oracle.layer_norm(x, np.ones(32), None, 1e-5)
    np.testing.assert_allclose(oracle.layer_norm(x, g, b, 1e-5), n * g + b, atol=1e-14)


def test_layer_norm_matches_torch_float64():
    x = _rng(4).standard_normal((16, 48))
    g = 1 + 0.1 * _rng(5).standard_normal(48)
    b = 0.1 * _rng(6).standard_normal(48)
    ref = F.layer_norm(torch.from_numpy(x), (48,), torch.from_numpy(g), torch.from_numpy(b), 1e-5)
    np.testing.assert_allclose(oracle.layer_norm(x, g, b, 1e-5), ref.numpy(), rtol=0, atol=1e-12)


def test_rms_norm_moment_and_torch():
    x = _rng(7).standard_normal((16, 96)) * 2.0
    eps = 1e-6
    n = oracle.rms_norm(x, np.ones(96), eps)
    ms = (x * x).mean(axis=-1)
    np.testing.assert_allclose((n * n).mean(axis=-1), ms / (ms + eps), atol=1e-12)
    w = 1 + 0.1 * _rng(8).standard_normal(96)
    ref = F.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), eps)
    np.testing.assert_allclose(oracle.rms_norm(x, w, eps), ref.numpy(), rtol=0, atol=1e-12)


def test_rms_norm_is_scale_invariant_layernorm_is_shift_invariant():
    x = _rng(9).standard_normal((4, 64))
    w = np.ones(64)
    np.testing.assert_allclose(oracle.rms_norm(5.0 * x, w, 0.0), oracle.rms_norm(x, w, 0.0), atol=1e-13)
    np.testing.assert_allclose(oracle.layer_norm(x + 3.0, w, None, 0.0),
                               oracle.layer_norm(x, w, None, 0.0), atol=1e-12)


def test_activations_match_torch_float64():
    z = np.linspace(-12, 12, 2001)
    tz = torch.from_numpy(z)
    np.testing.assert_allclose(oracle.silu(z), F.silu(tz).numpy(), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(oracle.gelu_tanh(z), F.gelu(tz, approximate="tanh").numpy(),
                               rtol=1e-14, atol=1e-15)
    # closed forms
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    assert abs(oracle.gelu_tanh(np.array([1.0]))[0]
               - 0.5 * (1 + math.tanh(math.sqrt(2 / math.pi) * 1.044715))) < 1e-15


def test_linear_convention_out_in():
    """Linear(in, out) keeps W[out, in] and y = x W^T + b (nnterp Printout)."""
    x = np.array([[1.0, 2.0, 3.0]])
    w = np.array([[1.0, 0.0, 0.0], [0.0, 0.0, 2.0]])   # out=2, in=3
    np.testing.assert_array_equal(oracle.linear(x, w, np.array([0.5, -1.0])), [[1.5, 5.0]])


@pytest.mark.parametrize("n", [1, 5])
def test_split_qkv_interleaved_order(n):
    """Head-interleaved fused QKV: output rows run [head][q, k, v][d]."""
    H, d = 2, 3
    y = np.arange(n * H * 3 * d, dtype=np.float64).reshape(1, n, H * 3 * d)
    q, k, v = oracle.split_qkv(y, H, H, d, "head_interleaved")
    # head 1's q occupies columns 9..11 (after head 0's q, k, v)
    np.testing.assert_array_equal(q[0, 0, d:2 * d], y[0, 0, 9:12])
    np.testing.assert_array_equal(k[0, 0, :d], y[0, 0, 3:6])
    np.testing.assert_array_equal(v[0, 0, d:], y[0, 0, 15:18])
    qs, ks, vs = oracle.split_qkv(y[..., :H * 3 * d], H, H, d, "stacked")
    np.testing.assert_array_equal(ks[0, 0], y[0, 0, 6:12])
