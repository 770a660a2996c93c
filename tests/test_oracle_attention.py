"""Oracle pins: causal attention, ALiBi, GQA.

nnterp "stablelm" 03 Notes (query scale head_dim^-0.5; no window, softcap or
sink, eager == sdpa; GQA on 12B), "Bloom in a sovereign engine" Contribution
(ALiBi: per-head geometric slope, linear pre-softmax bias).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _x(shape, seed=0):
    return np.random.Generator(np.random.PCG64(seed)).standard_normal(shape)


def _qkv(B=2, H=4, Hk=4, S=19, d=8, seed=0):
    return _x((B, H, S, d), seed), _x((B, Hk, S, d), seed + 1), _x((B, Hk, S, d), seed + 2)


def test_causal_rows_sum_to_one_and_mask_upper_triangle():
    q, k, v = _qkv()
    _, p = oracle.attention(q, k, v, return_probs=True)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-13)
    iu = np.triu_indices(p.shape[-1], 1)
    assert np.all(p[..., iu[0], iu[1]] == 0.0)


def test_first_row_is_first_value_exactly():
    q, k, v = _qkv(seed=3)
    o = oracle.attention(q, k, v)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0])


def test_zero_queries_give_running_mean():
    """q = 0 makes every score 0: row i averages v_0..v_i (closed form)."""
    _, k, v = _qkv(seed=5)
    q = np.zeros((2, 4, 19, 8))
    o = oracle.attention(q, k, v)
    running = np.cumsum(v, axis=2) / np.arange(1, 20)[None, None, :, None]
    np.testing.assert_allclose(o, running, atol=1e-13)


def test_causality_future_keys_do_not_matter():
    q, k, v = _qkv(seed=7)
    o1 = oracle.attention(q, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 11:] += 5.0
    v2[:, :, 11:] -= 3.0
    o2 = oracle.attention(q, k2, v2)
    np.testing.assert_array_equal(o1[:, :, :11], o2[:, :, :11])
    assert not np.allclose(o1[:, :, 11:], o2[:, :, 11:])


@pytest.mark.parametrize("alibi", [False, True])
def test_matches_torch_sdpa_float64(alibi):
    q, k, v = _qkv(S=23, d=16, seed=11)
    S = 23
    slopes = oracle.alibi_slopes(4) if alibi else None
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    mask = np.where(j > i, -np.inf, 0.0)[None, None].repeat(4, axis=1)
    if alibi:
        mask = mask - slopes[None, :, None, None] * (i - j)[None, None]
    ref = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                         torch.from_numpy(v), attn_mask=torch.from_numpy(mask))
    np.testing.assert_allclose(oracle.attention(q, k, v, slopes=slopes), ref.numpy(),
                               rtol=0, atol=1e-12)


def test_scale_is_inverse_sqrt_head_dim():
    q, k, v = _qkv(d=16, seed=13)
    np.testing.assert_allclose(oracle.attention(q, k, v),
                               oracle.attention(q, k, v, scale=0.25), atol=0)
    assert not np.allclose(oracle.attention(q, k, v), oracle.attention(q, k, v, scale=1.0))


def test_gqa_equals_mha_with_replicated_kv():
    """kv head j serves query heads j*H/Hk .. (j+1)*H/Hk - 1 (nnterp stablelm, GQA on 12B)."""
    q, k, v = _qkv(H=8, Hk=2, seed=17)
    ref = oracle.attention(q, np.repeat(k, 4, axis=1), np.repeat(v, 4, axis=1))
    np.testing.assert_allclose(oracle.attention(q, k, v), ref, atol=0)


def test_alibi_slopes_closed_form():
    np.testing.assert_array_equal(oracle.alibi_slopes(16), 2.0 ** (-0.5 * (np.arange(16) + 1)))
    np.testing.assert_array_equal(oracle.alibi_slopes(8), 2.0 ** -(np.arange(8) + 1.0))
    s = oracle.alibi_slopes(32)
    np.testing.assert_allclose(s[1:] / s[:-1], 2.0 ** (-8 / 32), rtol=1e-15)
    assert s[0] == 2.0 ** (-0.25)
    with pytest.raises(ValueError):
        oracle.alibi_slopes(12)


def test_zero_slopes_reduce_to_plain_attention():
    q, k, v = _qkv(seed=19)
    np.testing.assert_array_equal(oracle.attention(q, k, v, slopes=np.zeros(4)),
                                  oracle.attention(q, k, v))


def test_alibi_relative_form_equals_key_position_form():
    """-slope (i - j) and +slope j differ by a per-row constant: same softmax."""
    q, k, v = _qkv(S=17, seed=23)
    slopes = oracle.alibi_slopes(4)
    S = 17
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    mask = np.where(j > i, -np.inf, 0.0)[None, None] + slopes[None, :, None, None] * j[None, None]
    ref = F.scaled_dot_product_attention(torch.from_numpy(q), torch.from_numpy(k),
                                         torch.from_numpy(v),
                                         attn_mask=torch.from_numpy(mask.repeat(2, axis=0)))
    np.testing.assert_allclose(oracle.attention(q, k, v, slopes=slopes), ref.numpy(), atol=1e-12)


def test_alibi_closed_form_with_zero_queries():
    """q = 0: weights exp(-slope (i - j)) over j <= i."""
    _, k, v = _qkv(S=9, seed=29)
    q = np.zeros((2, 4, 9, 8))
    slopes = oracle.alibi_slopes(4)
    o = oracle.attention(q, k, v, slopes=slopes)
    b, h, i = 1, 2, 6
    wts = np.array([math.exp(-slopes[h] * (i - j)) for j in range(i + 1)])
    np.testing.assert_allclose(o[b, h, i], (wts[:, None] * v[b, h, :i + 1]).sum(0) / wts.sum(),
                               atol=1e-14)


def test_query_subset_matches_full():
    q, k, v = _qkv(S=31, seed=31)
    full = oracle.attention(q, k, v, slopes=oracle.alibi_slopes(4))
    rows = np.array([0, 5, 17, 30])
    part = oracle.attention(q[:, :, rows], k, v, slopes=oracle.alibi_slopes(4), q_positions=rows)
    np.testing.assert_allclose(part, full[:, :, rows], atol=1e-14)
