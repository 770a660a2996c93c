"""Oracle pins: the whole block, every variant.

Block equations: nnterp "stablelm" 03 Notes ("The block is sequential on 1.6B
and 3B, parallel on 12B"; "The contributions are the modules' outputs"),
"OLMo-2: reordered (post) normalization" section 1, "Bloom in a sovereign
engine" Contribution (rotary gated off for ALiBi).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import brute
from workloads import BLOCK_CONFIGS, scaled

TINY = dict(batch=2, seq=5, hidden=8, n_heads=2, n_kv_heads=2, head_dim=4, intermediate=6)

VARIANTS = {
    "stablelm_r0": scaled(BLOCK_CONFIGS["tiny_stablelm2"], rotary_span=0, **TINY),
    "stablelm_r2": scaled(BLOCK_CONFIGS["tiny_stablelm2"], rotary_span=2, **TINY),
    "stablelm_r4": scaled(BLOCK_CONFIGS["tiny_stablelm2"], rotary_span=4, **TINY),
    "bloom": scaled(BLOCK_CONFIGS["bloom_560m"], **TINY),
    "olmo2": scaled(BLOCK_CONFIGS["olmo2_1b"], rotary_span=4, **TINY),
    "stablelm12b": scaled(BLOCK_CONFIGS["stablelm2_12b"], rotary_span=2,
                          **dict(TINY, n_heads=4, n_kv_heads=2)),
}


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_block_matches_loop_only_brute_force(name):
    cfg = VARIANTS[name]
    x, w = workloads.block_inputs(cfg)
    w = {k: (t * 25 if k in ("w_qkv", "w_o", "w_up", "w_gate", "w_down") else t)
         for k, t in w.items()}  # weights large enough that every term moves y
    ref = np.array(brute.block(cfg, x, w))
    y = oracle.block_forward(cfg, x, w)["y"]
    np.testing.assert_allclose(y, ref, rtol=0, atol=1e-12)


def _cfg_inputs(base, **kw):
    cfg = scaled(BLOCK_CONFIGS[base], **dict(dict(batch=2, seq=16, hidden=64, n_heads=4,
                                                  n_kv_heads=4, head_dim=16,
                                                  intermediate=96), **kw))
    x, w = workloads.block_inputs(cfg)
    return cfg, x, w


def test_sequential_identities():
    """post_attention_layernorm.input == x + attention_output; y == h + mlp_output."""
    cfg, x, w = _cfg_inputs("tiny_stablelm2", rotary_span=4)
    r = oracle.block_forward(cfg, x, w)
    xs = oracle.as_f64(x)
    np.testing.assert_array_equal(r["h"], xs + r["attn_out"])
    np.testing.assert_array_equal(r["y"], r["h"] + r["mlp_out"])
    np.testing.assert_allclose(r["n2"], oracle.layer_norm(r["h"], oracle.as_f64(w["mlp_norm_w"]),
                                                          oracle.as_f64(w["mlp_norm_b"]), 1e-5),
                               atol=0)


def test_parallel_identity():
    """x + attention_output + mlp_output == layer_output (12B shape)."""
    cfg, x, w = _cfg_inputs("stablelm2_12b", n_kv_heads=2, rotary_span=4)
    r = oracle.block_forward(cfg, x, w)
    np.testing.assert_array_equal(r["y"], oracle.as_f64(x) + r["attn_out"] + r["mlp_out"])
    assert r["n2"] is r["n1"]      # both sublayers read the one input norm


def test_post_norm_placement():
    """OLMo-2: the post norms act on sublayer outputs before the add, so
    (y - h) / w_post has unit RMS per row (up to eps)."""
    cfg, x, w = _cfg_inputs("olmo2_1b", rotary_span=16)
    r = oracle.block_forward(cfg, x, w)
    z = (r["y"] - r["h"]) / oracle.as_f64(w["post_mlp_norm_w"])
    ms = (r["mlp_out"] ** 2).mean(-1)
    np.testing.assert_allclose((z ** 2).mean(-1), (ms / (ms + cfg.eps)).reshape(z.shape[:-1]),
                               rtol=1e-9)
    # no input norm: the projections read raw x
    np.testing.assert_array_equal(r["n1"], oracle.as_f64(x))
    # negative control: the same weights in pre-norm order give another block
    pre = scaled(cfg, norm_place="pre")
    w_pre = dict(w, attn_norm_w=w["post_attn_norm_w"], mlp_norm_w=w["post_mlp_norm_w"])
    assert not np.allclose(oracle.block_forward(pre, x, w_pre)["y"], r["y"], atol=1e-3)


def test_full_width_qk_norm_is_not_per_head():
    cfg, x, w = _cfg_inputs("olmo2_1b", rotary_span=0)
    r = oracle.block_forward(cfg, x, w)
    qf = r["q"].transpose(0, 2, 1, 3).reshape(2, 16, -1) / oracle.as_f64(w["q_norm_w"])
    np.testing.assert_allclose((qf ** 2).mean(-1), 1.0, atol=1e-4)
    per_head = r["q"] / oracle.as_f64(w["q_norm_w"]).reshape(4, 16)[None, :, None]
    assert not np.allclose((per_head ** 2).mean(-1), 1.0, atol=1e-3)


def test_rotary_pass_through_equals_projection():
    """Queries past the span equal q_proj's output split into heads (nnterp stablelm 03 Notes)."""
    cfg, x, w = _cfg_inputs("tiny_stablelm2", rotary_span=4)
    r = oracle.block_forward(cfg, x, w)
    proj = oracle.linear(r["n1"], oracle.as_f64(w["w_qkv"]), oracle.as_f64(w["b_qkv"]))
    qh = oracle.split_heads(proj[..., :64], 4, 16)
    np.testing.assert_array_equal(r["q"][..., 4:], qh[..., 4:])
    assert not np.array_equal(r["q"][..., 1:, :4], qh[..., 1:, :4])


def test_per_head_qk_layernorm_before_rotary():
    cfg, x, w = _cfg_inputs("stablelm2_12b", n_kv_heads=2, rotary_span=4)
    r = oracle.block_forward(cfg, x, w)
    g = oracle.as_f64(w["k_norm_w"])                       # [Hk, d]
    past = r["k"][..., 4:] / g[None, :, None, 4:]
    # past the span the keys are a bias-free LayerNorm output: no shift added
    proj = oracle.linear(r["n1"], oracle.as_f64(w["w_qkv"]))
    kh = oracle.split_heads(proj[..., 64:64 + 32], 2, 16)
    ref = oracle.layer_norm(kh, np.ones(16), None, cfg.qk_norm_eps)
    np.testing.assert_allclose(past, ref[..., 4:], atol=1e-12)


def test_slots_each_matter_and_are_independent():
    """Every named weight slot moves y; the two norm slots are read
    independently (the OLMo-2 loader-clobber lesson)."""
    for base, kw in (("tiny_stablelm2", dict(rotary_span=4)), ("olmo2_1b", dict(rotary_span=4)),
                     ("bloom_560m", {}), ("stablelm2_12b", dict(n_kv_heads=2, rotary_span=4))):
        cfg, x, w = _cfg_inputs(base, **kw)
        y0 = oracle.block_forward(cfg, x, w)
        for name in w:
            w2 = dict(w)
            w2[name] = w[name] + 0.25
            y1 = oracle.block_forward(cfg, x, w2)
            assert not np.allclose(y1["y"], y0["y"], atol=1e-9), (base, name)
            if name in ("mlp_norm_w", "mlp_norm_b", "post_mlp_norm_w"):
                if y0["h"] is not None:   # sequential: only the MLP half moves
                    np.testing.assert_array_equal(y1["h"], y0["h"])


def test_alibi_with_rotary_off_is_finite_and_rotary_alibi_rejected():
    cfg, x, w = _cfg_inputs("bloom_560m")
    y = oracle.block_forward(cfg, x, w)["y"]
    assert np.isfinite(y).all()
    with pytest.raises(ValueError):
        oracle.block_forward(scaled(cfg, rotary_span=4), x, w)


def test_block_causality():
    cfg, x, w = _cfg_inputs("tiny_stablelm2", rotary_span=4)
    y0 = oracle.block_forward(cfg, x, w)["y"]
    x2 = x.clone()
    gen = torch.Generator().manual_seed(5)
    x2[:, 9:] = torch.randn(x2[:, 9:].shape, generator=gen, dtype=torch.float64).to(x2.dtype)
    y1 = oracle.block_forward(cfg, x2, w)["y"]
    np.testing.assert_array_equal(y0[:, :9], y1[:, :9])


@pytest.mark.parametrize("base", ["tiny_stablelm2", "bloom_560m", "olmo2_1b", "stablelm2_12b"])
def test_sampled_rows_match_full(base):
    kw = {"stablelm2_12b": dict(n_kv_heads=2, rotary_span=4),
          "olmo2_1b": dict(rotary_span=16)}.get(base, {})
    cfg, x, w = _cfg_inputs(base, **kw)
    full = oracle.block_forward(cfg, x, w)
    rows = np.array([0, 3, 15, 16, 20, 31])
    part = oracle.block_forward(cfg, x, w, rows=rows)
    for key in ("attn_premix", "attn_out", "mlp_out", "y"):
        np.testing.assert_allclose(part[key], full[key].reshape(32, -1)[rows], atol=1e-13)


def test_attention_forward_bias_then_rotary():
    cfg = workloads.scaled(workloads.ATTN_CONFIGS["attn_s512"], batch=1, seq=12, n_heads=2,
                           n_kv_heads=2, head_dim=8, rotary_span=4)
    q, k, v, b = workloads.attn_inputs(cfg)
    o = oracle.attention_forward(cfg, q, k, v, b)
    bq = oracle.as_f64(b[0]).reshape(2, 8)[None, :, None]
    bk = oracle.as_f64(b[1]).reshape(2, 8)[None, :, None]
    bv = oracle.as_f64(b[2]).reshape(2, 8)[None, :, None]
    pos = np.arange(12)
    ref = oracle.attention(oracle.rope(oracle.as_f64(q) + bq, pos, 4, 1e4),
                           oracle.rope(oracle.as_f64(k) + bk, pos, 4, 1e4), oracle.as_f64(v) + bv)
    np.testing.assert_array_equal(o, ref)
    rows = np.array([0, 7, 11])
    np.testing.assert_allclose(oracle.attention_forward(cfg, q, k, v, b, rows=rows),
                               ref[:, :, rows], atol=1e-14)
