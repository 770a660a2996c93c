"""fp64 oracle of one decode step of a whole block (test infrastructure,
like the rest of ``oracle``; the CUDA path never imports it).

The pages claim prefill only ("StableLM-2 ...": NOT claimed, generation);
a decode step is the adjacent step: one new token per sequence goes through
the block while the keys and values of the earlier tokens come from a cache
that the prefill wrote. It is written in the order of ``block_forward``
(nnterp "stablelm" 03 Notes for the block equations, "OLMo-2 ..." section 1
for the post-norm placement): norm, projection (+ bias), qk-norm, rotary at
the token's own position, its k and v appended to the cache, attention over
the cache up to and including it, output projection, residual and MLP.
Pinned by equality with the prefill: a decode step after a prefill of the
first S - 1 tokens gives the prefill's output for token S - 1.
"""
from __future__ import annotations

import numpy as np

from .block import (alibi_slopes, as_f64, attention_decode, layer_norm, linear, mlp,
                    qk_norm_full_rms, qk_norm_per_head_ln, rms_norm, rope, split_heads, split_qkv)


def block_decode_step(cfg, x_t, weights, k_cache, v_cache, lens):
    """x_t [B, D]: each sequence's new token, at position lens[b]; k_cache,
    v_cache [B, Hk, S_max, d] hold positions 0 .. lens[b] - 1 (after qk-norm
    and rotary, as the prefill leaves them). Returns (y_t [B, D], k_cache,
    v_cache) with the new token's key and value written at lens[b] (copies;
    the inputs are left unchanged)."""
    w = {kname: as_f64(t) for kname, t in weights.items()}
    x_t = as_f64(x_t)
    kc, vc = as_f64(k_cache).copy(), as_f64(v_cache).copy()
    lens = np.asarray(lens, dtype=np.int64)
    B, D = x_t.shape
    H, Hk, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    if (lens < 0).any() or (lens >= kc.shape[2]).any():
        raise ValueError("each sequence needs room for one more position in the cache")
    if cfg.alibi and cfg.rotary_span:
        raise ValueError("rotary and ALiBi are exclusive: the rotary path is off for ALiBi blocks")

    def norm(t, wn, bn):
        if cfg.norm == "layernorm":
            return layer_norm(t, w[wn], w.get(bn), cfg.eps)
        return rms_norm(t, w[wn], cfg.eps)

    x = x_t[:, None, :]                                            # [B, 1, D]
    n1 = norm(x, "attn_norm_w", "attn_norm_b") if cfg.norm_place == "pre" else x
    qf, kf, vf = split_qkv(linear(n1, w["w_qkv"], w.get("b_qkv")), H, Hk, d, cfg.qkv_layout)
    if cfg.qk_norm == "rms_full":
        qf = qk_norm_full_rms(qf, w["q_norm_w"], cfg.qk_norm_eps)
        kf = qk_norm_full_rms(kf, w["k_norm_w"], cfg.qk_norm_eps)
    q, k, v = split_heads(qf, H, d), split_heads(kf, Hk, d), split_heads(vf, Hk, d)
    if cfg.qk_norm == "ln_per_head":
        q = qk_norm_per_head_ln(q, w["q_norm_w"], cfg.qk_norm_eps)
        k = qk_norm_per_head_ln(k, w["k_norm_w"], cfg.qk_norm_eps)
    o = np.empty((B, H, d))
    slopes = alibi_slopes(H) if cfg.alibi else None
    for b in range(B):
        p = int(lens[b])
        qb = rope(q[b:b + 1], np.array([p]), cfg.rotary_span, cfg.rope_base)
        kb = rope(k[b:b + 1], np.array([p]), cfg.rotary_span, cfg.rope_base)
        kc[b, :, p] = kb[0, :, 0]
        vc[b, :, p] = v[b, :, 0]
        o[b] = attention_decode(qb[:, :, 0], kc[b:b + 1], vc[b:b + 1], np.array([p + 1]),
                                slopes=slopes)[0]
    attn_out = linear(o.reshape(B, H * d), w["w_o"], w.get("b_o"))
    xs, n1s = x_t, n1[:, 0]
    if cfg.residual == "parallel":
        _, m = mlp(n1s, w, cfg.act)
        y = xs + attn_out + m
    elif cfg.norm_place == "pre":
        h = xs + attn_out
        _, m = mlp(norm(h, "mlp_norm_w", "mlp_norm_b"), w, cfg.act)
        y = h + m
    else:
        h = xs + rms_norm(attn_out, w["post_attn_norm_w"], cfg.eps)
        _, m = mlp(h, w, cfg.act)
        y = h + rms_norm(m, w["post_mlp_norm_w"], cfg.eps)
    return y, kc, vc
