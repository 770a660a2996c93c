"""The block, step by step, in float64 NumPy (test infrastructure only).

Sources, cited by page title and section:

- [SLM] "StableLM-2: partial RoPE and a first LayerNorm-with-bias path in a
  dense ROCm engine" (Octoryn TR-2026-0016): Abstract, section 1 Contribution,
  section 4 Ablations (full-RoPE negative control).
- [BLM] "Bloom in a sovereign engine: ALiBi as the third positional paradigm"
  (Octoryn TR-2026-0010): Contribution (ALiBi as a per-head geometric slope,
  linear pre-softmax bias; fused-QKV de-interleave; rotary gated off).
- [NNT] nnterp encyclopedia, family "stablelm": 02 support() value table
  (layouts), Printout (module shapes, biases), Config, 03 Notes (block
  equations, partial rotary, query scale, qk_layernorm, QKV bias, GQA).
- [OLM] "OLMo-2: reordered (post) normalization and a loader-clobber
  root-cause": section 1 Contribution (no input norm; norms on sublayer
  outputs before the residual add; full-width QK RMSNorm).

Readings where the pages are silent (each repeated at its function):
  R1 rotary frequency over a partial span uses the span r: theta_j = base^(-2j/r).
  R2 rotate_half([a, b]) = [-b, a] (sign unpinned by the pages).
  R3 ALiBi slope for head i of H is 2^(-8(i+1)/H); bias -slope*(i-j), added
     after the d^-0.5 score scale, itself unscaled.
  R4 softmax scale d^-0.5 for every variant.
  R5 LayerNorm uses the population variance with eps inside the square root.
  R6 positions are 0..S-1 in every sequence (no BOS, no padding).
"""
from __future__ import annotations

import math

import numpy as np


def as_f64(t) -> np.ndarray | None:
    """Upcast a storage tensor (torch or NumPy) to float64 NumPy, exactly."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


# ---------------------------------------------------------------- norms ----

def layer_norm(x, gamma, beta, eps):
    """LayerNorm with bias over the last axis.

    [SLM] section 1 (the LayerNorm-with-bias path) and [NNT] Printout
    (LayerNorm((2048,), eps=1e-05, elementwise_affine=True, bias=True)).
    Reading R5: population variance, eps inside the square root.
    ``beta=None`` is the bias-free LayerNorm of the 12B per-head q/k norms.
    """
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    out = (x - mu) / np.sqrt(var + eps) * gamma
    if beta is not None:
        out = out + beta
    return out


def rms_norm(x, weight, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * weight.

    [OLM] section 1: the post-attention / post-feedforward norms and the
    full-width QK norm are RMSNorms.
    """
    ms = (x * x).mean(axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * weight


# -------------------------------------------------------- projections ----

def linear(x, w, b=None):
    """y = x W^T (+ b), torch Linear convention W[out, in] ([NNT] Printout)."""
    y = x @ w.T
    if b is not None:
        y = y + b
    return y


def split_heads(y, n_heads, head_dim):
    """[B, S, n*d] -> [B, n, S, d]: the layout of attention_queries/keys/values
    in [NNT] 02 support() ("Queries [batch num_heads seq qk_head_dim]")."""
    B, S, _ = y.shape
    return y.reshape(B, S, n_heads, head_dim).transpose(0, 2, 1, 3)


def merge_heads(o):
    """[B, H, S, d] -> [B, S, H*d]: attention_premix in [NNT] 02 support()
    ("HeadOutputs [batch seq num_heads head_dim]", what o_proj takes)."""
    B, H, S, d = o.shape
    return o.transpose(0, 2, 1, 3).reshape(B, S, H * d)


def split_qkv(y, n_heads, n_kv_heads, head_dim, layout):
    """Split the projection output into flat q [B,S,H*d], k and v [B,S,Hk*d].

    stacked: rows of W are [Wq; Wk; Wv] (separate q/k/v Linears, [NNT]
    Printout). head_interleaved: Bloom's fused QKV tensor, whose output rows
    run [head][q, k, v][d]; [BLM] Contribution names the de-interleave, the
    order per head is the workload's statement of it.
    """
    B, S, _ = y.shape
    H, Hk, d = n_heads, n_kv_heads, head_dim
    if layout == "stacked":
        q = y[..., : H * d]
        k = y[..., H * d: (H + Hk) * d]
        v = y[..., (H + Hk) * d: (H + 2 * Hk) * d]
    elif layout == "head_interleaved":
        if H != Hk:
            raise ValueError("head-interleaved QKV needs n_heads == n_kv_heads")
        t = y.reshape(B, S, H, 3, d)
        q = t[:, :, :, 0, :].reshape(B, S, H * d)
        k = t[:, :, :, 1, :].reshape(B, S, H * d)
        v = t[:, :, :, 2, :].reshape(B, S, H * d)
    else:
        raise ValueError(layout)
    return q, k, v


def qk_norm_full_rms(qf, weight, eps):
    """[OLM] section 1: RMSNorm over the whole Q (or K) projection row, not
    per head. qf is flat [B, S, n*d]; weight is [n*d]."""
    return rms_norm(qf, weight, eps)


def qk_norm_per_head_ln(qh, gamma, eps):
    """[NNT] 03 Notes, "Per-head LayerNorms on queries and keys on 12B": one
    bias-free LayerNorm per head, applied to the split heads before the
    rotary. qh is [B, n, S, d]; gamma is [n, d]."""
    return layer_norm(qh, gamma[None, :, None, :], None, eps)


# ----------------------------------------------------------- rotary ----

def rope_inv_freq(rotary_span, base):
    """theta_j = base^(-2j/r) for j < r/2 (reading R1: r is the rotary span)."""
    r = rotary_span
    j = np.arange(r // 2, dtype=np.float64)
    return base ** (-2.0 * j / r)


def rope(xh, positions, rotary_span, base):
    """NeoX split-half rotary over the first ``rotary_span`` dims of each head.

    [SLM] section 1: only the first r of the d head dims rotate, split-half
    over that span, the rest pass through. [NNT] 03 Notes, "Rotary turns a
    quarter of each head": on 1.6B the first 16 of 64 dims rotate as two
    halves of 8 (rotate_half); dims past 16 equal the projection output.
    Pairs are (j, j + r/2); x' = x cos + rotate_half(x) sin with
    rotate_half([a, b]) = [-b, a] (reading R2). xh is [B, n, S, d].
    """
    r = rotary_span
    out = np.array(xh, dtype=np.float64, copy=True)
    if r == 0:
        return out
    if r % 2 or r > xh.shape[-1]:
        raise ValueError("rotary span must be even and at most head_dim")
    half = r // 2
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_inv_freq(r, base)[None, :]
    c, s = np.cos(ang), np.sin(ang)                      # [S, r/2]
    a = xh[..., :half]
    b = xh[..., half:r]
    out[..., :half] = a * c - b * s
    out[..., half:r] = b * c + a * s
    return out


# ------------------------------------------------------------ ALiBi ----

def alibi_slopes(n_heads):
    """Per-head geometric slopes (reading R3): slope_i = 2^(-8(i+1)/H).

    [BLM] Contribution: a per-head geometric-series slope, a linear
    pre-softmax bias. The pages give no closed form for H not a power of two;
    the oracle refuses that case rather than guess.
    """
    H = int(n_heads)
    if H <= 0 or H & (H - 1):
        raise ValueError("ALiBi slopes are defined here for a power-of-two head count")
    return 2.0 ** (-8.0 * (np.arange(H, dtype=np.float64) + 1.0) / H)


# -------------------------------------------------------- attention ----

def attention(q, k, v, scale=None, slopes=None, causal=True, q_positions=None,
              return_probs=False, row_chunk=1024):
    """Causal softmax attention per (batch, head), scores materialised.

    [NNT] 03 Notes: query scale head_dim^-0.5 (R4 takes it for all variants),
    no window/softcap/sink; GQA maps kv head j to query heads
    j*H/Hk .. (j+1)*H/Hk - 1. [BLM] Contribution: ALiBi is a linear
    pre-softmax bias, here -slope_h * (i - j) (reading R3).

    q [B, H, Sq, d] holds the queries at positions ``q_positions`` (default
    0..Sq-1); k, v [B, Hk, S, d]. Returns o [B, H, Sq, d] (and the
    probabilities [B, H, Sq, S] when asked, for small cases).
    """
    B, H, Sq, d = q.shape
    Hk, S = k.shape[1], k.shape[2]
    if H % Hk:
        raise ValueError("n_heads must be a multiple of n_kv_heads")
    group = H // Hk
    if scale is None:
        scale = d ** -0.5
    pos_q = np.arange(Sq) if q_positions is None else np.asarray(q_positions)
    pos_k = np.arange(S)
    o = np.empty((B, H, Sq, v.shape[-1]), dtype=np.float64)
    probs = np.zeros((B, H, Sq, S)) if return_probs else None
    for b in range(B):
        for h in range(H):
            g = h // group
            for c0 in range(0, Sq, row_chunk):
                c1 = min(Sq, c0 + row_chunk)
                pq = pos_q[c0:c1]
                s = (q[b, h, c0:c1] @ k[b, g].T) * scale
                if slopes is not None:
                    s = s - slopes[h] * (pq[:, None] - pos_k[None, :])
                if causal:
                    s = np.where(pos_k[None, :] > pq[:, None], -np.inf, s)
                m = s.max(axis=-1, keepdims=True)
                e = np.exp(s - m)
                p = e / e.sum(axis=-1, keepdims=True)
                o[b, h, c0:c1] = p @ v[b, g]
                if return_probs:
                    probs[b, h, c0:c1] = p
    return (o, probs) if return_probs else o


def attention_decode(q, k_cache, v_cache, lens, scale=None, slopes=None):
    """One decode step of causal attention over a KV cache (the step after
    prefill; the pages state prefill only, this follows the same attention
    definition, [NNT] 03 Notes and [BLM] Contribution for ALiBi).

    q [B, H, d]: the newest token of each sequence, at position lens[b] - 1;
    k_cache, v_cache [B, Hk, S_max, d] hold positions 0 .. lens[b] - 1 (the
    newest included); entries at lens[b] and beyond are not part of the
    sequence. Returns o [B, H, d]: each query attends to its sequence's
    lens[b] keys, which is attention() with one query row at that position.
    """
    q, k_cache, v_cache = as_f64(q), as_f64(k_cache), as_f64(v_cache)
    B, H, d = q.shape
    o = np.empty((B, H, v_cache.shape[-1]), dtype=np.float64)
    for b in range(B):
        n = int(lens[b])
        if not 1 <= n <= k_cache.shape[2]:
            raise ValueError("lens must be in [1, S_max]")
        o[b] = attention(q[b:b + 1, :, None, :], k_cache[b:b + 1, :, :n], v_cache[b:b + 1, :, :n],
                         scale=scale, slopes=slopes, q_positions=[n - 1])[0, :, 0]
    return o


# -------------------------------------------------------------- MLP ----

def silu(z):
    """SiLU z * sigmoid(z) ([NNT] Printout: act_fn SiLUActivation)."""
    return z / (1.0 + np.exp(-z))


def gelu_tanh(z):
    """GELU, tanh form: 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))."""
    return 0.5 * z * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (z + 0.044715 * z ** 3)))


def mlp(n, w, act):
    """The MLP, returning (neurons, output).

    swiglu: down(silu(gate(n)) * up(n)), no biases ([NNT] Printout, 02
    support(): mlp_neurons = act(gate)*up on a gated MLP).
    gelu_tanh: W_down gelu_tanh(W_up n + b_up) + b_down (Bloom's MLP with biases).
    """
    if act == "swiglu":
        a = silu(linear(n, w["w_gate"])) * linear(n, w["w_up"])
    elif act == "gelu_tanh":
        a = gelu_tanh(linear(n, w["w_up"], w.get("b_up")))
    else:
        raise ValueError(act)
    return a, linear(a, w["w_down"], w.get("b_down"))


# ------------------------------------------------------------ block ----

def block_forward(cfg, x, weights, rows=None, positions=None):
    """The prefill forward of one decoder block, all variants.

    Sequential pre-norm ([NNT] 03 Notes, 1.6B): h = x + attn(LN1(x));
    out = h + mlp(LN2(h)). Parallel ([NNT] 03 Notes, 12B):
    n = LN(x); out = x + attn(n) + mlp(n). Reordered post-norm ([OLM]
    section 1): no input norm; h = x + RMS(attn(x)); out = h + RMS(mlp(h)).
    Dropout is the identity in eval ([NNT] 03 Notes).

    x is [B, S, D] (any float dtype; upcast to float64), weights a dict of
    slot name -> tensor. ``rows`` (optional) are flat token indices into
    B*S: keys and values are computed for every token, everything after the
    projections only for those rows. Returns a dict of float64 arrays: the
    per-token intermediates (n1, attn_premix, attn_out, h, n2, mlp_act,
    mlp_out, y; [B, S, .] or [n_rows, .] when rows are given) and q, k, v
    (head-split, after qk-norm and rotary, all tokens).
    """
    w = {kname: as_f64(t) for kname, t in weights.items()}
    x = as_f64(x)
    B, S, D = x.shape
    H, Hk, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    pos = np.arange(S) if positions is None else np.asarray(positions)

    def norm(t, wn, bn):
        if cfg.norm == "layernorm":
            return layer_norm(t, w[wn], w.get(bn), cfg.eps)
        return rms_norm(t, w[wn], cfg.eps)

    out = {}
    # input norm (absent in the reordered post-norm block)
    n1 = norm(x, "attn_norm_w", "attn_norm_b") if cfg.norm_place == "pre" else x
    # projection, split, qk-norm, rotary
    qf, kf, vf = split_qkv(linear(n1, w["w_qkv"], w.get("b_qkv")), H, Hk, d, cfg.qkv_layout)
    if cfg.qk_norm == "rms_full":
        qf = qk_norm_full_rms(qf, w["q_norm_w"], cfg.qk_norm_eps)
        kf = qk_norm_full_rms(kf, w["k_norm_w"], cfg.qk_norm_eps)
    q, k, v = split_heads(qf, H, d), split_heads(kf, Hk, d), split_heads(vf, Hk, d)
    if cfg.qk_norm == "ln_per_head":
        q = qk_norm_per_head_ln(q, w["q_norm_w"], cfg.qk_norm_eps)
        k = qk_norm_per_head_ln(k, w["k_norm_w"], cfg.qk_norm_eps)
    if cfg.alibi and cfg.rotary_span:
        raise ValueError("rotary and ALiBi are exclusive: the rotary path is off for ALiBi blocks")
    q = rope(q, pos, cfg.rotary_span, cfg.rope_base)
    k = rope(k, pos, cfg.rotary_span, cfg.rope_base)
    out["q"], out["k"], out["v"] = q, k, v
    slopes = alibi_slopes(H) if cfg.alibi else None

    # attention, for every query or only the sampled rows
    if rows is None:
        o = attention(q, k, v, slopes=slopes)
        premix = merge_heads(o)                                      # [B, S, H*d]
        sel = lambda t: t                                            # noqa: E731
    else:
        rows = np.asarray(rows)
        premix = np.empty((len(rows), H * d))
        for b in range(B):
            mine = np.nonzero(rows // S == b)[0]
            if len(mine) == 0:
                continue
            qi = rows[mine] % S
            ob = attention(q[b:b + 1, :, qi], k[b:b + 1], v[b:b + 1], slopes=slopes,
                           q_positions=pos[qi])
            premix[mine] = ob[0].transpose(1, 0, 2).reshape(len(mine), H * d)
        sel = lambda t: t.reshape(B * S, -1)[rows]                  # noqa: E731
    xs, n1s = sel(x), sel(n1)
    attn_out = linear(premix, w["w_o"], w.get("b_o"))
    out.update(n1=n1s, attn_premix=premix, attn_out=attn_out)

    if cfg.residual == "parallel":
        a, m = mlp(n1s, w, cfg.act)
        out.update(h=None, n2=n1s, mlp_act=a, mlp_out=m, y=xs + attn_out + m)
    elif cfg.norm_place == "pre":
        h = xs + attn_out
        n2 = norm(h, "mlp_norm_w", "mlp_norm_b")
        a, m = mlp(n2, w, cfg.act)
        out.update(h=h, n2=n2, mlp_act=a, mlp_out=m, y=h + m)
    else:
        h = xs + rms_norm(attn_out, w["post_attn_norm_w"], cfg.eps)
        a, m = mlp(h, w, cfg.act)
        out.update(h=h, n2=h, mlp_act=a, mlp_out=m,
                   y=h + rms_norm(m, w["post_mlp_norm_w"], cfg.eps))
    return out


def attention_forward(cfg, q, k, v, biases=None, rows=None):
    """Attention-only workload: optional q/k/v bias, rotary over the span,
    causal attention ([NNT] 03 Notes: the bias is added before the rotary).

    q [B, H, S, d], k and v [B, Hk, S, d] storage tensors; biases
    (bq [H*d], bk [Hk*d], bv [Hk*d]) or None. ``rows`` (optional) are query
    positions to evaluate in every (batch, head). Returns o [B, H, Sq, d].
    """
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    H, Hk, d = q.shape[1], k.shape[1], q.shape[3]
    if biases is not None:
        bq, bk, bv = (as_f64(t) for t in biases)
        q = q + bq.reshape(H, d)[None, :, None, :]
        k = k + bk.reshape(Hk, d)[None, :, None, :]
        v = v + bv.reshape(Hk, d)[None, :, None, :]
    S = q.shape[2]
    pos = np.arange(S)
    q = rope(q, pos, cfg.rotary_span, cfg.rope_base)
    k = rope(k, pos, cfg.rotary_span, cfg.rope_base)
    slopes = alibi_slopes(H) if cfg.alibi else None
    if rows is None:
        return attention(q, k, v, slopes=slopes)
    rows = np.asarray(rows)
    return attention(q[:, :, rows], k, v, slopes=slopes, q_positions=rows)
