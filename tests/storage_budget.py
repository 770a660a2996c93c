"""Error floor of bf16 storage, computed from the oracle (test infrastructure).

The block with every intermediate the CUDA path stores in the storage dtype
rounded to it (q, k, v after qk-norm and rotary; the attention output; the
MLP input and activation; the output y), everything else exact. The
difference from the exact oracle is the error that no kernel storing those
tensors can avoid. Only oracle functions and torch's dtype conversion are
used; nothing here comes from the CUDA path.
"""
import numpy as np
import torch

import oracle
from oracle import as_f64


def _round(a, dtype):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).double().numpy()


def post_norm_block_with_storage_rounding(cfg, x, w):
    """y of the reordered post-norm block (no input norm, RMS on sublayer
    outputs) with the storage roundings above, in float64 otherwise."""
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float16
    W = {k: as_f64(t) for k, t in w.items()}
    X = as_f64(x)
    H, Hk, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    pos = np.arange(cfg.seq)
    qf, kf, vf = oracle.split_qkv(oracle.linear(X, W["w_qkv"], W.get("b_qkv")), H, Hk, d,
                                  cfg.qkv_layout)
    qf = oracle.qk_norm_full_rms(qf, W["q_norm_w"], cfg.qk_norm_eps)
    kf = oracle.qk_norm_full_rms(kf, W["k_norm_w"], cfg.qk_norm_eps)
    q = _round(oracle.rope(oracle.split_heads(qf, H, d), pos, cfg.rotary_span, cfg.rope_base), dt)
    k = _round(oracle.rope(oracle.split_heads(kf, Hk, d), pos, cfg.rotary_span, cfg.rope_base), dt)
    v = _round(oracle.split_heads(vf, Hk, d), dt)
    o = _round(oracle.merge_heads(oracle.attention(q, k, v)), dt)
    h = X + oracle.rms_norm(oracle.linear(o, W["w_o"]), W["post_attn_norm_w"], cfg.eps)
    h16 = _round(h, dt)
    a = _round(oracle.silu(oracle.linear(h16, W["w_gate"])) * oracle.linear(h16, W["w_up"]), dt)
    y = h + oracle.rms_norm(oracle.linear(a, W["w_down"]), W["post_mlp_norm_w"], cfg.eps)
    return _round(y, dt)


def post_norm_block_from_stored_qkv(cfg, x, w, q, k, v, rows=None):
    """y of the reordered post-norm block continued, in float64, from the
    head-split q, k, v a kernel stored (after qk-norm and rotary, in the
    storage dtype), with the block's remaining storage roundings: the
    attention output, the bf16 copy of h that feeds the MLP, the MLP
    activation (y itself is returned unrounded). ``rows`` (optional): flat token indices into B*S, for
    which alone the attention and everything after it are evaluated. No
    rounding decision here depends on a softmax near-tie resolved
    differently from the kernel, because q and k are the kernel's own."""
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float16
    W = {kk: as_f64(t) for kk, t in w.items()}
    X = as_f64(x)
    B, S, D = X.shape
    H, d = cfg.n_heads, cfg.head_dim
    q, k, v = as_f64(q), as_f64(k), as_f64(v)
    if rows is None:
        o = oracle.merge_heads(oracle.attention(q, k, v)).reshape(B * S, H * d)
        xs = X.reshape(B * S, D)
    else:
        rows = np.asarray(rows)
        o = np.empty((len(rows), H * d))
        for b in range(B):
            mine = np.nonzero(rows // S == b)[0]
            if len(mine) == 0:
                continue
            qi = rows[mine] % S
            ob = oracle.attention(q[b:b + 1, :, qi], k[b:b + 1], v[b:b + 1], q_positions=qi)
            o[mine] = ob[0].transpose(1, 0, 2).reshape(len(mine), H * d)
        xs = X.reshape(B * S, D)[rows]
    o = _round(o, dt)
    h = xs + oracle.rms_norm(oracle.linear(o, W["w_o"]), W["post_attn_norm_w"], cfg.eps)
    h16 = _round(h, dt)
    a = _round(oracle.silu(oracle.linear(h16, W["w_gate"])) * oracle.linear(h16, W["w_up"]), dt)
    # y is left unrounded: the kernel's stored y then differs from it by at
    # most half an ulp of the storage type, as it does from the exact oracle
    return h + oracle.rms_norm(oracle.linear(a, W["w_down"]), W["post_mlp_norm_w"], cfg.eps)
