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
