"""Seeded synthetic workloads for the prefill forward of one decoder block.

This module holds shapes, seeds and random draws only. It contains none of
the block's arithmetic: both the fp64 oracle (``oracle/``) and the CUDA path
(``alibi_attention_block_gb300``) take their inputs from here, and neither
imports the other.

Recipe (every tensor): draw fp64 from NumPy ``PCG64(seed)`` in the fixed
name order of ``_DRAW_ORDER``, then round once to the storage dtype
(fp16 or bf16) with torch's CPU conversion. Both sides read the same bits.

- activations x ~ N(0, 1)
- projection weights ~ N(0, 0.02), biases ~ N(0, 0.02)
- norm gains ~ 1 + N(0, 0.02), norm shifts ~ N(0, 0.02)

The block shapes follow the model printouts and configs on the pages:
StableLM-2-1.6B (nnterp encyclopedia "stablelm", Printout and Config),
Bloom-560m (Octoryn TR-2026-0010, Contribution), OLMo-2-1B (Octoryn
"OLMo-2: reordered (post) normalization", section 1) and StableLM-2-12B
(nnterp "stablelm", Notes: parallel residual, qk_layernorm, GQA).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass

import numpy as np
import torch

__all__ = [
    "BlockConfig", "AttnConfig", "BLOCK_CONFIGS", "ATTN_CONFIGS",
    "block_inputs", "attn_inputs", "weight_shapes", "storage_dtype", "scaled", "draw",
    "sample_rows",
]


@dataclass(frozen=True)
class BlockConfig:
    name: str
    batch: int
    seq: int
    hidden: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    dtype: str                 # "fp16" | "bf16" (storage); accumulation is fp32 on the GPU
    norm: str                  # "layernorm" | "rmsnorm"
    norm_place: str            # "pre" | "post" (post: OLMo-2 reordered norm, no input norm)
    residual: str              # "sequential" | "parallel"
    eps: float
    qkv_layout: str            # "stacked" ([Wq;Wk;Wv]) | "head_interleaved" ([H][q,k,v][d])
    qkv_bias: bool
    o_bias: bool
    qk_norm: str               # "none" | "rms_full" | "ln_per_head"
    qk_norm_eps: float
    rotary_span: int           # 0 = no rotary
    rope_base: float
    alibi: bool
    act: str                   # "swiglu" | "gelu_tanh"
    mlp_bias: bool
    seed: int

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    @property
    def qkv_out(self) -> int:
        return (self.n_heads + 2 * self.n_kv_heads) * self.head_dim


@dataclass(frozen=True)
class AttnConfig:
    """Attention-only workload: q, k, v already projected, head-split."""
    name: str
    batch: int
    seq: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    rotary_span: int
    rope_base: float
    qkv_bias: bool
    alibi: bool
    dtype: str
    seed: int


_STABLELM2 = dict(norm="layernorm", norm_place="pre", residual="sequential", eps=1e-5,
                  qkv_layout="stacked", qkv_bias=True, o_bias=False, qk_norm="none",
                  qk_norm_eps=1e-5, rotary_span=16, rope_base=10000.0, alibi=False,
                  act="swiglu", mlp_bias=False)

BLOCK_CONFIGS: dict[str, BlockConfig] = {
    # Tiny StableLM-2-style block: small enough for the oracle in seconds.
    "tiny_stablelm2": BlockConfig(
        name="tiny_stablelm2", batch=1, seq=128, hidden=256, n_heads=4, n_kv_heads=4,
        head_dim=64, intermediate=688, dtype="fp16", seed=1000, **_STABLELM2),
    # StableLM-2-1.6B-shaped block (nnterp stablelm Printout/Config).
    "stablelm2_1p6b": BlockConfig(
        name="stablelm2_1p6b", batch=4, seq=2048, hidden=2048, n_heads=32, n_kv_heads=32,
        head_dim=64, intermediate=5632, dtype="bf16", seed=1001, **_STABLELM2),
    # Bloom-560m-shaped ALiBi block with fused head-interleaved QKV.
    "bloom_560m": BlockConfig(
        name="bloom_560m", batch=8, seq=1024, hidden=1024, n_heads=16, n_kv_heads=16,
        head_dim=64, intermediate=4096, dtype="fp16", norm="layernorm", norm_place="pre",
        residual="sequential", eps=1e-5, qkv_layout="head_interleaved", qkv_bias=True,
        o_bias=True, qk_norm="none", qk_norm_eps=1e-5, rotary_span=0, rope_base=10000.0,
        alibi=True, act="gelu_tanh", mlp_bias=True, seed=1002),
    # OLMo-2-1B-shaped post-norm block with full-width QK RMSNorm.
    "olmo2_1b": BlockConfig(
        name="olmo2_1b", batch=2, seq=4096, hidden=2048, n_heads=16, n_kv_heads=16,
        head_dim=128, intermediate=8192, dtype="bf16", norm="rmsnorm", norm_place="post",
        residual="sequential", eps=1e-6, qkv_layout="stacked", qkv_bias=False,
        o_bias=False, qk_norm="rms_full", qk_norm_eps=1e-6, rotary_span=128,
        rope_base=500000.0, alibi=False, act="swiglu", mlp_bias=False, seed=1003),
    # StableLM-2-12B-shaped parallel block: GQA 32/8, d=160, rotary span 40,
    # per-head qk LayerNorm, no biases. The MLP width 13824 is not on the pages
    # (an assumption; the 12B variant is measured attention-only).
    "stablelm2_12b": BlockConfig(
        name="stablelm2_12b", batch=2, seq=4096, hidden=5120, n_heads=32, n_kv_heads=8,
        head_dim=160, intermediate=13824, dtype="bf16", norm="layernorm", norm_place="pre",
        residual="parallel", eps=1e-5, qkv_layout="stacked", qkv_bias=False, o_bias=False,
        qk_norm="ln_per_head", qk_norm_eps=1e-5, rotary_span=40, rope_base=10000.0,
        alibi=False, act="swiglu", mlp_bias=False, seed=1004),
}

# Attention-only sequence sweep at StableLM-2 head shapes (batch x seq = 32768 tokens).
ATTN_CONFIGS: dict[str, AttnConfig] = {
    f"attn_s{s}": AttnConfig(name=f"attn_s{s}", batch=32768 // s, seq=s, n_heads=32,
                             n_kv_heads=32, head_dim=64, rotary_span=16, rope_base=10000.0,
                             qkv_bias=True, alibi=False, dtype="bf16", seed=1005 + i)
    for i, s in enumerate((512, 2048, 8192, 16384))
}
ATTN_CONFIGS["attn_12b"] = AttnConfig(
    name="attn_12b", batch=2, seq=4096, n_heads=32, n_kv_heads=8, head_dim=160,
    rotary_span=40, rope_base=10000.0, qkv_bias=False, alibi=False, dtype="bf16", seed=1009)


def storage_dtype(name: str) -> torch.dtype:
    return {"fp16": torch.float16, "bf16": torch.bfloat16, "fp32": torch.float32}[name]


def scaled(cfg, **changes):
    """A copy of a config with some fields changed (smaller parity cases)."""
    return dataclasses.replace(cfg, **changes)


def weight_shapes(cfg: BlockConfig) -> dict[str, tuple[tuple[int, ...], str]]:
    """Every weight slot the config uses: name -> (shape, distribution kind).

    kind: "w" = N(0, 0.02) weight, "b" = N(0, 0.02) bias/shift, "g" = 1 + N(0, 0.02) gain.
    Slots are distinct names: no slot aliases another.
    """
    D, F, H, Hk, d = cfg.hidden, cfg.intermediate, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    s: dict[str, tuple[tuple[int, ...], str]] = {}
    if cfg.norm_place == "pre":
        s["attn_norm_w"] = ((D,), "g")
        if cfg.norm == "layernorm":
            s["attn_norm_b"] = ((D,), "b")
        if cfg.residual == "sequential":
            s["mlp_norm_w"] = ((D,), "g")
            if cfg.norm == "layernorm":
                s["mlp_norm_b"] = ((D,), "b")
    else:
        s["post_attn_norm_w"] = ((D,), "g")
        s["post_mlp_norm_w"] = ((D,), "g")
    s["w_qkv"] = ((cfg.qkv_out, D), "w")
    if cfg.qkv_bias:
        s["b_qkv"] = ((cfg.qkv_out,), "b")
    if cfg.qk_norm == "rms_full":
        s["q_norm_w"] = ((H * d,), "g")
        s["k_norm_w"] = ((Hk * d,), "g")
    elif cfg.qk_norm == "ln_per_head":
        s["q_norm_w"] = ((H, d), "g")
        s["k_norm_w"] = ((Hk, d), "g")
    s["w_o"] = ((D, H * d), "w")
    if cfg.o_bias:
        s["b_o"] = ((D,), "b")
    if cfg.act == "swiglu":
        s["w_gate"] = ((F, D), "w")
    s["w_up"] = ((F, D), "w")
    if cfg.mlp_bias:
        s["b_up"] = ((F,), "b")
    s["w_down"] = ((D, F), "w")
    if cfg.mlp_bias:
        s["b_down"] = ((D,), "b")
    return s


_DRAW_ORDER = ("attn_norm_w", "attn_norm_b", "mlp_norm_w", "mlp_norm_b", "post_attn_norm_w",
               "post_mlp_norm_w", "w_qkv", "b_qkv", "q_norm_w", "k_norm_w", "w_o", "b_o",
               "w_gate", "w_up", "b_up", "w_down", "b_down")


def _draw(rng: np.random.Generator, shape, kind: str) -> np.ndarray:
    z = rng.standard_normal(shape)
    if kind == "x":
        return z
    z *= 0.02
    if kind == "g":
        z += 1.0
    return z


def _to_storage(a: np.ndarray, dtype: str) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(storage_dtype(dtype))


def block_inputs(cfg: BlockConfig, seed: int | None = None):
    """(x, weights) for one block, as CPU tensors in the storage dtype.

    x is [batch, seq, hidden]; weights maps slot name -> tensor.
    """
    rng = np.random.Generator(np.random.PCG64(cfg.seed if seed is None else seed))
    x = _to_storage(_draw(rng, (cfg.batch, cfg.seq, cfg.hidden), "x"), cfg.dtype)
    shapes = weight_shapes(cfg)
    weights = {}
    for name in _DRAW_ORDER:
        if name in shapes:
            shape, kind = shapes[name]
            weights[name] = _to_storage(_draw(rng, shape, kind), cfg.dtype)
    return x, weights


def model_inputs(cfg: BlockConfig, n_layers: int, vocab: int, embed_norm: bool = False,
                 final_norm: str = "layernorm", seed: int | None = None):
    """(tokens, model weights) for the model-level wrap, as CPU tensors:
    tokens int32 [batch, seq] uniform over the vocabulary; embed [vocab, D]
    ~ N(0, 1); per layer the block's weights (drawn as ``block_inputs`` does,
    seed + 1 + layer); norm gains ~ 1 + N(0, 0.02^2), shifts and lm_head
    ~ N(0, 0.02^2)."""
    base = cfg.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(base))
    tokens = torch.from_numpy(rng.integers(0, vocab, size=(cfg.batch, cfg.seq)).astype(np.int32))
    mw = {"embed": _to_storage(_draw(rng, (vocab, cfg.hidden), "x"), cfg.dtype)}
    if embed_norm:
        mw["embed_norm_w"] = _to_storage(_draw(rng, (cfg.hidden,), "g"), cfg.dtype)
        mw["embed_norm_b"] = _to_storage(_draw(rng, (cfg.hidden,), "b"), cfg.dtype)
    mw["layers"] = [block_inputs(cfg, seed=base + 1 + layer)[1] for layer in range(n_layers)]
    mw["final_norm_w"] = _to_storage(_draw(rng, (cfg.hidden,), "g"), cfg.dtype)
    if final_norm == "layernorm":
        mw["final_norm_b"] = _to_storage(_draw(rng, (cfg.hidden,), "b"), cfg.dtype)
    mw["lm_head"] = _to_storage(_draw(rng, (vocab, cfg.hidden), "w"), cfg.dtype)
    return tokens, mw


def attn_inputs(cfg: AttnConfig, seed: int | None = None):
    """Head-split q [B,H,S,d], k and v [B,Hk,S,d] ~ N(0,1), plus optional biases.

    Returns (q, k, v, biases) with biases = (bq [H*d], bk [Hk*d], bv [Hk*d]) or None.
    """
    rng = np.random.Generator(np.random.PCG64(cfg.seed if seed is None else seed))
    B, S, H, Hk, d = cfg.batch, cfg.seq, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    q = _to_storage(_draw(rng, (B, H, S, d), "x"), cfg.dtype)
    k = _to_storage(_draw(rng, (B, Hk, S, d), "x"), cfg.dtype)
    v = _to_storage(_draw(rng, (B, Hk, S, d), "x"), cfg.dtype)
    biases = None
    if cfg.qkv_bias:
        biases = tuple(_to_storage(_draw(rng, (n * d,), "b"), cfg.dtype) for n in (H, Hk, Hk))
    return q, k, v, biases


def sample_rows(n_tokens: int, n: int, seed: int = 7) -> np.ndarray:
    """A seeded, sorted sample of token rows (always includes the first and last)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if n >= n_tokens:
        return np.arange(n_tokens)
    pick = rng.choice(np.arange(1, n_tokens - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, n_tokens - 1], pick]))


def draw(shape, dtype: str, seed: int, kind: str = "x", scale: float = 1.0) -> torch.Tensor:
    """One seeded tensor in a storage dtype: kind "x" ~ N(0, scale^2), "w"/"b"
    ~ N(0, 0.02^2), "g" ~ 1 + N(0, 0.02^2)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = _draw(rng, tuple(shape), kind)
    if kind == "x" and scale != 1.0:
        a = a * scale
    return _to_storage(a, dtype)
