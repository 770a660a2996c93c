"""fp64 oracle of the model-level wrap: token embedding, an optional
embedding LayerNorm, a stack of blocks, the final norm and the vocabulary
projection.

TEST INFRASTRUCTURE, like the rest of ``oracle``: only tests, the smoke test
and bench.py's CPU legs use it; the CUDA path never imports it.

Steps in the pages' order:
- embedding rows of the token ids (nnterp "stablelm" Printout: embed_tokens;
  token_embeddings is what enters the first block);
- for Bloom, a layernorm on the embeddings before the first block ("Bloom in
  a sovereign engine", Contribution (2));
- the blocks (``block_forward``), each one's output the next one's input
  (nnterp "stablelm" 03 Notes);
- the final norm, then lm_head with its own weights (nnterp "stablelm"
  Printout: norm is a LayerNorm with bias, lm_head hidden -> vocab; Config:
  tie_word_embeddings False). Reading: the final norm has the kind of the
  block's norms (a LayerNorm with bias for StableLM-2 and Bloom, an RMSNorm
  for OLMo-2, whose page is silent on it).
"""
from __future__ import annotations

import numpy as np

from .block import as_f64, block_forward, layer_norm, linear, rms_norm


def model_forward(cfg, tokens, mw, embed_norm=False, final_norm="layernorm", final_eps=1e-5):
    """Logits [B, S, vocab] (float64) of token ids [B, S].

    mw: ``embed`` [vocab, D], optional ``embed_norm_w`` / ``embed_norm_b``,
    ``layers`` (list of block weight dicts), ``final_norm_w``, optional
    ``final_norm_b``, ``lm_head`` [vocab, D]. Ids outside [0, vocab) are
    rejected.
    """
    ids = np.asarray(tokens, dtype=np.int64)
    emb = as_f64(mw["embed"])
    if ids.min() < 0 or ids.max() >= emb.shape[0]:
        raise ValueError("token id outside the vocabulary")
    x = emb[ids]                                   # [B, S, D]
    if embed_norm:
        x = layer_norm(x, as_f64(mw["embed_norm_w"]), as_f64(mw.get("embed_norm_b")), cfg.eps)
    for lw in mw.get("layers", []):
        x = block_forward(cfg, x, lw)["y"]
    if final_norm == "layernorm":
        n = layer_norm(x, as_f64(mw["final_norm_w"]), as_f64(mw.get("final_norm_b")), final_eps)
    else:
        n = rms_norm(x, as_f64(mw["final_norm_w"]), final_eps)
    return linear(n, as_f64(mw["lm_head"]))
