"""Why the post-norm (OLMo-2-shaped) block cannot be held to 2e-2 against
the exact oracle, and what it is held to instead.

Its full-width QK RMSNorm makes q and k unit-scale per element, so with
random weights the attention logits have a spread of about sqrt(head_dim)
and the softmax is nearly one-hot: rounding q/k to bf16 (the configured
storage) moves near-ties. The emulation below shows that an otherwise exact
computation that stores the same tensors in bf16 already misses the exact
oracle by more than 2e-2 (and by less than 5e-2, the floor check the GPU
block keeps against the exact oracle). The GPU block itself is held to the
usual 2e-2 and per-row cosine 0.9999 against the oracle continued from the
q/k/v it stored (tests/test_gpu_block.py)."""
import numpy as np

import oracle
import workloads
from tests.storage_budget import post_norm_block_with_storage_rounding
from workloads import BLOCK_CONFIGS, scaled

POST_NORM_ABS_TOL = 5e-2


def test_continuation_from_exact_qkv_is_the_storage_emulation():
    """The continuation helper, fed the oracle's own q/k/v rounded to bf16,
    reproduces the full storage emulation bit for bit, at every row and at
    sampled rows (so the GPU gate built on it measures only the kernels)."""
    from tests.storage_budget import _round, post_norm_block_from_stored_qkv
    import torch
    cfg = scaled(BLOCK_CONFIGS["olmo2_1b"], batch=2, seq=70, hidden=128, n_heads=1,
                 n_kv_heads=1, intermediate=256)
    x, w = workloads.block_inputs(cfg)
    ref = oracle.block_forward(cfg, x, w)
    q, k, v = (_round(ref[n], torch.bfloat16) for n in ("q", "k", "v"))
    full = _round(post_norm_block_from_stored_qkv(cfg, x, w, q, k, v), torch.bfloat16)
    stored = post_norm_block_with_storage_rounding(cfg, x, w).reshape(cfg.tokens, cfg.hidden)
    assert np.array_equal(full, stored)
    rows = np.array([0, 5, 69, 70, 139])
    part = post_norm_block_from_stored_qkv(cfg, x, w, q, k, v, rows=rows)
    assert np.array_equal(_round(part, torch.bfloat16), stored[rows])


def test_bf16_storage_floor_of_post_norm_block():
    cfg = scaled(BLOCK_CONFIGS["olmo2_1b"], batch=2, seq=300, hidden=256, n_heads=2,
                 n_kv_heads=2, intermediate=512)
    x, w = workloads.block_inputs(cfg)
    exact = oracle.block_forward(cfg, x, w)["y"]
    stored = post_norm_block_with_storage_rounding(cfg, x, w)
    err = np.abs(stored - exact).max()
    assert 2e-2 < err < POST_NORM_ABS_TOL, err
