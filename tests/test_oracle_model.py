"""Pins of the model-level oracle (CPU): the pieces around the blocks against
torch's float64 library routines, composition of the blocks, causality at
model level, and rejection of ids outside the vocabulary."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads
from workloads import BLOCK_CONFIGS, scaled

CFG = BLOCK_CONFIGS["tiny_stablelm2"]
VOCAB = 96


def _t64(t):
    return torch.as_tensor(np.asarray(t.double() if isinstance(t, torch.Tensor) else t,
                                      dtype=np.float64))


@pytest.mark.parametrize("embed_norm,final_norm", [(False, "layernorm"), (True, "layernorm"),
                                                    (False, "rms"), (True, "rms")])
def test_no_layers_is_norms_and_projection(embed_norm, final_norm):
    """With no blocks the logits are lm_head(norm(LN?(embed[ids]))), the
    library's layer_norm / rms_norm / linear in float64."""
    tokens, mw = workloads.model_inputs(CFG, 0, VOCAB, embed_norm, final_norm)
    got = oracle.model_forward(CFG, tokens, mw, embed_norm, final_norm, 1e-5)
    x = _t64(mw["embed"])[tokens.long()]
    D = CFG.hidden
    if embed_norm:
        x = F.layer_norm(x, (D,), _t64(mw["embed_norm_w"]), _t64(mw["embed_norm_b"]), CFG.eps)
    if final_norm == "layernorm":
        n = F.layer_norm(x, (D,), _t64(mw["final_norm_w"]), _t64(mw["final_norm_b"]), 1e-5)
    else:
        n = F.rms_norm(x, (D,), _t64(mw["final_norm_w"]), 1e-5)
    ref = F.linear(n, _t64(mw["lm_head"])).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_blocks_compose_in_order():
    """Two layers: the second block reads the first block's output, and
    swapping the layers changes the logits (the order matters)."""
    tokens, mw = workloads.model_inputs(CFG, 2, VOCAB)
    got = oracle.model_forward(CFG, tokens, mw)
    x = np.asarray(mw["embed"].double())[tokens.long().numpy()]
    for lw in mw["layers"]:
        x = oracle.block_forward(CFG, x, lw)["y"]
    n = oracle.layer_norm(x, mw["final_norm_w"].double().numpy(), mw["final_norm_b"].double().numpy(),
                          1e-5)
    np.testing.assert_allclose(got, n @ mw["lm_head"].double().numpy().T, rtol=1e-12, atol=1e-12)
    swapped = dict(mw, layers=mw["layers"][::-1])
    assert np.abs(oracle.model_forward(CFG, tokens, swapped) - got).max() > 1e-3


def test_causal_at_model_level():
    """Changing the last token of a sequence leaves every earlier position's
    logits bit-equal and changes the last position's."""
    cfg = scaled(CFG, seq=24)
    tokens, mw = workloads.model_inputs(cfg, 2, VOCAB)
    a = oracle.model_forward(cfg, tokens, mw)
    t2 = tokens.clone()
    t2[0, -1] = (int(t2[0, -1]) + 1) % VOCAB
    b = oracle.model_forward(cfg, t2, mw)
    assert np.array_equal(a[0, :-1], b[0, :-1])
    assert np.abs(a[0, -1] - b[0, -1]).max() > 1e-6


def test_rejects_ids_outside_the_vocabulary():
    tokens, mw = workloads.model_inputs(CFG, 0, VOCAB)
    tokens[0, 3] = VOCAB
    with pytest.raises(ValueError):
        oracle.model_forward(CFG, tokens, mw)
