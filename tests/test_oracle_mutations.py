"""Planted mistakes in the oracle must each fail a pin.

Each case swaps one oracle function for a plausibly wrong version (on the
CPU, inside this test only) and checks that the named pin then fails. This is
evidence that the pins constrain the oracle, not a test of the GPU path.
"""
import numpy as np
import pytest

import oracle
import oracle.block as ob
from tests import test_oracle_attention as ta
from tests import test_oracle_block as tb
from tests import test_oracle_norms as tn
from tests import test_oracle_rope as tr

_ORIG = {n: getattr(ob, n) for n in ("attention", "split_qkv")}


def _rope_sign_flipped(xh, positions, rotary_span, base):
    out = np.array(xh, dtype=np.float64, copy=True)
    r = rotary_span
    if r == 0:
        return out
    h = r // 2
    ang = np.asarray(positions, dtype=np.float64)[:, None] * ob.rope_inv_freq(r, base)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = xh[..., :h], xh[..., h:r]
    out[..., :h] = a * c + b * s
    out[..., h:r] = b * c - a * s
    return out


def _rope_interleaved_pairs(xh, positions, rotary_span, base):
    out = np.array(xh, dtype=np.float64, copy=True)
    r = rotary_span
    if r == 0:
        return out
    ang = np.asarray(positions, dtype=np.float64)[:, None] * ob.rope_inv_freq(r, base)[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = xh[..., 0:r:2], xh[..., 1:r:2]
    out[..., 0:r:2] = a * c - b * s
    out[..., 1:r:2] = b * c + a * s
    return out


def _inv_freq_head_dim(rotary_span, base):
    j = np.arange(rotary_span // 2, dtype=np.float64)
    return base ** (-2.0 * j / (2 * rotary_span))


def _ln_sample_var(x, gamma, beta, eps):
    mu = x.mean(axis=-1, keepdims=True)
    var = x.var(axis=-1, ddof=1, keepdims=True)
    out = (x - mu) / np.sqrt(var + eps) * gamma
    return out if beta is None else out + beta


def _slopes_off_by_one(n):
    return 2.0 ** (-8.0 * np.arange(n, dtype=np.float64) / n)


def _attention_gqa_modulo(q, k, v, scale=None, slopes=None, causal=True, q_positions=None,
                          return_probs=False, row_chunk=1024):
    Hk = k.shape[1]
    idx = np.arange(q.shape[1]) % Hk
    return _ORIG["attention"](q, k[:, idx], v[:, idx], scale, slopes, causal, q_positions,
                              return_probs, row_chunk)


def _attention_no_scale(q, k, v, scale=None, **kw):
    return _ORIG["attention"](q, k, v, 1.0, **kw)


def _split_qkv_wrong_interleave(y, n_heads, n_kv_heads, head_dim, layout):
    if layout != "head_interleaved":
        return _ORIG["split_qkv"](y, n_heads, n_kv_heads, head_dim, layout)
    B, S, _ = y.shape
    t = y.reshape(B, S, 3, n_heads, head_dim)        # [q|k|v][H][d] instead of [H][q,k,v][d]
    return tuple(t[:, :, i].reshape(B, S, -1) for i in range(3))


MUTATIONS = [
    ("rope", _rope_sign_flipped, tr.test_closed_form_single_pair),
    ("rope", _rope_interleaved_pairs, tr.test_frequency_uses_the_span_and_pairs_split_half),
    ("rope_inv_freq", _inv_freq_head_dim, tr.test_frequency_uses_the_span_and_pairs_split_half),
    ("layer_norm", _ln_sample_var, tn.test_layer_norm_matches_torch_float64),
    ("alibi_slopes", _slopes_off_by_one, ta.test_alibi_slopes_closed_form),
    ("attention", _attention_gqa_modulo, ta.test_gqa_equals_mha_with_replicated_kv),
    ("attention", _attention_no_scale, ta.test_scale_is_inverse_sqrt_head_dim),
    ("split_qkv", _split_qkv_wrong_interleave,
     lambda: tb.test_block_matches_loop_only_brute_force("bloom")),
]


@pytest.mark.parametrize("i", range(len(MUTATIONS)))
def test_planted_mistake_is_caught(i, monkeypatch):
    name, bad, pin = MUTATIONS[i]
    monkeypatch.setattr(ob, name, bad)
    monkeypatch.setattr(oracle, name, bad, raising=False)
    with pytest.raises((AssertionError, ValueError)):
        pin()


# ---- the newer oracles (Q8_0 weights, the whole-block decode step): each
# mistake is planted in its own module, so the prefill oracle that the
# decode pin compares against stays the true one
import oracle.decode_step as ods  # noqa: E402
import oracle.quant as oq  # noqa: E402
from tests import test_oracle_decode_step as tds  # noqa: E402
from tests import test_oracle_quant as tq  # noqa: E402

_Q8 = oq.q8_0_quantize


def _q8_scale_over_128(w):
    w = np.asarray(w, dtype=np.float64)
    out_f, in_f = w.shape
    blocks = w.reshape(out_f, in_f // 32, 32)
    d = (np.abs(blocks).max(axis=-1) / 128.0).astype(np.float16)
    df = d.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(df[..., None] > 0, blocks / df[..., None], 0.0)
    q = np.clip(np.sign(r) * np.floor(np.abs(r) + 0.5), -127, 127).astype(np.int8)
    return q.reshape(out_f, in_f), d


def _q8_truncating(w):
    q, d = _Q8(w)
    w = np.asarray(w, dtype=np.float64)
    df = np.repeat(d.astype(np.float64), 32, axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(df > 0, w / df, 0.0)
    return np.clip(np.trunc(r), -127, 127).astype(np.int8), d


def _q8_divides_by_fp16_scale(w):
    """The order the GGML format does not use: the scale rounded to fp16
    first, the codes divided by it (and clipped)."""
    w = np.asarray(w, dtype=np.float64)
    out_f, in_f = w.shape
    blocks = w.reshape(out_f, in_f // 32, 32)
    d = (np.abs(blocks).max(axis=-1) / 127.0).astype(np.float16)
    df = d.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(df[..., None] > 0, blocks / df[..., None], 0.0)
    q = np.clip(np.sign(r) * np.floor(np.abs(r) + 0.5), -127, 127).astype(np.int8)
    return q.reshape(out_f, in_f), d


def _rope_at_next_position(xh, positions, rotary_span, base):
    return ob.rope(xh, np.asarray(positions) + 1, rotary_span, base)


def _attend_without_the_new_token(q, k_cache, v_cache, lens, scale=None, slopes=None):
    return ob.attention_decode(q, k_cache, v_cache, np.asarray(lens) - 1, scale, slopes)


_DECODE_PIN = lambda: tds.test_decode_step_equals_prefill_last_row("stablelm2")  # noqa: E731

MODULE_MUTATIONS = [
    (oq, "q8_0_quantize", _q8_scale_over_128, tq.test_error_bound_is_half_a_step_per_block),
    (oq, "q8_0_quantize", _q8_truncating, tq.test_error_bound_is_half_a_step_per_block),
    (oq, "q8_0_quantize", _q8_divides_by_fp16_scale,
     tq.test_codes_are_rounded_against_the_float32_scale_not_the_fp16_one),
    (ods, "rope", _rope_at_next_position, _DECODE_PIN),
    (ods, "attention_decode", _attend_without_the_new_token, _DECODE_PIN),
]


@pytest.mark.parametrize("i", range(len(MODULE_MUTATIONS)))
def test_planted_mistake_in_a_newer_oracle_is_caught(i, monkeypatch):
    mod, name, bad, pin = MODULE_MUTATIONS[i]
    monkeypatch.setattr(mod, name, bad)
    if mod is oq:
        monkeypatch.setattr(oracle, name, bad)
    with pytest.raises((AssertionError, ValueError)):
        pin()


import oracle.model as om  # noqa: E402
from tests import test_oracle_model as tm  # noqa: E402


def _norm_skipped(x, gamma, beta, eps):
    return np.asarray(x, dtype=np.float64)


def test_model_oracle_without_its_norms_fails_its_pin(monkeypatch):
    """Skipping the embedding / final LayerNorm in the model oracle fails the
    pin against torch's float64 layer_norm and linear."""
    monkeypatch.setattr(om, "layer_norm", _norm_skipped)
    with pytest.raises(AssertionError):
        tm.test_no_layers_is_norms_and_projection(True, "layernorm")
