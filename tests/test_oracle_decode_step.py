"""Pins of the whole-block decode step oracle (CPU): after a prefill of a
sequence's first tokens, a decode step on the next token equals the prefill
of the longer sequence at that position, on every block variant and at
ragged lengths; the cache gains exactly the new token's key and value."""
import numpy as np
import pytest

import oracle
import workloads
from workloads import BLOCK_CONFIGS, scaled

VARIANTS = {
    "stablelm2": scaled(BLOCK_CONFIGS["stablelm2_1p6b"], batch=2, seq=12, hidden=64, n_heads=2,
                        n_kv_heads=2, head_dim=32, intermediate=96, rotary_span=16),
    "bloom_alibi": scaled(BLOCK_CONFIGS["bloom_560m"], batch=2, seq=12, hidden=64, n_heads=4,
                          n_kv_heads=4, head_dim=16, intermediate=128),
    "olmo2_post_norm": scaled(BLOCK_CONFIGS["olmo2_1b"], batch=2, seq=12, hidden=64, n_heads=2,
                              n_kv_heads=2, head_dim=32, intermediate=96, rotary_span=32),
    "stablelm2_12b_parallel": scaled(BLOCK_CONFIGS["stablelm2_12b"], batch=2, seq=12, hidden=64,
                                     n_heads=4, n_kv_heads=2, head_dim=16, intermediate=96,
                                     rotary_span=8),
}


def _caches(k, v, lens, s_max):
    B, Hk, _, d = k.shape
    kc = np.full((B, Hk, s_max, d), np.nan)
    vc = np.full((B, Hk, s_max, d), np.nan)
    for b, n in enumerate(lens):
        kc[b, :, :n] = k[b, :, :n]
        vc[b, :, :n] = v[b, :, :n]
    return kc, vc


@pytest.mark.parametrize("name", sorted(VARIANTS))
def test_decode_step_equals_prefill_last_row(name):
    cfg = VARIANTS[name]
    x, w = workloads.block_inputs(cfg)
    S = cfg.seq
    full = oracle.block_forward(cfg, x, w)
    lens = np.array([S - 1, S - 1])
    kc, vc = _caches(full["k"], full["v"], lens, S + 3)
    y, kc2, vc2 = oracle.block_decode_step(cfg, x[:, S - 1], w, kc, vc, lens)
    np.testing.assert_allclose(y, full["y"][:, S - 1], rtol=1e-12, atol=1e-12)
    # the new key and value land at position S - 1; nothing else changes
    np.testing.assert_allclose(kc2[:, :, S - 1], full["k"][:, :, S - 1], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(vc2[:, :, S - 1], full["v"][:, :, S - 1], rtol=1e-12, atol=1e-12)
    assert np.array_equal(kc2[:, :, :S - 1], kc[:, :, :S - 1])
    assert np.isnan(kc2[:, :, S:]).all()


def test_decode_step_at_ragged_lengths():
    """Sequences at different lengths in one step: each matches the prefill
    of its own prefix."""
    cfg = VARIANTS["stablelm2"]
    x, w = workloads.block_inputs(cfg)
    lens = np.array([4, 9])
    full = oracle.block_forward(cfg, x, w)             # prefixes are causal: reuse k, v
    kc, vc = _caches(full["k"], full["v"], lens, cfg.seq)
    x_t = np.stack([np.asarray(x[b, n].double()) for b, n in enumerate(lens)])
    y, _, _ = oracle.block_decode_step(cfg, x_t, w, kc, vc, lens)
    for b, n in enumerate(lens):
        np.testing.assert_allclose(y[b], full["y"][b, n], rtol=1e-12, atol=1e-12)


def test_decode_step_needs_room_in_the_cache():
    cfg = VARIANTS["stablelm2"]
    x, w = workloads.block_inputs(cfg)
    full = oracle.block_forward(cfg, x, w)
    kc, vc = _caches(full["k"], full["v"], [cfg.seq, cfg.seq], cfg.seq)
    with pytest.raises(ValueError):
        oracle.block_decode_step(cfg, x[:, -1], w, kc, vc, [cfg.seq, cfg.seq])
