"""Pins of the Q8_0 weight oracle (CPU): closed forms and exact cases."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

RNG = np.random.Generator(np.random.PCG64(77))


def test_error_bound_is_half_a_step_per_block():
    """|w - d q| <= D / 2 + 127 |D - d| everywhere, with D = absmax / 127 the
    exact scale the codes are rounded against and d its stored fp16 value;
    the block's largest |w| maps to |q| = 127."""
    w = RNG.standard_normal((48, 256)) * 0.02
    w = w.astype(np.float32).astype(np.float64)
    q, d = oracle.q8_0_quantize(w)
    err = np.abs(w - oracle.q8_0_dequantize(q, d)).reshape(48, 8, 32)
    exact = np.abs(w.reshape(48, 8, 32)).max(axis=-1) / 127.0
    df = d.astype(np.float64)
    # the stored scale is absmax / 127 to fp16 precision (11 significant bits)
    assert (np.abs(df - exact) <= exact * 2.0 ** -11).all()
    bound = exact / 2 * (1 + 1e-5) + 127 * np.abs(exact - df)
    assert (err <= bound[..., None] + 1e-12).all()
    top = np.abs(q.reshape(48, 8, 32)).max(axis=-1)
    assert (top == 127).all()


def test_codes_are_rounded_against_the_float32_scale_not_the_fp16_one():
    """GGML's order: codes from w * (1 / (absmax / 127)) before the scale is
    rounded to fp16. With absmax = 1 the exact code of w is round(127 w); a
    weight at 63.497 / 127 lies 0.003 below the half-step, far outside
    float32 rounding, so its code is 63. Dividing by the stored fp16 scale
    instead (1032 * 2^-17, 6e-5 below 1/127) would push it over 63.5 to 64.
    Every code of a random block is checked against exact rational
    arithmetic wherever that exact value is not within 1e-4 of a half-step."""
    from fractions import Fraction

    w = np.zeros((1, 32), dtype=np.float32)
    w[0, 0] = 1.0
    w[0, 1] = np.float32(63.497 / 127)
    w[0, 2] = -np.float32(63.497 / 127)
    q, d = oracle.q8_0_quantize(w)
    assert float(d[0, 0]) == 1032 * 2.0 ** -17
    assert q[0, 0] == 127 and q[0, 1] == 63 and q[0, 2] == -63

    blocks = (RNG.standard_normal((64, 32)) * 0.02).astype(np.float32)
    qb, _ = oracle.q8_0_quantize(blocks)
    checked = 0
    for row in range(64):
        amax = max(Fraction(float(abs(v))) for v in blocks[row])
        for j in range(32):
            r = Fraction(float(blocks[row, j])) * 127 / amax
            frac = abs(r) - int(abs(r))
            if abs(frac - Fraction(1, 2)) < Fraction(1, 10000):
                continue
            expect = int(abs(r) + Fraction(1, 2)) * (1 if r >= 0 else -1)
            assert int(qb[row, j]) == expect, (row, j, float(r))
            checked += 1
    assert checked > 2000


def test_exact_round_trip_of_representable_weights():
    """A weight that is already d * q with |q| <= 127 and an fp16 d comes
    back bit-exactly (and so does its linear)."""
    d = np.float16(0.0009765625)          # 2^-10, exact in fp16
    qv = RNG.integers(-127, 128, size=(16, 64))
    qv[:, ::32] = 127                     # every block reaches the full range
    w = qv * float(d)
    q, dd = oracle.q8_0_quantize(w)
    assert np.array_equal(q.astype(np.int64), qv) and (dd == d).all()
    x = RNG.standard_normal((5, 64))
    np.testing.assert_array_equal(oracle.linear_q8_0(x, q, dd), x @ w.T)


def test_zero_block_and_rounding_direction():
    w = np.zeros((2, 64))
    w[1, 32:] = np.linspace(-1, 1, 32)
    q, d = oracle.q8_0_quantize(w)
    assert d[0, 0] == 0 and d[0, 1] == 0 and d[1, 0] == 0 and not q[0].any() and not q[1, :32].any()
    # half away from zero: +-0.5 steps round outwards
    d1 = np.float16(0.5)
    w2 = np.full((1, 32), 0.25)
    w2[0, 0] = 63.5                        # absmax -> d = 0.5; 0.25 / 0.5 = 0.5 -> 1
    q2, dd2 = oracle.q8_0_quantize(w2)
    assert dd2[0, 0] == d1 and q2[0, 1] == 1 and q2[0, 0] == 127
    q3, _ = oracle.q8_0_quantize(-w2)
    assert q3[0, 1] == -1


def test_linear_matches_the_library_on_dequantized_weights():
    """The quantized linear is torch's float64 linear on d * q (a library
    routine on the dequantized weight)."""
    w = RNG.standard_normal((40, 96)) * 0.02
    b = RNG.standard_normal(40) * 0.02
    x = RNG.standard_normal((7, 96))
    q, d = oracle.q8_0_quantize(w)
    ref = F.linear(torch.from_numpy(x), torch.from_numpy(oracle.q8_0_dequantize(q, d)),
                   torch.from_numpy(b)).numpy()
    np.testing.assert_allclose(oracle.linear_q8_0(x, q, d, b), ref, rtol=1e-12, atol=1e-12)


def test_rejects_widths_not_a_multiple_of_32():
    with pytest.raises(ValueError):
        oracle.q8_0_quantize(np.ones((2, 40)))


@pytest.mark.parametrize("name", ["stablelm2_1p6b", "olmo2_1b"])
def test_block_with_q8_0_projections_stays_within_the_pages_gate(name):
    """Context for the pages' q8 figures ("StableLM-2 ...", section 3: q8
    logit cosine 0.998910; "OLMo-2 ...", section 4: int8 0.998700, both on
    real weights through whole models): one block whose five projections
    are Q8_0-quantized, against the same block with the original weights, on
    synthetic N(0, 0.02) weights. The sublayer part of the output (y - x)
    keeps a per-row cosine above the pages' 0.999 gate (measured: StableLM-2
    0.99994, OLMo-2 0.99989 at these sizes)."""
    import workloads
    cfg = workloads.scaled(workloads.BLOCK_CONFIGS[name], batch=1, seq=128, hidden=512,
                           n_heads=8 if name == "stablelm2_1p6b" else 4,
                           n_kv_heads=8 if name == "stablelm2_1p6b" else 4,
                           intermediate=1408 if name == "stablelm2_1p6b" else 1024)
    x, w = workloads.block_inputs(cfg)
    dense = oracle.block_forward(cfg, x, w)["y"].reshape(-1, cfg.hidden)
    deq = dict(w)
    for slot in ("w_qkv", "w_o", "w_gate", "w_up", "w_down"):
        if slot in w:
            deq[slot] = oracle.q8_0_dequantize(*oracle.q8_0_quantize(w[slot]))
    q8 = oracle.block_forward(cfg, x, deq)["y"].reshape(-1, cfg.hidden)
    xa = oracle.as_f64(x).reshape(-1, cfg.hidden)
    a, b = q8 - xa, dense - xa
    cos = (a * b).sum(-1) / np.linalg.norm(a, axis=-1) / np.linalg.norm(b, axis=-1)
    assert 0.999 <= cos.min() < 1.0
