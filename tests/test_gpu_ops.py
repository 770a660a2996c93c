"""GPU parity of each C-ABI call against the fp64 oracle (element by element).

Sizes span several tiles with ragged tails (rows, tokens, columns and
sequence lengths that are not multiples of the 128-row tiles)."""
import numpy as np
import pytest
import torch

import alibi_attention_block_gb300 as blk
import oracle
import workloads
from tests.parity import check, f64, row_cosine, to_dev
from workloads import draw

pytestmark = pytest.mark.gpu

DTYPES = ["fp16", "bf16"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from alibi_attention_block_gb300 import build
    build.build()
    yield
    blk.check_device_status()


# ------------------------------------------------------------------ norms --
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("rows,cols", [(1, 256), (77, 1024), (1000, 2048), (33, 5120), (5, 16384)])
@pytest.mark.parametrize("kind", ["layernorm", "layernorm_nobias", "rmsnorm"])
def test_norm(dt, rows, cols, kind):
    seed = rows * 7 + cols
    x = draw((rows, cols), dt, seed, scale=2.0)
    g = draw((cols,), dt, seed + 1, "g")
    b = draw((cols,), dt, seed + 2, "b")
    res = draw((rows, cols), dt, seed + 3) if rows % 2 else None
    eps = 1e-5
    if kind == "rmsnorm":
        out = blk.rmsnorm(to_dev(x), to_dev(g), residual=to_dev(res), eps=eps)
        ref = oracle.rms_norm(f64(x), f64(g), eps)
    else:
        beta = b if kind == "layernorm" else None
        out = blk.layernorm_bias(to_dev(x), to_dev(g), to_dev(beta), residual=to_dev(res), eps=eps)
        ref = oracle.layer_norm(f64(x), f64(g), None if beta is None else f64(beta), eps)
    if res is not None:
        ref = ref + f64(res)
    check(out, ref, f"{kind} {rows}x{cols}", unit_scale=True)


def test_norm_in_place():
    x = to_dev(draw((64, 2048), "bf16", 5))
    g = to_dev(draw((2048,), "bf16", 6, "g"))
    ref = oracle.rms_norm(f64(x), f64(g), 1e-6)
    blk.rmsnorm(x, g, eps=1e-6, out=x)
    check(x, ref, "rmsnorm in place", unit_scale=True)


# ----------------------------------------------------------------- linear --
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("m,n,k", [(128, 256, 256), (200, 264, 688), (1000, 2048, 2048),
                                   (37, 8, 8), (300, 768, 5632), (513, 1024, 64),
                                   (129, 512, 256), (257, 256, 4096)])
def test_linear(dt, m, n, k):
    seed = m + n + k
    x = draw((m, k), dt, seed)
    w = draw((n, k), dt, seed + 1, "w")
    bias = draw((n,), dt, seed + 2, "b") if m % 2 else None
    r1 = draw((m, n), dt, seed + 3) if n % 3 else None
    r2 = draw((m, n), dt, seed + 4) if k > 1000 else None
    y = blk.linear(to_dev(x), to_dev(w), to_dev(bias), to_dev(r1), to_dev(r2))
    ref = oracle.linear(f64(x), f64(w), None if bias is None else f64(bias))
    for r in (r1, r2):
        if r is not None:
            ref = ref + f64(r)
    check(y, ref, f"linear {m}x{n}x{k}")


def test_linear_persistent_multi_wave():
    """More output tiles than SMs: every CTA loops over several tiles and
    both TMEM accumulators."""
    x = draw((4096, 1024), "bf16", 11)
    w = draw((4096, 1024), "bf16", 12, "w")
    y = blk.linear(to_dev(x), to_dev(w))
    rows = workloads.sample_rows(4096, 64)
    ref = f64(x)[rows] @ f64(w).T
    check(y[torch.as_tensor(rows, device="cuda")], ref, "linear multi-wave")


@pytest.mark.parametrize("m,n,k", [(5000, 1000, 512), (2304, 2560, 320), (300, 1536, 256)])
def test_linear_partial_last_round(m, n, k):
    """Several rounds of 256 x 256 output tiles with a partial last one (80 =
    76 + 4 and 90 = 76 + 14 tiles on 76 CTA pairs) and a single partial round
    of 12 tiles, ragged in M and N, with bias and a residual."""
    seed = m + n + k
    x = draw((m, k), "bf16", seed)
    w = draw((n, k), "bf16", seed + 1, "w")
    bias = draw((n,), "bf16", seed + 2, "b")
    r1 = draw((m, n), "bf16", seed + 3)
    y = blk.linear(to_dev(x), to_dev(w), to_dev(bias), to_dev(r1))
    ref = oracle.linear(f64(x), f64(w), f64(bias)) + f64(r1)
    check(y, ref, f"linear last round {m}x{n}x{k}")


# -------------------------------------------------------------------- MLP --
@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("act,T,D,F", [("swiglu", 128, 256, 688), ("swiglu", 300, 512, 1024),
                                       ("gelu_tanh", 200, 256, 1024), ("gelu_tanh", 64, 1024, 4096)])
def test_mlp(dt, act, T, D, F):
    seed = T + D + F
    x = draw((T, D), dt, seed)
    w_up = draw((F, D), dt, seed + 1, "w")
    w_down = draw((D, F), dt, seed + 2, "w")
    w = {"w_up": f64(w_up), "w_down": f64(w_down)}
    kw = {}
    if act == "swiglu":
        w_gate = draw((F, D), dt, seed + 3, "w")
        w["w_gate"] = f64(w_gate)
        kw["w_gate"] = to_dev(w_gate)
    else:
        b_up = draw((F,), dt, seed + 4, "b")
        b_down = draw((D,), dt, seed + 5, "b")
        w["b_up"], w["b_down"] = f64(b_up), f64(b_down)
        kw["b_up"], kw["b_down"] = to_dev(b_up), to_dev(b_down)
    res = draw((T, D), dt, seed + 6)
    y = blk.mlp(to_dev(x), to_dev(w_up), to_dev(w_down), res1=to_dev(res), act=act, **kw)
    _, m = oracle.mlp(f64(x), w, act)
    check(y, m + f64(res), f"mlp {act}")


def test_mlp_gelu_large_preactivations():
    """GELU(tanh) where the up projection's outputs reach the hundreds: the
    epilogue's exponential overflows for large negative inputs (the result
    must go to zero, not NaN) and vanishes for large positive ones."""
    T, D, F = 200, 256, 1024
    x = draw((T, D), "fp16", 7, scale=60.0)
    w_up = draw((F, D), "fp16", 8, "w")
    w_down = draw((D, F), "fp16", 9, "w")
    b_up = draw((F,), "fp16", 10, "b")
    b_down = draw((D,), "fp16", 11, "b")
    res = draw((T, D), "fp16", 12)
    y = blk.mlp(to_dev(x), to_dev(w_up), to_dev(w_down), b_up=to_dev(b_up), b_down=to_dev(b_down),
                res1=to_dev(res), act="gelu_tanh")
    w = {"w_up": f64(w_up), "w_down": f64(w_down), "b_up": f64(b_up), "b_down": f64(b_down)}
    pre = f64(x) @ f64(w_up).T + f64(b_up)
    assert np.abs(pre).max() > 60.0, np.abs(pre).max()  # the regime this test is for
    _, m = oracle.mlp(f64(x), w, "gelu_tanh")
    check(y, m + f64(res), "mlp gelu large pre-activations")


# -------------------------------------------------------------------- QKV --
QKV_CASES = {
    # name: (B, S, D, H, Hk, d, layout, qk_norm, r, base, bias)
    "stablelm_fused_rope": (2, 200, 256, 4, 4, 64, "stacked", "none", 16, 1e4, True),
    "bloom_interleaved": (2, 130, 256, 4, 4, 64, "head_interleaved", "none", 0, 1e4, True),
    "olmo_rms_full_r128": (2, 150, 256, 2, 2, 128, "stacked", "rms_full", 128, 5e5, False),
    "gqa_ln_per_head_r40": (1, 140, 320, 8, 2, 160, "stacked", "ln_per_head", 40, 1e4, False),
    "gqa_ln_per_head_r40_bias": (2, 70, 320, 8, 2, 160, "stacked", "ln_per_head", 40, 1e4, True),
    "full_span_r64": (1, 128, 256, 4, 4, 64, "stacked", "none", 64, 1e4, True),
    "ln_per_head_d128_r32": (1, 140, 256, 4, 2, 128, "stacked", "ln_per_head", 32, 1e4, True),
    "rms_full_d64_r16_gqa": (2, 100, 256, 8, 2, 64, "stacked", "rms_full", 16, 1e4, False),
    "rms_full_d96_r24": (1, 90, 192, 2, 2, 96, "stacked", "rms_full", 24, 1e4, True),
    # the position-block path: bias, a partial span, 32 query heads (8 units
    # per thread) beside 8 kv heads, ragged last block
    "rms_full_d128_r64_bias": (1, 77, 256, 4, 4, 128, "stacked", "rms_full", 64, 1e4, True),
    "rms_full_h32_d128_bias": (1, 43, 256, 32, 8, 128, "stacked", "rms_full", 128, 5e5, True),
    "rms_full_d64_r0": (2, 33, 256, 4, 2, 64, "stacked", "rms_full", 0, 1e4, False),
    "ln_per_head_d96_r24_bias": (1, 90, 192, 2, 1, 96, "stacked", "ln_per_head", 24, 1e4, True),
    # the projection's TMA stores into q/k/v (S % 32 == 0, more than 128
    # tokens: CTA-pair GEMM): boxes of 64 columns (head_dim 64, 128; stacked
    # and interleaved; M = 320 leaves the last pair tile part past M), and
    # of 32 columns at head_dim 160
    "tma_boxes_d64_rope16": (2, 256, 256, 4, 4, 64, "stacked", "none", 16, 1e4, True),
    "tma_boxes_interleaved": (2, 192, 256, 4, 4, 64, "head_interleaved", "none", 0, 1e4, True),
    "tma_boxes_d128_rms_full": (2, 160, 256, 2, 2, 128, "stacked", "rms_full", 128, 5e5, False),
    "tma_boxes_d160_gqa": (1, 256, 320, 8, 2, 160, "stacked", "ln_per_head", 40, 1e4, True),
}


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("name", sorted(QKV_CASES))
def test_qkv_bias_rope_partial(dt, name):
    B, S, D, H, Hk, d, layout, qkn, r, base, bias = QKV_CASES[name]
    seed = 100 * sorted(QKV_CASES).index(name) + 7
    n_out = (H + 2 * Hk) * d
    x = draw((B, S, D), dt, seed)
    w = draw((n_out, D), dt, seed + 1, "w")
    b = draw((n_out,), dt, seed + 2, "b") if bias else None
    qnw = knw = None
    if qkn == "rms_full":
        qnw, knw = draw((H * d,), dt, seed + 3, "g"), draw((Hk * d,), dt, seed + 4, "g")
    elif qkn == "ln_per_head":
        qnw, knw = draw((H, d), dt, seed + 3, "g"), draw((Hk, d), dt, seed + 4, "g")
    q, k, v = blk.qkv_bias_rope_partial(to_dev(x), to_dev(w), to_dev(b), n_heads=H, n_kv_heads=Hk,
                                        head_dim=d, layout=layout, qk_norm=qkn, qk_norm_eps=1e-5,
                                        rotary_span=r, rope_base=base, q_norm_w=to_dev(qnw),
                                        k_norm_w=to_dev(knw))
    qf, kf, vf = oracle.split_qkv(oracle.linear(f64(x), f64(w), None if b is None else f64(b)),
                                  H, Hk, d, layout)
    if qkn == "rms_full":
        qf = oracle.qk_norm_full_rms(qf, f64(qnw), 1e-5)
        kf = oracle.qk_norm_full_rms(kf, f64(knw), 1e-5)
    qh, kh, vh = oracle.split_heads(qf, H, d), oracle.split_heads(kf, Hk, d), oracle.split_heads(vf, Hk, d)
    if qkn == "ln_per_head":
        qh = oracle.qk_norm_per_head_ln(qh, f64(qnw), 1e-5)
        kh = oracle.qk_norm_per_head_ln(kh, f64(knw), 1e-5)
    pos = np.arange(S)
    # With a qk-norm the raw projection is stored in the storage type before
    # it is normalised, and the normalised value is stored again: two
    # roundings of a unit-scale value, each up to half an ulp (1/64 in bf16
    # for |x| in [4, 8)), on top of the 2e-2 arithmetic budget.
    qk_tol = 2e-2 + (2 * 2.0 ** -6 if qkn != "none" and dt == "bf16" else 0.0)
    check(q, oracle.rope(qh, pos, r, base), f"{name} q", abs_tol=qk_tol)
    check(k, oracle.rope(kh, pos, r, base), f"{name} k", abs_tol=qk_tol)
    check(v, vh, f"{name} v")
    if qkn == "none" and 0 < r < d:
        # past the span the queries are the projection output unchanged: bit-equal
        # to the same projection with the rotary off
        q0, k0, _ = blk.qkv_bias_rope_partial(to_dev(x), to_dev(w), to_dev(b), n_heads=H,
                                              n_kv_heads=Hk, head_dim=d, layout=layout,
                                              rotary_span=0)
        assert torch.equal(q[..., r:], q0[..., r:]) and torch.equal(k[..., r:], k0[..., r:])
        assert not torch.equal(q[..., 1:, :r], q0[..., 1:, :r])


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("H,d,r,bias", [
    (4, 64, 16, True), (4, 64, 0, True), (4, 64, 64, False),
    # spans that are not a multiple of 16 and other head sizes take the
    # head-row path: its rotary partner slot is (r/2) mod 8, its lane offset
    # (r/2) / 8; the cases cover offsets 0..16 lanes and slots 0, 2, 3, 4, 5
    (4, 64, 20, True),     # r/2 = 10: slot 2, one lane
    (3, 96, 24, False),    # head_dim 96, r/2 = 12: slot 4
    (72, 160, 40, True),   # 72 heads x 160: r/2 = 20, slot 4, two lanes
    (2, 160, 160, False),  # full span at 160: slot 0, ten lanes
    (5, 48, 6, True),      # head_dim 48 (six active lanes), r/2 = 3: slot 3, zero lanes
    (4, 104, 26, True),    # head_dim 104, r/2 = 13: slot 5
    (2, 256, 250, True),   # head_dim 256 (every lane active), r/2 = 125: slot 5, 15 lanes
])
def test_rope_inplace(dt, H, d, r, bias):
    x = draw((2, H, 100, d), dt, 21 + r + H)
    b = draw((H * d,), dt, 22, "b") if bias else None
    xd = to_dev(x)
    blk.rope_inplace(xd, to_dev(b), rotary_span=r, rope_base=1e4)
    ref = f64(x)
    if bias:
        ref = ref + f64(b).reshape(H, d)[None, :, None, :]
    check(xd, oracle.rope(ref, np.arange(100), r, 1e4), f"rope H={H} d={d} r={r}")


# -------------------------------------------------------------- attention --
ATTN_CASES = [
    # (B, H, Hk, S, d, alibi)
    (1, 2, 2, 128, 64, False),
    (2, 4, 4, 200, 64, False),
    (1, 4, 2, 1000, 64, False),
    (2, 4, 4, 384, 64, True),
    (1, 2, 2, 1, 64, False),
    (1, 3, 3, 640, 64, False),     # odd tile count: the last pair has one query tile
    (1, 2, 2, 129, 64, True),      # second query tile of one row
    (4, 16, 4, 1152, 64, False),   # more items than SMs: several items per CTA
    (1, 2, 2, 333, 128, False),
    (2, 16, 4, 1536, 128, False),  # more items than SMs at head_dim 128, GQA
    (1, 3, 3, 640, 128, False),    # odd tile count: the last pair has one query tile
    (1, 4, 4, 256, 128, True),
    # ALiBi (key tiles walked from the diagonal down) with more items than
    # SMs, an odd tile count (the last pair has one query tile) and a ragged S
    (2, 16, 16, 1100, 64, True),
    (2, 16, 16, 1100, 128, True),
    (1, 4, 1, 300, 160, False),
    (2, 2, 2, 129, 160, False),
    # GQA-packed tiles (the group's query heads in the rows of one tile)
    (1, 8, 2, 300, 128, False),    # 4 heads x 32 positions per tile, ragged S
    (1, 2, 1, 257, 128, True),     # 2 heads x 64 positions, ALiBi per row's head
    (2, 32, 8, 520, 160, False),   # the 12B grouping (kv head j serves 4j..4j+3)
    (1, 6, 2, 200, 160, False),    # 3 heads x 40 positions: 8 padding rows
    (1, 8, 2, 200, 160, True),     # ALiBi with each row's own head slope
    (3, 8, 1, 700, 160, False),    # 8 heads x 16 positions
    (1, 32, 1, 136, 128, False),   # a group of 32: two chunks of 16 heads x 8 positions
    (1, 16, 2, 1, 160, False),     # one position
]


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: "B{}H{}Hk{}S{}d{}{}".format(*c[:5], "_alibi" if c[5] else ""))
def test_attention(dt, case):
    B, H, Hk, S, d, alibi = case
    seed = B * 1000 + H * 100 + S + d
    q = draw((B, H, S, d), dt, seed)
    k = draw((B, Hk, S, d), dt, seed + 1)
    v = draw((B, Hk, S, d), dt, seed + 2)
    o = blk.attn_prefill(to_dev(q), to_dev(k), to_dev(v), alibi=alibi)
    ref = oracle.attention(f64(q), f64(k), f64(v), slopes=oracle.alibi_slopes(H) if alibi else None)
    # outputs are convex combinations of unit-scale value rows: unit scale
    check(o, ref.transpose(0, 2, 1, 3), f"attention {case}", unit_scale=True)


@pytest.mark.parametrize("name", ["attn_s16384", "attn_12b"])
def test_attention_sweep_full_size_sampled(name):
    """The attention sweep at its full sizes (B2 S16384 H32x64 with QKV bias
    and r16; the 12B shape B2 S4096 H32/Hk8 x160 r40), run as bench.py runs
    it: bias and rotary in place (blk_rope_inplace), then blk_attn_prefill,
    on sampled query rows of every (batch, head). Each step is held to its
    own bar, and the two together to the floor the storage dtype sets:
    - rotary: within one bf16 ulp of the oracle's bias + rotary;
    - attention: the usual gate against the oracle on exactly the q/k/v
      the kernel received;
    - both: per row, no worse than the oracle's own q/k/v rounded to the
      storage dtype do against the exact oracle (minus 1e-4), and max abs
      within 2e-2. That floor falls with the sequence length (min cosine
      ~0.9995 at S=16384: a late row averages thousands of value rows, and
      the logit perturbation of bf16 q/k does not average out); any
      bf16 tensor-core attention shares it."""
    c = workloads.ATTN_CONFIGS[name]
    q, k, v, biases = workloads.attn_inputs(c)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    bd = [to_dev(t) for t in biases] if biases else None
    blk.rope_inplace(qd, bd[0] if bd else None, rotary_span=c.rotary_span, rope_base=c.rope_base)
    blk.rope_inplace(kd, bd[1] if bd else None, rotary_span=c.rotary_span, rope_base=c.rope_base)
    if bd:
        blk.rope_inplace(vd, bd[2], rotary_span=0, rope_base=c.rope_base)
    o = blk.attn_prefill(qd, kd, vd, alibi=c.alibi)
    blk.check_device_status()
    rows = workloads.sample_rows(c.seq, 24, seed=c.seed)
    H, Hk, d = c.n_heads, c.n_kv_heads, c.head_dim
    # the oracle's bias + rotary in fp64
    pos = np.arange(c.seq)
    qf, kf, vf = f64(q), f64(k), f64(v)
    if biases is not None:
        qf = qf + f64(biases[0]).reshape(H, d)[None, :, None, :]
        kf = kf + f64(biases[1]).reshape(Hk, d)[None, :, None, :]
        vf = vf + f64(biases[2]).reshape(Hk, d)[None, :, None, :]
    qf = oracle.rope(qf, pos, c.rotary_span, c.rope_base)
    kf = oracle.rope(kf, pos, c.rotary_span, c.rope_base)
    # 1. rotary: one bf16 ulp (2^-7 relative) of the exact value, plus the
    # fp32 rotation's own absolute error (angles to ~1e-6 rad on unit-scale
    # inputs) where a rotated value cancels to near zero
    for gpu_t, ref_t, label in ((qd, qf, "q"), (kd, kf, "k"), (vd, vf, "v")):
        g = f64(gpu_t)
        assert (np.abs(g - ref_t) <= 2.0 ** -7 * np.abs(ref_t) + 4e-6).all(), f"{name} rotary {label}"
    # 2. attention on exactly what the kernel received
    qg, kg, vg = f64(qd), f64(kd), f64(vd)
    slopes = oracle.alibi_slopes(H) if c.alibi else None
    got = f64(o[:, torch.as_tensor(rows, device=o.device)].permute(0, 2, 1, 3))
    ref_k = oracle.attention(qg[:, :, rows], kg, vg, slopes=slopes, q_positions=rows)
    check(got, ref_k, f"{name} attention kernel", unit_scale=True)
    # 3. composition against the exact oracle, at the storage floor
    exact = oracle.attention(qf[:, :, rows], kf, vf, slopes=slopes, q_positions=rows)
    bf = lambda a: torch.from_numpy(a).to(qd.dtype).double().numpy()
    stored = oracle.attention(bf(qf)[:, :, rows], bf(kf), bf(vf), slopes=slopes, q_positions=rows)
    floor = row_cosine(stored, exact)
    cos = row_cosine(got, exact)
    assert (cos >= np.minimum(floor, 0.9999) - 1e-4).all(), f"{name}: below the storage floor"
    assert np.abs(got - exact).max() <= 2e-2


@pytest.mark.parametrize("d", [64, 128, 160])
def test_attention_growing_logits_rescale(d):
    """Keys scaled up along the sequence make the running row max grow tile
    after tile, so O is rescaled in flight many times."""
    B, H, S = 1, 2, 900
    q = draw((B, H, S, d), "bf16", 70 + d)
    k = draw((B, H, S, d), "bf16", 71 + d)
    v = draw((B, H, S, d), "bf16", 72 + d)
    ramp = (1.0 + torch.arange(S, dtype=torch.float64) / 48.0).view(1, 1, S, 1)
    k = (k.double() * ramp).to(torch.bfloat16)
    o = blk.attn_prefill(to_dev(q), to_dev(k), to_dev(v))
    ref = oracle.attention(f64(q), f64(k), f64(v))
    check(o, ref.transpose(0, 2, 1, 3), f"attention growing logits d={d}", unit_scale=True)


def test_gqa_packed_equals_replicated_heads():
    """Packing a group's query heads into one tile changes only which rows
    share a tile: at head_dim 160 (where MHA and GQA run the same kernel)
    the GQA result is bit-identical to MHA with each kv head repeated for
    its group, and at head_dim 128 it meets the gate against it."""
    B, H, Hk, S = 2, 8, 2, 333
    for d in (160, 128):
        q = draw((B, H, S, d), "bf16", 90 + d)
        k = draw((B, Hk, S, d), "bf16", 91 + d)
        v = draw((B, Hk, S, d), "bf16", 92 + d)
        o = blk.attn_prefill(to_dev(q), to_dev(k), to_dev(v))
        rep = lambda t: t.repeat_interleave(H // Hk, dim=1).contiguous()  # noqa: E731
        o_mha = blk.attn_prefill(to_dev(q), to_dev(rep(k)), to_dev(rep(v)))
        if d == 160:
            assert torch.equal(o, o_mha)
        else:
            check(o, f64(o_mha), "gqa vs replicated d=128", unit_scale=True)


def test_attention_explicit_slopes_and_scale():
    B, H, S, d = 1, 4, 256, 64
    q, k, v = (draw((B, H, S, d), "bf16", 40 + i) for i in range(3))
    slopes = torch.tensor([0.5, 0.1, 0.0, 1.5], dtype=torch.float32)
    o = blk.attn_prefill(to_dev(q), to_dev(k), to_dev(v), alibi=True, slopes=slopes.cuda(),
                         scale=0.2)
    ref = oracle.attention(f64(q), f64(k), f64(v), scale=0.2, slopes=slopes.double().numpy())
    check(o, ref.transpose(0, 2, 1, 3), "attention explicit slopes", unit_scale=True)


def test_attention_large_scores_stay_finite():
    """Sharp softmax (scores of order 100) exercises the rescale path."""
    B, H, S, d = 1, 2, 512, 64
    q = draw((B, H, S, d), "bf16", 50, scale=6.0)
    k = draw((B, H, S, d), "bf16", 51, scale=6.0)
    v = draw((B, H, S, d), "bf16", 52)
    o = blk.attn_prefill(to_dev(q), to_dev(k), to_dev(v))
    ref = oracle.attention(f64(q), f64(k), f64(v))
    check(o, ref.transpose(0, 2, 1, 3), "attention sharp", unit_scale=True)


def test_attention_deterministic():
    q, k, v = (to_dev(draw((2, 4, 700, 64), "bf16", 60 + i)) for i in range(3))
    o1 = blk.attn_prefill(q, k, v)
    o2 = blk.attn_prefill(q, k, v)
    assert torch.equal(o1, o2)
