"""GPU parity of blk_attn_decode (one decode step over a KV cache) against
the fp64 oracle (oracle.attention_decode), through the C ABI."""
import numpy as np
import pytest
import torch

import alibi_attention_block_gb300 as blk
import oracle
from tests.parity import check, f64, to_dev
from workloads import draw

pytestmark = pytest.mark.gpu

CASES = [
    # (B, H, Hk, S_max, d, lens, alibi)
    (2, 4, 4, 100, 64, [1, 100], False),
    (3, 8, 2, 333, 128, [7, 200, 333], False),
    (2, 16, 2, 4096, 64, [4096, 2050], False),
    (1, 16, 16, 1024, 64, [1000], True),
    (4, 32, 32, 2048, 64, [2048, 1, 1500, 64], False),
    (2, 8, 1, 700, 128, [700, 33], False),
    # head_dim 128 with grouped heads: two warps per item share its K/V ring,
    # each with half of the group's query heads
    (2, 4, 2, 513, 128, [513, 64], True),
    (2, 32, 8, 4096, 128, [4096, 1], False),
    (2, 4, 4, 300, 128, [300, 17], False),   # MHA at head_dim 128: one warp per item
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from alibi_attention_block_gb300 import build
    build.build()


def _inputs(B, H, Hk, S, d, seed):
    q = draw((B, H, d), "bf16", seed)
    k = draw((B, Hk, S, d), "bf16", seed + 1)
    v = draw((B, Hk, S, d), "bf16", seed + 2)
    return q, k, v


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}Hk{}S{}d{}{}".format(*c[:5], "_alibi" if c[6] else ""))
def test_decode_matches_oracle(case):
    B, H, Hk, S, d, lens, alibi = case
    q, k, v = _inputs(B, H, Hk, S, d, 100 + B + H + S + d)
    kd, vd = to_dev(k), to_dev(v)
    # entries past each length are not part of the sequence: poison them
    for b, n in enumerate(lens):
        kd[b, :, n:] = float("nan")
        vd[b, :, n:] = float("nan")
    lens_d = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o = blk.attn_decode(to_dev(q), kd, vd, lens_d, alibi=alibi)
    blk.check_device_status()
    ref = oracle.attention_decode(f64(q), f64(k), f64(v), lens,
                                  slopes=oracle.alibi_slopes(H) if alibi else None)
    # outputs are convex combinations of unit-scale value rows
    check(o, ref, f"decode {case}", unit_scale=True)


def test_decode_equals_last_prefill_row():
    """The decode step of the last token over a cache written by prefill is
    the prefill attention's last row (up to the prefill's bf16 P)."""
    B, H, S, d = 2, 8, 512, 64
    q = draw((B, H, S, d), "bf16", 5)
    k = draw((B, H, S, d), "bf16", 6)
    v = draw((B, H, S, d), "bf16", 7)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o_pre = blk.attn_prefill(qd, kd, vd)  # [B, S, H, d]
    lens = torch.full((B,), S, dtype=torch.int32, device="cuda")
    o_dec = blk.attn_decode(qd[:, :, -1].contiguous(), kd, vd, lens)
    check(o_dec, f64(o_pre[:, -1]), "decode vs prefill last row", unit_scale=True, abs_tol=1e-2)


def test_decode_lengths_clamped_and_deterministic():
    B, H, S, d = 3, 4, 64, 64
    q, k, v = _inputs(B, H, H, S, d, 11)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    o = blk.attn_decode(qd, kd, vd, torch.tensor([0, 64, 999], dtype=torch.int32, device="cuda"))
    o_full = blk.attn_decode(qd, kd, vd, torch.tensor([64, 64, 64], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert torch.count_nonzero(o[0]) == 0           # length 0: zero row
    assert torch.equal(o[1:], o_full[1:])           # 999 clamps to the cache length
    again = blk.attn_decode(qd, kd, vd, torch.tensor([0, 64, 999], dtype=torch.int32, device="cuda"))
    assert torch.equal(o, again)
