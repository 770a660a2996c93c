"""GPU parity of the Q8_0 weight path against the fp64 oracle (oracle/quant.py).

- blk_q8_0_quantize: codes and scales bit for bit against the oracle's
  float32 GGML-order quantizer (the integer decision taken in float32 on both
  sides), including all-zero blocks and weights a hair below a half-step.
- blk_linear_q8_0: the W8A16 GEMM against the oracle's linear on the
  dequantized weight d * q, on codes and scales made by the oracle (so the
  GEMM is checked independently of the GPU quantizer), ragged m, n and k.
- blk_forward_q8_0: every block variant with Q8_0 projections against the
  oracle block on the dequantized weights, small and full size, by both of
  its paths (W8A16 GEMMs; weights expanded once for the dense GEMM)."""
import numpy as np
import pytest
import torch

import alibi_attention_block_gb300 as blk
import oracle
import workloads
from tests.parity import check, f64, to_dev
from workloads import BLOCK_CONFIGS, draw, scaled

pytestmark = pytest.mark.gpu

DTYPES = ["bf16", "fp16"]


def _oracle_q8(w):
    """Oracle codes [n, k] int8 and scales transposed to the library's
    block-major [k/32, n] fp16, as CUDA tensors."""
    q, d = oracle.q8_0_quantize(w)
    return (torch.from_numpy(q).cuda(), torch.from_numpy(np.ascontiguousarray(d.T)).cuda())


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("n,k", [(8, 32), (264, 96), (688, 2048), (1000, 160)])
def test_quantize_bit_exact(dt, n, k):
    w = draw((n, k), dt, 500 + n + k, "w")
    w[3 % n, :32] = 0                                  # an all-zero block
    if n > 5:
        w[5, 32:64] = w[5, 32:64] * 50                 # a block with a wide range
    q, d = blk.q8_0_quantize(to_dev(w))
    blk.check_device_status()
    q_ref, d_ref = oracle.q8_0_quantize(w)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), np.ascontiguousarray(d_ref.T).view(np.uint16))


def test_quantize_half_step_cases():
    """Weights just below a half-step of the float32 scale (the GGML order
    rounds them down; dividing by the fp16 scale would round them up)."""
    w = torch.zeros((4, 64), dtype=torch.float32)
    w[:, 0] = 1.0
    w[:, 1] = 63.497 / 127
    w[:, 2] = -63.497 / 127
    w[:, 33] = 0.75
    w[:, 40] = 0.75 * (31.49 / 127)
    w = w.to(torch.bfloat16)
    q, d = blk.q8_0_quantize(to_dev(w))
    q_ref, d_ref = oracle.q8_0_quantize(w)
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), np.ascontiguousarray(d_ref.T).view(np.uint16))


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("m,n,k,extras", [(300, 264, 96, True), (128, 8, 32, False),
                                          (1000, 688, 2048, True), (257, 512, 1024, False),
                                          (2048, 2048, 5632, True)])
def test_linear_q8_0(dt, m, n, k, extras):
    seed = m + 7 * n + k
    x = draw((m, k), dt, seed)
    w = draw((n, k), dt, seed + 1, "w")
    q, d = _oracle_q8(w)
    bias = draw((n,), dt, seed + 2, "b") if extras else None
    res = draw((m, n), dt, seed + 3) if extras else None
    y = blk.linear_q8_0(to_dev(x), q, d, bias=to_dev(bias), res1=to_dev(res))
    blk.check_device_status()
    qo, do = oracle.q8_0_quantize(w)
    ref = oracle.linear_q8_0(f64(x), qo, do, None if bias is None else f64(bias))
    if res is not None:
        ref = ref + f64(res)
    check(y, ref, f"linear_q8_0 m{m} n{n} k{k}", unit_scale=extras)


def test_linear_q8_0_matches_gpu_quantizer_path():
    """Quantizing on the GPU and multiplying gives the same bits as the
    oracle's codes fed to the same GEMM (the quantizer is bit-exact)."""
    x = draw((200, 256), "bf16", 11)
    w = draw((96, 256), "bf16", 12, "w")
    qg, dg = blk.q8_0_quantize(to_dev(w))
    qo, do = _oracle_q8(w)
    assert torch.equal(blk.linear_q8_0(to_dev(x), qg, dg), blk.linear_q8_0(to_dev(x), qo, do))


PROJ = {"qkv": "w_qkv", "o": "w_o", "gate": "w_gate", "up": "w_up", "down": "w_down"}

Q8_SMALL = {
    "stablelm2_small": scaled(BLOCK_CONFIGS["stablelm2_1p6b"], batch=2, seq=260, hidden=256,
                              n_heads=4, n_kv_heads=4, intermediate=704),
    "bloom_small": scaled(BLOCK_CONFIGS["bloom_560m"], batch=2, seq=256, hidden=256, n_heads=4,
                          n_kv_heads=4, intermediate=1024),
    "olmo2_small": scaled(BLOCK_CONFIGS["olmo2_1b"], batch=2, seq=300, hidden=256, n_heads=2,
                          n_kv_heads=2, intermediate=512),
    "stablelm2_12b_small": scaled(BLOCK_CONFIGS["stablelm2_12b"], batch=2, seq=260, hidden=320,
                                  n_heads=8, n_kv_heads=2, intermediate=512),
}


# blk_forward_q8_0's two ways to run the projections, chosen by the workspace
# size (every case here has at least 512 tokens): W8A16 GEMMs that expand the
# codes on chip, or the weights expanded once into the workspace's tail and
# multiplied by the dense GEMM
PATHS = {"w8a16": blk.forward_workspace_size, "dequant": blk.forward_q8_0_workspace_size}


def _q8_inputs(cfg, w):
    """The dense slots on the GPU, oracle-made Q8_0 codes and scales, and the
    oracle's dequantized weights."""
    dense = {k: to_dev(t) for k, t in w.items() if k not in PROJ.values()}
    q8, deq = {}, dict(w)
    for name, slot in PROJ.items():
        if slot not in w:
            continue
        qo, do = oracle.q8_0_quantize(w[slot])
        q8["q_" + name] = torch.from_numpy(qo).cuda()
        q8["d_" + name] = torch.from_numpy(np.ascontiguousarray(do.T)).cuda()
        deq[slot] = oracle.q8_0_dequantize(qo, do)
    return dense, q8, deq


def _q8_run(cfg, x, dense, q8, path):
    assert cfg.tokens >= 512  # below it both workspaces take the W8A16 GEMMs
    ws = torch.empty(PATHS[path](cfg, cfg.batch, cfg.seq), dtype=torch.uint8, device="cuda")
    y = blk.forward_q8_0(cfg, dense, q8, to_dev(x), workspace=ws)
    blk.check_device_status()
    return y


def _q8_block(cfg, x, w, path="w8a16"):
    """GPU block with Q8_0 projections (oracle-made codes) and the oracle
    block on the dequantized weights."""
    dense, q8, deq = _q8_inputs(cfg, w)
    return _q8_run(cfg, x, dense, q8, path), deq


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("name", sorted(Q8_SMALL))
def test_block_q8_small(name, path):
    cfg = Q8_SMALL[name]
    x, w = workloads.block_inputs(cfg)
    y, deq = _q8_block(cfg, x, w, path)
    ref = oracle.block_forward(cfg, x, deq)["y"]
    tol = 5e-2 if cfg.norm_place == "post" else 2e-2   # post-norm: the bf16 storage floor
    check(y, ref, f"q8 block {name} ({path})", unit_scale=True, abs_tol=tol, storage=cfg.dtype)


def test_block_q8_full_size_sampled_rows():
    """The StableLM-2-1.6B block with Q8_0 projections at full size, both
    paths, on 48 seeded rows the oracle evaluates one by one."""
    cfg = BLOCK_CONFIGS["stablelm2_1p6b"]
    x, w = workloads.block_inputs(cfg)
    dense, q8, deq = _q8_inputs(cfg, w)
    rows = workloads.sample_rows(cfg.tokens, 48, seed=cfg.seed)
    ref = oracle.block_forward(cfg, x, deq, rows=rows)["y"]
    idx = torch.as_tensor(rows, device="cuda")
    for path in sorted(PATHS):
        y = _q8_run(cfg, x, dense, q8, path)
        got = y.reshape(cfg.tokens, cfg.hidden)[idx]
        check(got, ref, f"q8 stablelm2_1p6b sampled rows ({path})", unit_scale=True,
              storage=cfg.dtype)
