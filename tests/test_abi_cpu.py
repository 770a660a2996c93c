"""The C-ABI library without a GPU: it builds, loads, exports every function
include/blk.h declares, rejects bad arguments before any CUDA call, and links
no vendor BLAS/DNN library (the pages' linkage audit: "StableLM-2: partial
RoPE ..." section 6, "Bloom in a sovereign engine" Methods, "OLMo-2 ..."
section 6)."""
import ctypes as C
import os
import re
import subprocess

import pytest

from alibi_attention_block_gb300 import _abi, build

FAKE = 0x100000  # 16-byte-aligned stand-in address; validation rejects before any access


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _abi.load()


def test_exports_every_declared_function(lib):
    names = _abi.header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_abi._PROTOS), "binding and header disagree"
    nm = subprocess.run(["nm", "-D", "--defined-only", _abi.LIB_PATH], capture_output=True,
                        text=True).stdout
    exported = set(re.findall(r"\sT\s(blk_\w+)", nm))
    assert set(names) <= exported


def test_links_no_vendor_math_library(lib):
    out = subprocess.run(["ldd", _abi.LIB_PATH], capture_output=True, text=True).stdout
    for bad in ("cublas", "cudnn", "cutlass", "cusparse", "nccl"):
        assert bad not in out.lower(), out


def test_sources_use_only_tcgen05_and_no_multicast():
    """Tensor-core work goes through tcgen05 (no legacy mma.sync / wmma, no
    Hopper wgmma). No kernel issues a multicast of any kind: every TMA load
    and every MMA-completion arrival targets the issuing CTA's own shared
    memory, and nothing uses NVLink multimem, so the same library is safe to
    run as independent replicas on several GPUs."""
    root = os.path.dirname(_abi.HERE)
    dirs = [os.path.join(root, "alibi_attention_block_gb300", "csrc"), os.path.join(root, "include")]
    seen = 0
    for d in dirs:
        for f in os.listdir(d):
            path = os.path.join(d, f)
            if not os.path.isfile(path):
                continue
            text = open(path).read()
            seen += 1
            assert "wgmma" not in text and "mma.sync" not in text and "wmma" not in text, f
            assert "multicast" not in text.lower(), f
            assert "multimem" not in text, f
    assert seen >= 10


def test_status_strings_and_version(lib):
    assert lib.blk_status_string(_abi.BLK_EINVAL) == b"BLK_EINVAL"
    assert lib.blk_status_string(_abi.BLK_ETIMEOUT) == b"BLK_ETIMEOUT"
    assert lib.blk_version() >> 16 == 1


def _err(lib):
    return lib.blk_last_error().decode()


def test_norm_validation(lib):
    st = lib.blk_layernorm_bias(None, None, FAKE, None, FAKE, 4, 64, 1e-5, 0, None)
    assert st == _abi.BLK_EINVAL and "x is NULL" in _err(lib)
    st = lib.blk_rmsnorm(FAKE, None, FAKE, FAKE, 4, 60, 1e-5, 1, None)
    assert st == _abi.BLK_EINVAL and "multiple of 8" in _err(lib)
    st = lib.blk_rmsnorm(FAKE + 4, None, FAKE, FAKE, 4, 64, 1e-5, 1, None)
    assert st == _abi.BLK_EINVAL and "aligned" in _err(lib)
    st = lib.blk_layernorm_bias(FAKE, None, FAKE, None, FAKE, 4, 64, 1e-5, 7, None)
    assert st == _abi.BLK_EINVAL and "dtype" in _err(lib)


def test_attention_validation(lib):
    d = _abi.AttnDesc(1, 128, 4, 4, 96, -1.0, 1, 0)
    assert lib.blk_attn_prefill(C.byref(d), FAKE, FAKE, FAKE, None, FAKE, 1, None) == _abi.BLK_EUNSUPPORTED
    d = _abi.AttnDesc(1, 128, 4, 4, 64, -1.0, 0, 0)
    assert lib.blk_attn_prefill(C.byref(d), FAKE, FAKE, FAKE, None, FAKE, 1, None) == _abi.BLK_EUNSUPPORTED
    assert "causal" in _err(lib)
    d = _abi.AttnDesc(1, 128, 6, 4, 64, -1.0, 1, 0)
    assert lib.blk_attn_prefill(C.byref(d), FAKE, FAKE, FAKE, None, FAKE, 1, None) == _abi.BLK_EINVAL
    d = _abi.AttnDesc(1, 128, 12, 12, 64, -1.0, 1, 1)   # standard slopes need 2^k heads
    assert lib.blk_attn_prefill(C.byref(d), FAKE, FAKE, FAKE, None, FAKE, 1, None) == _abi.BLK_EUNSUPPORTED
    d = _abi.AttnDesc(1, 128, 4, 4, 64, -1.0, 1, 0)     # slopes with alibi off
    assert lib.blk_attn_prefill(C.byref(d), FAKE, FAKE, FAKE, FAKE, FAKE, 1, None) == _abi.BLK_EINVAL


def test_qkv_validation(lib):
    d = _abi.QkvDesc(1, 16, 256, 4, 4, 64, _abi.BLK_QKV_STACKED, 0, 1e-5, 15, 1e4)
    assert lib.blk_qkv_bias_rope_partial(C.byref(d), FAKE, FAKE, None, None, None, FAKE, FAKE,
                                         FAKE, 1, None) == _abi.BLK_EINVAL     # odd span
    d = _abi.QkvDesc(1, 16, 256, 4, 2, 64, _abi.BLK_QKV_HEAD_INTERLEAVED, 0, 1e-5, 0, 1e4)
    assert lib.blk_qkv_bias_rope_partial(C.byref(d), FAKE, FAKE, None, None, None, FAKE, FAKE,
                                         FAKE, 1, None) == _abi.BLK_EINVAL     # interleaved GQA
    d = _abi.QkvDesc(1, 16, 256, 4, 4, 64, _abi.BLK_QKV_STACKED, 1, 1e-6, 0, 1e4)
    assert lib.blk_qkv_bias_rope_partial(C.byref(d), FAKE, FAKE, None, None, None, FAKE, FAKE,
                                         FAKE, 1, None) == _abi.BLK_EINVAL     # missing q_norm_w
    assert "q_norm_w" in _err(lib)


def _block(**kw):
    q = _abi.QkvDesc(1, 128, 256, 4, 4, 64, 0, 0, 1e-5, 16, 1e4)
    for k, v in kw.pop("qkv", {}).items():
        setattr(q, k, v)
    d = _abi.BlockDesc(q, _abi.BLK_NORM_LAYERNORM, _abi.BLK_NORM_PRE,
                       _abi.BLK_RESIDUAL_SEQUENTIAL, 1e-5, 0, 688, _abi.BLK_ACT_SWIGLU)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def _weights(**kw):
    base = dict(attn_norm_w=FAKE, mlp_norm_w=FAKE, w_qkv=FAKE, w_o=FAKE, w_gate=FAKE, w_up=FAKE,
                w_down=FAKE)
    base.update(kw)
    return _abi.BlockWeights(*[base.get(n) for n in _abi.WEIGHT_SLOTS])


def _fwd(lib, d, w, ws_bytes=1 << 40):
    return lib.blk_forward(C.byref(d), C.byref(w), FAKE, FAKE + 4096, FAKE, ws_bytes, 1, None)


def test_forward_rejects_rotary_with_alibi(lib):
    assert _fwd(lib, _block(alibi=1), _weights()) == _abi.BLK_EUNSUPPORTED
    assert "exclusive" in _err(lib)


def test_forward_slot_rules(lib):
    """A weight in a slot the block does not read is an error, never ignored;
    a required slot left empty is an error (the loader-clobber lesson,
    "OLMo-2 ..." section 1 and section 6)."""
    post = dict(norm_kind=_abi.BLK_NORM_RMS, norm_place=_abi.BLK_NORM_POST)
    w_post = dict(attn_norm_w=None, mlp_norm_w=None, post_attn_norm_w=FAKE, post_mlp_norm_w=FAKE)
    # post-norm block handed a pre-norm slot
    assert _fwd(lib, _block(**post), _weights(**dict(w_post, mlp_norm_w=FAKE))) == _abi.BLK_EINVAL
    assert "mlp_norm_w" in _err(lib)
    # post-norm block missing its MLP norm
    assert _fwd(lib, _block(**post), _weights(**dict(w_post, post_mlp_norm_w=None))) == _abi.BLK_EINVAL
    assert "post_mlp_norm_w" in _err(lib)
    # parallel block has no MLP norm
    par = dict(residual=_abi.BLK_RESIDUAL_PARALLEL)
    assert _fwd(lib, _block(**par), _weights()) == _abi.BLK_EINVAL
    # GELU block must not get a gate weight
    assert _fwd(lib, _block(act=_abi.BLK_ACT_GELU_TANH), _weights()) == _abi.BLK_EINVAL
    assert "w_gate" in _err(lib)


def test_forward_workspace_check(lib):
    assert _fwd(lib, _block(), _weights(), ws_bytes=16) == _abi.BLK_EWORKSPACE
    need = C.c_size_t(0)
    assert lib.blk_forward_workspace_size(C.byref(_block()), C.byref(need)) == _abi.BLK_OK
    # n1, q, k, v, o, h (fp32), n2, a, h16, tmp (fp32) for T = 128 tokens
    T, D, F = 128, 256, 688
    split = 256 * 128 * 256 * 4 + 1024 * 4  # split GEMM rounds: partial tiles + counters
    assert need.value == 2 * T * (7 * D + 4 * 256 + F) + split


def test_forward_q8_0_workspace_size(lib):
    """The dequantize-once path's workspace: the block's, then every
    projection's weights in the storage dtype (QKV, output, gate for SwiGLU,
    up, down), each 256-byte aligned."""
    base, q8 = C.c_size_t(0), C.c_size_t(0)
    D, qkv = 256, 3 * 4 * 64
    al = lambda b: -(-b // 256) * 256
    for kw, F, n_up in ((dict(), 688, 2), (dict(act=_abi.BLK_ACT_GELU_TANH), 688, 1),
                        (dict(intermediate=2048), 2048, 2)):
        d = _block(**kw)
        assert lib.blk_forward_workspace_size(C.byref(d), C.byref(base)) == _abi.BLK_OK
        assert lib.blk_forward_q8_0_workspace_size(C.byref(d), C.byref(q8)) == _abi.BLK_OK
        want = al(2 * qkv * D) + al(2 * D * 256) + n_up * al(2 * F * D) + al(2 * D * F)
        assert q8.value - base.value == want
    bad = _block(intermediate=12)
    assert lib.blk_forward_q8_0_workspace_size(C.byref(bad), C.byref(q8)) == _abi.BLK_EINVAL


def test_mlp_validation(lib):
    d = _abi.MlpDesc(128, 256, 688, _abi.BLK_ACT_SWIGLU)
    st = lib.blk_mlp(C.byref(d), FAKE, None, FAKE, None, FAKE, None, None, None, FAKE, FAKE,
                     1 << 30, 1, None)
    assert st == _abi.BLK_EINVAL and "w_gate" in _err(lib)
    st = lib.blk_mlp(C.byref(d), FAKE, FAKE, FAKE, None, FAKE, None, None, None, FAKE, FAKE, 8,
                     1, None)
    assert st == _abi.BLK_EWORKSPACE


def test_linear_validation(lib):
    assert lib.blk_linear(FAKE, FAKE, None, None, None, FAKE, 128, 100, 256, 1, None) == _abi.BLK_EINVAL
    assert lib.blk_linear(FAKE, FAKE, None, None, None, FAKE, 0, 128, 256, 1, None) == _abi.BLK_OK


def test_binding_refuses_cpu_tensors():
    import torch

    import alibi_attention_block_gb300 as blk
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        blk.rmsnorm(x, torch.ones(64, dtype=torch.bfloat16))


def test_graph_handle_validation(lib):
    """The graph entry points reject a missing handle before any CUDA call;
    destroying NULL is a no-op."""
    assert lib.blk_forward_graph_create(C.byref(_block()), C.byref(_weights()), FAKE, FAKE + 4096,
                                        FAKE, 1 << 30, 1, None, 0, None, None,
                                        None) == _abi.BLK_EINVAL
    assert "out" in _err(lib)
    assert lib.blk_graph_launch(None, None) == _abi.BLK_EINVAL
    assert lib.blk_graph_destroy(None) == _abi.BLK_OK


def test_forward_host_validation(lib):
    """blk_forward_host checks its host/device buffers and chunk count before
    any CUDA call."""
    args = (C.byref(_block()), C.byref(_weights()))
    assert lib.blk_forward_host(*args, None, FAKE, FAKE, FAKE + 4096, FAKE, 1 << 30, 2, 1,
                                None) == _abi.BLK_EINVAL
    assert lib.blk_forward_host(*args, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, 2, 1,
                                None) == _abi.BLK_EINVAL  # y_dev aliases x_dev
    assert lib.blk_forward_host(*args, FAKE, FAKE, FAKE, FAKE + 4096, FAKE, 1 << 30, 0, 1,
                                None) == _abi.BLK_EINVAL
    assert "n_chunks" in _err(lib)
    assert lib.blk_forward_host(*args, FAKE, FAKE, FAKE, FAKE + 4096, FAKE, 16, 2, 1,
                                None) == _abi.BLK_EWORKSPACE
    assert lib.blk_graph_set_events(None, None, 0) == _abi.BLK_EINVAL


def test_host_pipe_validation(lib):
    """blk_host_pipe_*: sizes, depth range and argument checks without a GPU;
    destroying NULL is a no-op."""
    d = _block()
    n = C.c_size_t(0)
    ws = C.c_size_t(0)
    assert lib.blk_forward_workspace_size(C.byref(d), C.byref(ws)) == _abi.BLK_OK
    assert lib.blk_host_pipe_mem_size(C.byref(d), 2, C.byref(n)) == _abi.BLK_OK
    io = d.qkv.batch * d.qkv.seq * d.qkv.hidden * 2
    io = (io + 255) // 256 * 256
    assert n.value == 4 * io + ws.value  # two slots of x and y, then the workspace
    for bad in (1, 5):
        assert lib.blk_host_pipe_mem_size(C.byref(d), bad, C.byref(n)) == _abi.BLK_EINVAL
        assert "depth" in _err(lib)
    out = C.c_void_p()
    assert lib.blk_host_pipe_create(C.byref(d), 2, 1, FAKE, 1 << 40, None) == _abi.BLK_EINVAL
    assert lib.blk_host_pipe_create(C.byref(d), 2, 7, FAKE, 1 << 40, C.byref(out)) == _abi.BLK_EINVAL
    assert lib.blk_host_pipe_create(C.byref(d), 2, 1, None, 1 << 40, C.byref(out)) == _abi.BLK_EINVAL
    assert lib.blk_host_pipe_create(C.byref(d), 2, 1, FAKE, 16, C.byref(out)) == _abi.BLK_EWORKSPACE
    assert out.value is None
    assert lib.blk_host_pipe_submit(None, C.byref(_weights()), FAKE, FAKE, None) == _abi.BLK_EINVAL
    assert lib.blk_host_pipe_flush(None, None) == _abi.BLK_EINVAL
    assert lib.blk_host_pipe_destroy(None) == _abi.BLK_OK


def test_model_validation(lib):
    """blk_model_*: descriptor and argument checks before any CUDA call."""
    d = _abi.ModelDesc(_block(), 2, 1000, 0, _abi.BLK_NORM_LAYERNORM, 1e-5)
    need, blk = C.c_size_t(0), C.c_size_t(0)
    assert lib.blk_model_workspace_size(C.byref(d), C.byref(need)) == _abi.BLK_OK
    assert lib.blk_forward_workspace_size(C.byref(d.block), C.byref(blk)) == _abi.BLK_OK
    q = d.block.qkv
    act = (q.batch * q.seq * q.hidden * 2 + 255) // 256 * 256
    assert need.value == 3 * act + blk.value  # two activations, the final norm, one block
    for bad in (_abi.ModelDesc(_block(), -1, 1000, 0, 0, 1e-5),   # n_layers
                _abi.ModelDesc(_block(), 2, 1004, 0, 0, 1e-5),    # vocab % 8
                _abi.ModelDesc(_block(), 2, 1000, 2, 0, 1e-5),    # embed_norm
                _abi.ModelDesc(_block(), 2, 1000, 0, 7, 1e-5)):   # final_norm
        assert lib.blk_model_workspace_size(C.byref(bad), C.byref(need)) == _abi.BLK_EINVAL
    layers = (_abi.BlockWeights * 2)(_weights(), _weights())
    w = _abi.ModelWeights(FAKE, None, None, layers, FAKE, FAKE, FAKE)
    args = (C.byref(d), C.byref(w))
    assert lib.blk_model_forward(*args, None, FAKE, FAKE, 1 << 40, 1, None) == _abi.BLK_EINVAL
    assert "tokens" in _err(lib)
    assert lib.blk_model_forward(*args, FAKE, FAKE, FAKE, 16, 1, None) == _abi.BLK_EWORKSPACE
    no_head = _abi.ModelWeights(FAKE, None, None, layers, FAKE, FAKE, None)
    assert lib.blk_model_forward(C.byref(d), C.byref(no_head), FAKE, FAKE, FAKE, 1 << 40, 1,
                                 None) == _abi.BLK_EINVAL
    stray = _abi.ModelWeights(FAKE, FAKE, None, layers, FAKE, FAKE, FAKE)  # embed_norm is 0
    assert lib.blk_model_forward(C.byref(d), C.byref(stray), FAKE, FAKE, FAKE, 1 << 40, 1,
                                 None) == _abi.BLK_EINVAL
    rms = _abi.ModelDesc(_block(), 2, 1000, 0, _abi.BLK_NORM_RMS, 1e-6)  # RMS has no bias
    assert lib.blk_model_forward(C.byref(rms), C.byref(w), FAKE, FAKE, FAKE, 1 << 40, 1,
                                 None) == _abi.BLK_EINVAL
    empty = _abi.ModelWeights(FAKE, None, None, None, FAKE, FAKE, FAKE)  # layers NULL
    assert lib.blk_model_forward(C.byref(d), C.byref(empty), FAKE, FAKE, FAKE, 1 << 40, 1,
                                 None) == _abi.BLK_EINVAL


def test_decode_validation(lib):
    """blk_attn_decode: shape rules and workspace size without a GPU."""
    d = _abi.DecodeDesc(4, 2048, 32, 8, 64, -1.0, 0)
    need = C.c_size_t(0)
    assert lib.blk_attn_decode_workspace_size(C.byref(d), C.byref(need)) == _abi.BLK_OK
    assert need.value == 4 * 32 * 32 * (64 + 2) * 4  # parts <= ceil(2048 / 64) = 32
    bad = _abi.DecodeDesc(4, 2048, 32, 8, 96, -1.0, 0)
    assert lib.blk_attn_decode_workspace_size(C.byref(bad), C.byref(need)) == _abi.BLK_EUNSUPPORTED
    bad = _abi.DecodeDesc(4, 2048, 24, 8, 64, -1.0, 0)  # group of 3
    assert lib.blk_attn_decode_workspace_size(C.byref(bad), C.byref(need)) == _abi.BLK_EUNSUPPORTED
    assert lib.blk_attn_decode(C.byref(d), FAKE, FAKE, FAKE, None, None, FAKE, FAKE, 1 << 30, 1,
                               None) == _abi.BLK_EINVAL  # lens NULL
    assert lib.blk_attn_decode(C.byref(d), FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 16, 1,
                               None) == _abi.BLK_EWORKSPACE
    ali = _abi.DecodeDesc(1, 16, 12, 12, 64, -1.0, 1)  # standard slopes need 2^k heads
    assert lib.blk_attn_decode(C.byref(ali), FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 1 << 30, 1,
                               None) == _abi.BLK_EUNSUPPORTED


def test_q8_validation(lib):
    st = lib.blk_q8_0_quantize(FAKE, 16, 48, FAKE, FAKE, _abi.BLK_BF16, None)
    assert st == _abi.BLK_EINVAL and "multiple of 32" in _err(lib)
    st = lib.blk_q8_0_quantize(FAKE, 16, 64, None, FAKE, _abi.BLK_BF16, None)
    assert st == _abi.BLK_EINVAL and "q is NULL" in _err(lib)
    assert lib.blk_q8_0_quantize(FAKE, 0, 64, FAKE, FAKE, _abi.BLK_BF16, None) == _abi.BLK_OK
    st = lib.blk_linear_q8_0(FAKE, FAKE, FAKE, None, None, None, FAKE, 4, 64, 40, _abi.BLK_BF16, None)
    assert st == _abi.BLK_EINVAL and "multiple of 32" in _err(lib)
    st = lib.blk_linear_q8_0(FAKE, FAKE, FAKE + 8, None, None, None, FAKE, 4, 64, 64, _abi.BLK_BF16, None)
    assert st == _abi.BLK_EINVAL and "aligned" in _err(lib)
    assert lib.blk_linear_q8_0(FAKE, FAKE, FAKE, None, None, None, FAKE, 0, 64, 64,
                               _abi.BLK_F16, None) == _abi.BLK_OK


def test_q8_block_slot_rules(lib):
    """blk_forward_q8_0 takes its projections from the Q8_0 struct only: a
    dense projection slot is rejected, a missing Q8_0 slot too, and widths
    must be multiples of 32."""
    import workloads
    from alibi_attention_block_gb300 import block_desc
    cfg = workloads.scaled(workloads.BLOCK_CONFIGS["stablelm2_1p6b"], batch=1, seq=64, hidden=256,
                           n_heads=4, n_kv_heads=4, intermediate=704)
    desc = block_desc(cfg, 1, 64)
    dense = {n: FAKE for n in ("attn_norm_w", "attn_norm_b", "mlp_norm_w", "mlp_norm_b", "b_qkv")}
    q8 = {n: FAKE for n in _abi.Q8_SLOTS}
    w = _abi.BlockWeights(*[dense.get(n) for n in _abi.WEIGHT_SLOTS])
    qw = _abi.Q8Weights(*[q8.get(n) for n in _abi.Q8_SLOTS])
    ws = C.c_size_t(0)
    assert lib.blk_forward_workspace_size(C.byref(desc), C.byref(ws)) == _abi.BLK_OK
    call = lambda w_, q_: lib.blk_forward_q8_0(C.byref(desc), C.byref(w_), C.byref(q_), FAKE,  # noqa: E731
                                               FAKE + 4096, FAKE, ws.value, _abi.BLK_BF16, None)
    w2 = _abi.BlockWeights(*[dict(dense, w_o=FAKE).get(n) for n in _abi.WEIGHT_SLOTS])
    assert call(w2, qw) == _abi.BLK_EINVAL and "w_o" in _err(lib)
    q2 = _abi.Q8Weights(*[dict(q8, d_down=None).get(n) for n in _abi.Q8_SLOTS])
    assert call(w, q2) == _abi.BLK_EINVAL and "d_down" in _err(lib)
    odd = block_desc(workloads.scaled(cfg, intermediate=688), 1, 64)
    assert lib.blk_forward_q8_0(C.byref(odd), C.byref(w), C.byref(qw), FAKE, FAKE + 4096, FAKE,
                                1 << 30, _abi.BLK_BF16, None) == _abi.BLK_EINVAL
    assert "multiples of 32" in _err(lib)
