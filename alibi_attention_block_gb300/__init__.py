"""GB300 (sm_103a) prefill forward of one decoder block.

A thin torch-facing binding over the C ABI in ``include/blk.h``
(``lib/libblk.so``): it checks tensors, passes device pointers and the current
CUDA stream, and raises ``BlkError`` on a non-OK status. Every step of the
block runs in the library's CUDA kernels; nothing here computes.

Block variants (nnterp encyclopedia "stablelm", 03 Notes; "OLMo-2: reordered
(post) normalization", section 1; "Bloom in a sovereign engine",
Contribution): sequential pre-norm, parallel residual, reordered post-norm;
LayerNorm-with-bias or RMSNorm; stacked or head-interleaved QKV with bias;
full-width or per-head qk-norm; partial NeoX rotary or ALiBi.
"""
from __future__ import annotations

import ctypes as C

import torch

from . import _abi
from ._abi import BlkError  # noqa: F401

__all__ = ["layernorm_bias", "rmsnorm", "qkv_bias_rope_partial", "rope_inplace", "attn_prefill",
           "attn_decode", "attn_decode_workspace_size", "decode_desc",
           "linear", "mlp", "block_desc", "forward_workspace_size", "forward_q8_0_workspace_size", "forward", "forward_host", "ForwardGraph", "HostPipe", "model_desc",
           "model_workspace_size", "model_forward",
           "check_device_status", "BlkError", "library_path"]

library_path = _abi.LIB_PATH


def _lib():
    return _abi.load()


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return _abi.BLK_F16
    if t.dtype == torch.bfloat16:
        return _abi.BLK_BF16
    raise TypeError(f"storage dtype must be float16 or bfloat16, got {t.dtype}")


def _p(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError("tensors passed to the block library must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the block library must be contiguous")
    return t.data_ptr()


def _same(dt_tensor, *ts):
    for t in ts:
        if t is not None and t.dtype != dt_tensor.dtype:
            raise TypeError(f"all tensors must share dtype {dt_tensor.dtype}, got {t.dtype}")


def _stream():
    return C.c_void_p(torch.cuda.current_stream().cuda_stream)


def layernorm_bias(x, gamma, beta=None, residual=None, eps=1e-5, out=None):
    """y = LN(x) * gamma + beta [+ residual] over the last axis."""
    _same(x, gamma, beta, residual, out)
    out = torch.empty_like(x) if out is None else out
    cols = x.shape[-1]
    _abi.check(_lib().blk_layernorm_bias(_p(x), _p(residual), _p(gamma), _p(beta), _p(out),
                                         x.numel() // cols, cols, eps, _dt(x), _stream()),
               "blk_layernorm_bias")
    return out


def rmsnorm(x, weight, residual=None, eps=1e-6, out=None):
    """y = x / rms(x) * weight [+ residual] over the last axis."""
    _same(x, weight, residual, out)
    out = torch.empty_like(x) if out is None else out
    cols = x.shape[-1]
    _abi.check(_lib().blk_rmsnorm(_p(x), _p(residual), _p(weight), _p(out), x.numel() // cols,
                                  cols, eps, _dt(x), _stream()), "blk_rmsnorm")
    return out


_LAYOUT = {"stacked": _abi.BLK_QKV_STACKED, "head_interleaved": _abi.BLK_QKV_HEAD_INTERLEAVED}
_QKN = {"none": _abi.BLK_QKNORM_NONE, "rms_full": _abi.BLK_QKNORM_RMS_FULL,
        "ln_per_head": _abi.BLK_QKNORM_LN_PER_HEAD}


def _qkv_desc(batch, seq, hidden, n_heads, n_kv_heads, head_dim, layout, qk_norm, qk_norm_eps,
              rotary_span, rope_base):
    return _abi.QkvDesc(batch, seq, hidden, n_heads, n_kv_heads, head_dim, _LAYOUT[layout],
                        _QKN[qk_norm], qk_norm_eps, rotary_span, rope_base)


def qkv_bias_rope_partial(x, w_qkv, b_qkv=None, *, n_heads, n_kv_heads, head_dim,
                          layout="stacked", qk_norm="none", qk_norm_eps=1e-5, rotary_span=0,
                          rope_base=10000.0, q_norm_w=None, k_norm_w=None):
    """x [B, S, D] -> head-split q [B, H, S, d], k and v [B, Hk, S, d]."""
    _same(x, w_qkv, b_qkv, q_norm_w, k_norm_w)
    B, S, D = x.shape
    desc = _qkv_desc(B, S, D, n_heads, n_kv_heads, head_dim, layout, qk_norm, qk_norm_eps,
                     rotary_span, rope_base)
    q = torch.empty((B, n_heads, S, head_dim), dtype=x.dtype, device=x.device)
    k = torch.empty((B, n_kv_heads, S, head_dim), dtype=x.dtype, device=x.device)
    v = torch.empty_like(k)
    _abi.check(_lib().blk_qkv_bias_rope_partial(C.byref(desc), _p(x), _p(w_qkv), _p(b_qkv),
                                                _p(q_norm_w), _p(k_norm_w), _p(q), _p(k), _p(v),
                                                _dt(x), _stream()), "blk_qkv_bias_rope_partial")
    return q, k, v


def rope_inplace(x, bias=None, rotary_span=0, rope_base=10000.0):
    """In place on x [B, n, S, d]: x += bias (per head), then partial NeoX rotary."""
    _same(x, bias)
    B, n, S, d = x.shape
    _abi.check(_lib().blk_rope_inplace(_p(x), _p(bias), B, n, S, d, rotary_span, rope_base,
                                       _dt(x), _stream()), "blk_rope_inplace")
    return x


def attn_prefill(q, k, v, alibi=False, slopes=None, scale=None, out=None):
    """Causal attention: q [B, H, S, d], k/v [B, Hk, S, d] -> o [B, S, H, d]."""
    _same(q, k, v, out)
    B, H, S, d = q.shape
    Hk = k.shape[1]
    if slopes is not None and slopes.dtype != torch.float32:
        raise TypeError("ALiBi slopes are fp32")
    desc = _abi.AttnDesc(B, S, H, Hk, d, -1.0 if scale is None else scale, 1, 1 if alibi else 0)
    o = torch.empty((B, S, H, d), dtype=q.dtype, device=q.device) if out is None else out
    _abi.check(_lib().blk_attn_prefill(C.byref(desc), _p(q), _p(k), _p(v), _p(slopes), _p(o),
                                       _dt(q), _stream()), "blk_attn_prefill")
    return o


def decode_desc(batch, max_seq, n_heads, n_kv_heads, head_dim, alibi=False, scale=None):
    return _abi.DecodeDesc(batch, max_seq, n_heads, n_kv_heads, head_dim,
                           -1.0 if scale is None else scale, 1 if alibi else 0)


def attn_decode_workspace_size(desc) -> int:
    need = C.c_size_t(0)
    _abi.check(_lib().blk_attn_decode_workspace_size(C.byref(desc), C.byref(need)),
               "blk_attn_decode_workspace_size")
    return need.value


def attn_decode(q, k_cache, v_cache, lens, alibi=False, slopes=None, scale=None, out=None,
                workspace=None):
    """One decode step: q [B, H, d] (newest token of each sequence, at position
    lens[b] - 1) against k/v caches [B, Hk, S_max, d]; lens int32 [B] on the
    device. Returns o [B, H, d]."""
    _same(q, k_cache, v_cache, out)
    B, H, d = q.shape
    Hk, S_max = k_cache.shape[1], k_cache.shape[2]
    if lens.dtype != torch.int32:
        raise TypeError("lens are int32")
    if slopes is not None and slopes.dtype != torch.float32:
        raise TypeError("ALiBi slopes are fp32")
    desc = decode_desc(B, S_max, H, Hk, d, alibi, scale)
    if workspace is None:
        workspace = torch.empty(attn_decode_workspace_size(desc), dtype=torch.uint8,
                                device=q.device)
    o = torch.empty_like(q) if out is None else out
    _abi.check(_lib().blk_attn_decode(C.byref(desc), _p(q), _p(k_cache), _p(v_cache), _p(lens),
                                      _p(slopes), _p(o), _p(workspace), workspace.numel(), _dt(q),
                                      _stream()), "blk_attn_decode")
    return o


def linear(x, w, bias=None, res1=None, res2=None, out=None):
    """y = x W^T [+ bias] [+ res1] [+ res2]; x [..., k], w [n, k]."""
    _same(x, w, bias, res1, res2, out)
    k = x.shape[-1]
    n = w.shape[0]
    m = x.numel() // k
    out = torch.empty((*x.shape[:-1], n), dtype=x.dtype, device=x.device) if out is None else out
    _abi.check(_lib().blk_linear(_p(x), _p(w), _p(bias), _p(res1), _p(res2), _p(out), m, n, k,
                                 _dt(x), _stream()), "blk_linear")
    return out


def q8_0_quantize(w):
    """Q8_0 of a weight w [n, k] (k % 32 == 0) on the GPU: (codes int8
    [n, k], scales fp16 [k/32, n], block-major)."""
    n, k = w.shape
    q = torch.empty((n, k), dtype=torch.int8, device=w.device)
    d = torch.empty((k // 32, n), dtype=torch.float16, device=w.device)
    _abi.check(_lib().blk_q8_0_quantize(_p(w), n, k, _p(q), _p(d), _dt(w), _stream()),
               "blk_q8_0_quantize")
    return q, d


def linear_q8_0(x, q, d, bias=None, res1=None, res2=None, out=None):
    """y = x W^T [+ bias] [+ res1] [+ res2] with W in Q8_0 form (q, d)."""
    _same(x, bias, res1, res2, out)
    if q.dtype != torch.int8 or d.dtype != torch.float16:
        raise TypeError("Q8_0 codes are int8 and scales fp16")
    k = x.shape[-1]
    n = q.shape[0]
    m = x.numel() // k
    out = torch.empty((*x.shape[:-1], n), dtype=x.dtype, device=x.device) if out is None else out
    _abi.check(_lib().blk_linear_q8_0(_p(x), _p(q), _p(d), _p(bias), _p(res1), _p(res2), _p(out),
                                      m, n, k, _dt(x), _stream()), "blk_linear_q8_0")
    return out


def mlp(x, w_up, w_down, w_gate=None, b_up=None, b_down=None, res1=None, res2=None,
        act="swiglu", workspace=None, out=None):
    """SwiGLU or GELU(tanh) MLP with optional biases and residual adds."""
    _same(x, w_up, w_down, w_gate, b_up, b_down, res1, res2, out)
    D = x.shape[-1]
    T = x.numel() // D
    F = w_up.shape[0]
    desc = _abi.MlpDesc(T, D, F, _abi.BLK_ACT_SWIGLU if act == "swiglu" else _abi.BLK_ACT_GELU_TANH)
    need = C.c_size_t(0)
    _abi.check(_lib().blk_mlp_workspace_size(C.byref(desc), C.byref(need)), "blk_mlp_workspace_size")
    if workspace is None:
        workspace = torch.empty(need.value, dtype=torch.uint8, device=x.device)
    out = torch.empty_like(x) if out is None else out
    _abi.check(_lib().blk_mlp(C.byref(desc), _p(x), _p(w_gate), _p(w_up), _p(b_up), _p(w_down),
                              _p(b_down), _p(res1), _p(res2), _p(out), _p(workspace),
                              workspace.numel(), _dt(x), _stream()), "blk_mlp")
    return out


def block_desc(cfg, batch: int, seq: int) -> _abi.BlockDesc:
    """Descriptor from a config object with the block's fields (hidden,
    n_heads, n_kv_heads, head_dim, intermediate, norm, norm_place, residual,
    eps, qkv_layout, qk_norm, qk_norm_eps, rotary_span, rope_base, alibi, act)."""
    q = _qkv_desc(batch, seq, cfg.hidden, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim,
                  cfg.qkv_layout, cfg.qk_norm, cfg.qk_norm_eps, cfg.rotary_span, cfg.rope_base)
    return _abi.BlockDesc(
        q,
        _abi.BLK_NORM_LAYERNORM if cfg.norm == "layernorm" else _abi.BLK_NORM_RMS,
        _abi.BLK_NORM_PRE if cfg.norm_place == "pre" else _abi.BLK_NORM_POST,
        _abi.BLK_RESIDUAL_SEQUENTIAL if cfg.residual == "sequential" else _abi.BLK_RESIDUAL_PARALLEL,
        cfg.eps, 1 if cfg.alibi else 0, cfg.intermediate,
        _abi.BLK_ACT_SWIGLU if cfg.act == "swiglu" else _abi.BLK_ACT_GELU_TANH)


def forward_workspace_size(cfg, batch: int, seq: int) -> int:
    desc = block_desc(cfg, batch, seq)
    need = C.c_size_t(0)
    _abi.check(_lib().blk_forward_workspace_size(C.byref(desc), C.byref(need)),
               "blk_forward_workspace_size")
    return need.value


def forward(cfg, weights: dict, x, workspace=None, out=None):
    """The block's prefill forward: x [B, S, D] -> y [B, S, D].

    weights maps slot names (``attn_norm_w``, ``w_qkv``, ...) to CUDA tensors;
    absent slots are NULL. workspace: a uint8 CUDA tensor of at least
    ``forward_workspace_size`` bytes (allocated here when None).
    """
    B, S, _ = x.shape
    desc = block_desc(cfg, B, S)
    ws_need = forward_workspace_size(cfg, B, S)
    if workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=x.device)
    unknown = set(weights) - set(_abi.WEIGHT_SLOTS)
    if unknown:
        raise KeyError(f"unknown weight slots: {sorted(unknown)}")
    for name, t in weights.items():
        if name != "alibi_slopes":
            _same(x, t)
    w = _abi.BlockWeights(*[_p(weights.get(n)) for n in _abi.WEIGHT_SLOTS])
    out = torch.empty_like(x) if out is None else out
    _abi.check(_lib().blk_forward(C.byref(desc), C.byref(w), _p(x), _p(out), _p(workspace),
                                  workspace.numel(), _dt(x), _stream()), "blk_forward")
    return out


Q8_PROJECTIONS = ("qkv", "o", "gate", "up", "down")


def forward_q8_0_workspace_size(cfg, batch: int, seq: int) -> int:
    """Workspace bytes of blk_forward_q8_0's dequantize-once path."""
    desc = block_desc(cfg, batch, seq)
    need = C.c_size_t(0)
    _abi.check(_lib().blk_forward_q8_0_workspace_size(C.byref(desc), C.byref(need)),
               "blk_forward_q8_0_workspace_size")
    return need.value


def forward_q8_0(cfg, weights: dict, q8: dict, x, workspace=None, out=None):
    """The block with Q8_0 projection weights (blk_forward_q8_0). weights:
    the non-projection slots as for ``forward``; q8 maps ``q_<name>`` (int8
    codes) and ``d_<name>`` (fp16 scales) for name in qkv, o, gate, up, down
    (gate for SwiGLU only). workspace: ``forward_q8_0_workspace_size`` bytes
    (allocated here when None) take the dequantize-once path from 512 tokens
    on; ``forward_workspace_size`` bytes keep the W8A16 GEMMs."""
    B, S, _ = x.shape
    desc = block_desc(cfg, B, S)
    if workspace is None:
        workspace = torch.empty(forward_q8_0_workspace_size(cfg, B, S), dtype=torch.uint8,
                                device=x.device)
    unknown = set(weights) - set(_abi.WEIGHT_SLOTS)
    if unknown:
        raise KeyError(f"unknown weight slots: {sorted(unknown)}")
    unknown = set(q8) - set(_abi.Q8_SLOTS)
    if unknown:
        raise KeyError(f"unknown Q8_0 slots: {sorted(unknown)}")
    for name, t in weights.items():
        if name != "alibi_slopes":
            _same(x, t)
    for name, t in q8.items():
        want = torch.int8 if name.startswith("q_") else torch.float16
        if t.dtype != want or not t.is_cuda or not t.is_contiguous():
            raise TypeError(f"{name}: expected a contiguous CUDA {want} tensor")
    w = _abi.BlockWeights(*[_p(weights.get(n)) for n in _abi.WEIGHT_SLOTS])
    qw = _abi.Q8Weights(*[_p(q8.get(n)) for n in _abi.Q8_SLOTS])
    out = torch.empty_like(x) if out is None else out
    _abi.check(_lib().blk_forward_q8_0(C.byref(desc), C.byref(w), C.byref(qw), _p(x), _p(out),
                                       _p(workspace), workspace.numel(), _dt(x), _stream()),
               "blk_forward_q8_0")
    return out


def model_desc(cfg, batch: int, seq: int, n_layers: int, vocab: int, embed_norm: bool = False,
               final_norm: str = "layernorm", final_eps: float = 1e-5) -> _abi.ModelDesc:
    """Descriptor of an n_layers stack of cfg's block between the token
    embedding and the logits (blk_model_forward)."""
    return _abi.ModelDesc(block_desc(cfg, batch, seq), n_layers, vocab, 1 if embed_norm else 0,
                          _abi.BLK_NORM_LAYERNORM if final_norm == "layernorm" else _abi.BLK_NORM_RMS,
                          final_eps)


def model_workspace_size(cfg, batch: int, seq: int, n_layers: int, vocab: int, **kw) -> int:
    need = C.c_size_t(0)
    desc = model_desc(cfg, batch, seq, n_layers, vocab, **kw)
    _abi.check(_lib().blk_model_workspace_size(C.byref(desc), C.byref(need)),
               "blk_model_workspace_size")
    return need.value


_MODEL_SLOTS = ("embed", "embed_norm_w", "embed_norm_b", "layers", "final_norm_w",
                "final_norm_b", "lm_head")


def model_forward(cfg, model_w: dict, tokens, vocab: int, embed_norm: bool = False,
                  final_norm: str = "layernorm", final_eps: float = 1e-5, workspace=None,
                  out=None):
    """Token ids [B, S] (int32, CUDA) -> logits [B, S, vocab] in the storage
    dtype, through len(model_w["layers"]) blocks. model_w holds ``embed``
    [vocab, hidden], optional ``embed_norm_w``/``embed_norm_b``, ``layers``
    (a list of block weight dicts), ``final_norm_w``, optional
    ``final_norm_b`` and ``lm_head`` [vocab, hidden]."""
    unknown = set(model_w) - set(_MODEL_SLOTS)
    if unknown:
        raise KeyError(f"unknown model slots: {sorted(unknown)}")
    if tokens.dtype != torch.int32 or not tokens.is_cuda or tokens.dim() != 2:
        raise ValueError("tokens must be a CUDA int32 tensor [batch, seq]")
    B, S = tokens.shape
    emb = model_w["embed"]
    layers = model_w.get("layers", [])
    desc = model_desc(cfg, B, S, len(layers), vocab, embed_norm, final_norm, final_eps)
    need = model_workspace_size(cfg, B, S, len(layers), vocab, embed_norm=embed_norm,
                                final_norm=final_norm, final_eps=final_eps)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=tokens.device)
    arr = (_abi.BlockWeights * max(1, len(layers)))()
    for i, lw in enumerate(layers):
        bad = set(lw) - set(_abi.WEIGHT_SLOTS)
        if bad:
            raise KeyError(f"unknown weight slots in layer {i}: {sorted(bad)}")
        for name, t in lw.items():
            if name != "alibi_slopes":
                _same(emb, t)
        arr[i] = _abi.BlockWeights(*[_p(lw.get(n)) for n in _abi.WEIGHT_SLOTS])
    for n in ("embed_norm_w", "embed_norm_b", "final_norm_w", "final_norm_b", "lm_head"):
        _same(emb, model_w.get(n))
    mw = _abi.ModelWeights(_p(emb), _p(model_w.get("embed_norm_w")), _p(model_w.get("embed_norm_b")),
                           arr, _p(model_w.get("final_norm_w")), _p(model_w.get("final_norm_b")),
                           _p(model_w.get("lm_head")))
    out = torch.empty((B, S, vocab), dtype=emb.dtype, device=tokens.device) if out is None else out
    _same(emb, out)
    _abi.check(_lib().blk_model_forward(C.byref(desc), C.byref(mw), C.c_void_p(tokens.data_ptr()),
                                        _p(out), _p(workspace), workspace.numel(), _dt(emb),
                                        _stream()), "blk_model_forward")
    return out


def forward_host(cfg, weights: dict, x_host, y_host=None, x_dev=None, y_dev=None,
                 workspace=None, n_chunks=2):
    """The block on host tensors (pinned CPU memory), copies overlapped with
    compute over n_chunks groups of sequences. x_dev / y_dev / workspace are
    reusable device staging buffers (allocated here when None). Returns
    y_host; it is ready when the current stream reaches the end of the call."""
    if x_host.is_cuda or not x_host.is_pinned():
        raise ValueError("x_host must be a pinned CPU tensor")
    B, S, _ = x_host.shape
    dev = torch.device("cuda", torch.cuda.current_device())
    y_host = torch.empty_like(x_host).pin_memory() if y_host is None else y_host
    if y_host.is_cuda or not y_host.is_pinned() or y_host.shape != x_host.shape:
        raise ValueError("y_host must be a pinned CPU tensor shaped like x_host")
    x_dev = torch.empty(x_host.shape, dtype=x_host.dtype, device=dev) if x_dev is None else x_dev
    y_dev = torch.empty_like(x_dev) if y_dev is None else y_dev
    _same(x_host, x_dev, y_dev)
    desc = block_desc(cfg, B, S)
    ws_need = forward_workspace_size(cfg, B, S)
    if workspace is None:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=dev)
    unknown = set(weights) - set(_abi.WEIGHT_SLOTS)
    if unknown:
        raise KeyError(f"unknown weight slots: {sorted(unknown)}")
    for name, t in weights.items():
        if name != "alibi_slopes":
            _same(x_host, t)
    w = _abi.BlockWeights(*[_p(weights.get(n)) for n in _abi.WEIGHT_SLOTS])
    _abi.check(_lib().blk_forward_host(C.byref(desc), C.byref(w), C.c_void_p(x_host.data_ptr()),
                                       C.c_void_p(y_host.data_ptr()), _p(x_dev), _p(y_dev),
                                       _p(workspace), workspace.numel(), n_chunks, _dt(x_host),
                                       _stream()), "blk_forward_host")
    return y_host


class HostPipe:
    """Block forwards over a stream of pinned host batches (blk_host_pipe_*):
    submit() enqueues one batch on the current stream and returns; batch n's
    copy in overlaps batch n-1's forward and its copy out batch n+1's.
    x_host must hold the batch at submit time; y_host is complete once the
    stream has passed a later flush(). Host tensors must stay alive until
    then; the pipe's device memory (staging slots and workspace) is
    allocated here."""

    def __init__(self, cfg, batch, seq, dtype=torch.bfloat16, depth=2):
        self.desc = block_desc(cfg, batch, seq)
        self.shape = (batch, seq, cfg.hidden)
        self.dtype = dtype
        n = C.c_size_t(0)
        _abi.check(_lib().blk_host_pipe_mem_size(C.byref(self.desc), depth, C.byref(n)),
                   "blk_host_pipe_mem_size")
        dev = torch.device("cuda", torch.cuda.current_device())
        self.mem = torch.empty(n.value, dtype=torch.uint8, device=dev)
        handle = C.c_void_p()
        dt = _abi.BLK_F16 if dtype == torch.float16 else _abi.BLK_BF16
        _abi.check(_lib().blk_host_pipe_create(C.byref(self.desc), depth, dt, _p(self.mem),
                                               n.value, C.byref(handle)), "blk_host_pipe_create")
        self._h = handle

    def submit(self, weights: dict, x_host, y_host):
        for t in (x_host, y_host):
            if t.is_cuda or not t.is_pinned() or tuple(t.shape) != self.shape or t.dtype != self.dtype:
                raise ValueError(f"host batches must be pinned CPU tensors {self.shape} {self.dtype}")
        unknown = set(weights) - set(_abi.WEIGHT_SLOTS)
        if unknown:
            raise KeyError(f"unknown weight slots: {sorted(unknown)}")
        w = _abi.BlockWeights(*[_p(weights.get(n)) for n in _abi.WEIGHT_SLOTS])
        _abi.check(_lib().blk_host_pipe_submit(self._h, C.byref(w), C.c_void_p(x_host.data_ptr()),
                                               C.c_void_p(y_host.data_ptr()), _stream()),
                   "blk_host_pipe_submit")

    def flush(self):
        _abi.check(_lib().blk_host_pipe_flush(self._h, _stream()), "blk_host_pipe_flush")

    def close(self):
        if self._h:
            _abi.check(_lib().blk_host_pipe_destroy(self._h), "blk_host_pipe_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class ForwardGraph:
    """The block forward recorded once as a CUDA graph (blk_forward_graph_create)
    for fixed tensors x, y, workspace and weights; launch() replays it on the
    current stream. The tensors must stay alive while the graph is used."""

    def __init__(self, cfg, weights: dict, x, y, workspace, events=None):
        B, S, _ = x.shape
        self._keep = (weights, x, y, workspace)
        self.desc = block_desc(cfg, B, S)
        unknown = set(weights) - set(_abi.WEIGHT_SLOTS)
        if unknown:
            raise KeyError(f"unknown weight slots: {sorted(unknown)}")
        for name, t in weights.items():
            if name != "alibi_slopes":
                _same(x, t)
        _same(x, y)
        self.w = _abi.BlockWeights(*[_p(weights.get(n)) for n in _abi.WEIGHT_SLOTS])
        ev = None
        n_ev = 0
        if events:
            ev = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
            n_ev = len(events)
        self.kinds = (C.c_int32 * 12)()  # a block makes at most 12 launches
        self.n_launches = C.c_int(0)
        handle = C.c_void_p()
        _abi.check(_lib().blk_forward_graph_create(C.byref(self.desc), C.byref(self.w), _p(x), _p(y),
                                                   _p(workspace), workspace.numel(), _dt(x), ev,
                                                   n_ev, self.kinds, C.byref(self.n_launches),
                                                   C.byref(handle)), "blk_forward_graph_create")
        self._h = handle

    def launch(self, events=None):
        """Replay on the current stream; events (torch.cuda.Event, created) replace
        the recorded ones for this and later launches."""
        if events is not None:
            arr = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
            _abi.check(_lib().blk_graph_set_events(self._h, arr, len(events)),
                       "blk_graph_set_events")
        _abi.check(_lib().blk_graph_launch(self._h, _stream()), "blk_graph_launch")

    def close(self):
        if self._h:
            _abi.check(_lib().blk_graph_destroy(self._h), "blk_graph_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def check_device_status():
    """Synchronise the current stream and raise if an in-kernel wait timed out."""
    _abi.check(_lib().blk_check_device_status(_stream()), "blk_check_device_status")
