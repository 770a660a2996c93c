"""ctypes mirror of include/blk.h: structs, enums and function prototypes.

Argument marshalling only. Loading fails loudly when ``lib/libblk.so`` is
missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libblk.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "blk.h")

BLK_OK, BLK_EINVAL, BLK_EUNSUPPORTED, BLK_ECUDA, BLK_ETIMEOUT, BLK_EWORKSPACE = range(6)
BLK_F16, BLK_BF16 = 0, 1
BLK_QKV_STACKED, BLK_QKV_HEAD_INTERLEAVED = 0, 1
BLK_QKNORM_NONE, BLK_QKNORM_RMS_FULL, BLK_QKNORM_LN_PER_HEAD = 0, 1, 2
BLK_NORM_LAYERNORM, BLK_NORM_RMS = 0, 1
BLK_NORM_PRE, BLK_NORM_POST = 0, 1
BLK_RESIDUAL_SEQUENTIAL, BLK_RESIDUAL_PARALLEL = 0, 1
BLK_ACT_SWIGLU, BLK_ACT_GELU_TANH = 0, 1

vp = C.c_void_p
i64 = C.c_int64
i32 = C.c_int32
f32 = C.c_float


class QkvDesc(C.Structure):
    _fields_ = [("batch", i64), ("seq", i64), ("hidden", i64), ("n_heads", i64),
                ("n_kv_heads", i64), ("head_dim", i64), ("qkv_layout", i32), ("qk_norm", i32),
                ("qk_norm_eps", f32), ("rotary_span", i32), ("rope_base", f32)]


class AttnDesc(C.Structure):
    _fields_ = [("batch", i64), ("seq", i64), ("n_heads", i64), ("n_kv_heads", i64),
                ("head_dim", i64), ("softmax_scale", f32), ("causal", i32), ("alibi", i32)]


class DecodeDesc(C.Structure):
    _fields_ = [("batch", i64), ("max_seq", i64), ("n_heads", i64), ("n_kv_heads", i64),
                ("head_dim", i64), ("softmax_scale", f32), ("alibi", i32)]


class MlpDesc(C.Structure):
    _fields_ = [("tokens", i64), ("hidden", i64), ("intermediate", i64), ("act", i32)]


class BlockDesc(C.Structure):
    _fields_ = [("qkv", QkvDesc), ("norm_kind", i32), ("norm_place", i32), ("residual", i32),
                ("eps", f32), ("alibi", i32), ("intermediate", i64), ("act", i32)]


WEIGHT_SLOTS = ("attn_norm_w", "attn_norm_b", "mlp_norm_w", "mlp_norm_b", "post_attn_norm_w",
                "post_mlp_norm_w", "w_qkv", "b_qkv", "q_norm_w", "k_norm_w", "w_o", "b_o",
                "w_gate", "w_up", "b_up", "w_down", "b_down", "alibi_slopes")


class BlockWeights(C.Structure):
    _fields_ = [(n, vp) for n in WEIGHT_SLOTS]


Q8_SLOTS = ("q_qkv", "q_o", "q_gate", "q_up", "q_down", "d_qkv", "d_o", "d_gate", "d_up",
            "d_down")


class Q8Weights(C.Structure):
    _fields_ = [(n, vp) for n in Q8_SLOTS]


class ModelDesc(C.Structure):
    _fields_ = [("block", BlockDesc), ("n_layers", i32), ("vocab", i64), ("embed_norm", i32),
                ("final_norm", i32), ("final_eps", f32)]


class ModelWeights(C.Structure):
    _fields_ = [("embed", vp), ("embed_norm_w", vp), ("embed_norm_b", vp),
                ("layers", C.POINTER(BlockWeights)), ("final_norm_w", vp), ("final_norm_b", vp),
                ("lm_head", vp)]


_PROTOS = {
    "blk_status_string": (C.c_char_p, [C.c_int]),
    "blk_last_error": (C.c_char_p, []),
    "blk_version": (C.c_int, []),
    "blk_check_device_status": (C.c_int, [vp]),
    "blk_selftest_bounded_wait": (C.c_int, [C.c_uint64, vp]),
    "blk_layernorm_bias": (C.c_int, [vp, vp, vp, vp, vp, i64, i64, f32, C.c_int, vp]),
    "blk_rmsnorm": (C.c_int, [vp, vp, vp, vp, i64, i64, f32, C.c_int, vp]),
    "blk_qkv_bias_rope_partial": (C.c_int, [C.POINTER(QkvDesc), vp, vp, vp, vp, vp, vp, vp, vp,
                                            C.c_int, vp]),
    "blk_rope_inplace": (C.c_int, [vp, vp, i64, i64, i64, i64, i32, f32, C.c_int, vp]),
    "blk_attn_prefill": (C.c_int, [C.POINTER(AttnDesc), vp, vp, vp, vp, vp, C.c_int, vp]),
    "blk_linear": (C.c_int, [vp, vp, vp, vp, vp, vp, i64, i64, i64, C.c_int, vp]),
    "blk_mlp_workspace_size": (C.c_int, [C.POINTER(MlpDesc), C.POINTER(C.c_size_t)]),
    "blk_mlp": (C.c_int, [C.POINTER(MlpDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, C.c_size_t,
                          C.c_int, vp]),
    "blk_mlp_noalloc": (C.c_int, [C.POINTER(MlpDesc), vp, vp, vp, vp, vp, vp, vp, vp, vp, C.c_int,
                                  vp]),
    "blk_forward_workspace_size": (C.c_int, [C.POINTER(BlockDesc), C.POINTER(C.c_size_t)]),
    "blk_forward_q8_0_workspace_size": (C.c_int, [C.POINTER(BlockDesc), C.POINTER(C.c_size_t)]),
    "blk_forward": (C.c_int, [C.POINTER(BlockDesc), C.POINTER(BlockWeights), vp, vp, vp,
                              C.c_size_t, C.c_int, vp]),
    "blk_attn_decode_workspace_size": (C.c_int, [C.POINTER(DecodeDesc), C.POINTER(C.c_size_t)]),
    "blk_attn_decode": (C.c_int, [C.POINTER(DecodeDesc), vp, vp, vp, vp, vp, vp, vp, C.c_size_t,
                                  C.c_int, vp]),
    "blk_forward_graph_create": (C.c_int, [C.POINTER(BlockDesc), C.POINTER(BlockWeights), vp, vp,
                                           vp, C.c_size_t, C.c_int, C.POINTER(vp), C.c_int,
                                           C.POINTER(i32), C.POINTER(C.c_int), C.POINTER(vp)]),
    "blk_graph_launch": (C.c_int, [vp, vp]),
    "blk_graph_set_events": (C.c_int, [vp, C.POINTER(vp), C.c_int]),
    "blk_graph_destroy": (C.c_int, [vp]),
    "blk_forward_host": (C.c_int, [C.POINTER(BlockDesc), C.POINTER(BlockWeights), vp, vp, vp, vp,
                                   vp, C.c_size_t, i32, C.c_int, vp]),
    "blk_model_workspace_size": (C.c_int, [C.POINTER(ModelDesc), C.POINTER(C.c_size_t)]),
    "blk_model_forward": (C.c_int, [C.POINTER(ModelDesc), C.POINTER(ModelWeights), vp, vp, vp,
                                    C.c_size_t, C.c_int, vp]),
    "blk_host_pipe_mem_size": (C.c_int, [C.POINTER(BlockDesc), i32, C.POINTER(C.c_size_t)]),
    "blk_host_pipe_create": (C.c_int, [C.POINTER(BlockDesc), i32, C.c_int, vp, C.c_size_t,
                                       C.POINTER(vp)]),
    "blk_host_pipe_submit": (C.c_int, [vp, C.POINTER(BlockWeights), vp, vp, vp]),
    "blk_host_pipe_flush": (C.c_int, [vp, vp]),
    "blk_host_pipe_destroy": (C.c_int, [vp]),
    "blk_forward_ex": (C.c_int, [C.POINTER(BlockDesc), C.POINTER(BlockWeights), vp, vp, vp,
                                 C.c_size_t, C.c_int, vp, C.POINTER(vp), C.c_int,
                                 C.POINTER(i32), C.POINTER(C.c_int)]),
    "blk_q8_0_quantize": (C.c_int, [vp, i64, i64, vp, vp, C.c_int, vp]),
    "blk_linear_q8_0": (C.c_int, [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, C.c_int, vp]),
    "blk_forward_q8_0": (C.c_int, [C.POINTER(BlockDesc), C.POINTER(BlockWeights),
                                   C.POINTER(Q8Weights), vp, vp, vp, C.c_size_t, C.c_int, vp]),
    "blk_forward_q8_0_ex": (C.c_int, [C.POINTER(BlockDesc), C.POINTER(BlockWeights),
                                      C.POINTER(Q8Weights), vp, vp, vp, C.c_size_t, C.c_int, vp,
                                      C.POINTER(vp), C.c_int, C.POINTER(i32), C.POINTER(C.c_int)]),
}

STEP_NAMES = ("input_norm", "qkv", "qk_norm_rope", "attention", "o_proj", "post_attn_norm",
              "mlp_norm", "mlp_up", "mlp_down", "post_mlp_norm", "q8_dequant")

_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/blk.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**(blk_\w+)\s*\(", text,
                                 flags=re.M)))


def load() -> C.CDLL:
    """Load lib/libblk.so (built by ``build()``) and set every prototype."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: run alibi_attention_block_gb300.build.build() "
                           "(the CUDA library is required; there is no fallback)")
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in _PROTOS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class BlkError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        self.status = status
        names = ["BLK_OK", "BLK_EINVAL", "BLK_EUNSUPPORTED", "BLK_ECUDA", "BLK_ETIMEOUT",
                 "BLK_EWORKSPACE"]
        label = names[status] if 0 <= status < len(names) else str(status)
        super().__init__(f"{fn} -> {label}: {msg}")


def check(status: int, fn: str) -> None:
    if status != BLK_OK:
        raise BlkError(status, fn, load().blk_last_error().decode())
