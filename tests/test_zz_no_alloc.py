"""blk_mlp_noalloc through the C ABI: the MLP for callers that cannot
allocate device memory (an engine or plugin host that owns all device memory
after start-up, or latency-bound code that cannot take cudaMalloc's implicit
synchronisation). Its activation lives in the library's fixed 32 MiB device
array instead of a caller workspace, so its output must equal blk_mlp's, call
after call, and meet the MLP's parity gate against the fp64 oracle.

This file is collected last on purpose, and passes both on its own in a fresh
process and after the other GPU tests."""
import ctypes as C

import pytest
import torch

import oracle
from alibi_attention_block_gb300 import _abi, build
from tests.parity import check, f64, to_dev
from workloads import draw

pytestmark = pytest.mark.gpu


def _ptr(t):
    return None if t is None else t.data_ptr()


@pytest.mark.parametrize("act,T,D,F,dt", [("swiglu", 300, 512, 1024, "bf16"),
                                          ("gelu_tanh", 200, 256, 1024, "fp16")])
def test_noalloc_mlp_matches_workspace_mlp_twice(act, T, D, F, dt):
    build.build()
    lib = _abi.load()
    lib.blk_mlp_noalloc.restype = C.c_int
    lib.blk_mlp_noalloc.argtypes = [C.POINTER(_abi.MlpDesc)] + [C.c_void_p] * 9 + [C.c_int, C.c_void_p]
    seed = 7 * T + F
    x = to_dev(draw((T, D), dt, seed))
    w_up = to_dev(draw((F, D), dt, seed + 1, "w"))
    w_down = to_dev(draw((D, F), dt, seed + 2, "w"))
    w_gate = to_dev(draw((F, D), dt, seed + 3, "w")) if act == "swiglu" else None
    b_up = to_dev(draw((F,), dt, seed + 4, "b")) if act != "swiglu" else None
    b_down = to_dev(draw((D,), dt, seed + 5, "b"))
    res = to_dev(draw((T, D), dt, seed + 6))
    code = _abi.BLK_ACT_SWIGLU if act == "swiglu" else _abi.BLK_ACT_GELU_TANH
    desc = _abi.MlpDesc(T, D, F, code)
    dtc = _abi.BLK_F16 if dt == "fp16" else _abi.BLK_BF16
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)

    ws_bytes = C.c_size_t(0)
    _abi.check(lib.blk_mlp_workspace_size(C.byref(desc), C.byref(ws_bytes)), "blk_mlp_workspace_size")
    ws = torch.empty(ws_bytes.value, dtype=torch.uint8, device="cuda")
    ref = torch.empty_like(x)
    _abi.check(lib.blk_mlp(C.byref(desc), _ptr(x), _ptr(w_gate), _ptr(w_up), _ptr(b_up),
                           _ptr(w_down), _ptr(b_down), _ptr(res), None, _ptr(ref), _ptr(ws),
                           ws_bytes.value, dtc, stream), "blk_mlp")
    w = {"w_up": f64(w_up), "w_down": f64(w_down), "b_down": f64(b_down)}
    if act == "swiglu":
        w["w_gate"] = f64(w_gate)
    else:
        w["b_up"] = f64(b_up)
    _, m = oracle.mlp(f64(x), w, act)
    exact = m + f64(res)
    for _ in range(2):
        y = torch.full_like(x, float("nan"))
        _abi.check(lib.blk_mlp_noalloc(C.byref(desc), _ptr(x), _ptr(w_gate), _ptr(w_up), _ptr(b_up),
                                       _ptr(w_down), _ptr(b_down), _ptr(res), None, _ptr(y), dtc,
                                       stream), "blk_mlp_noalloc")
        torch.cuda.synchronize()
        check(y, ref.double().cpu().numpy(), f"noalloc {act}")
        check(y, exact, f"noalloc {act} vs oracle")
    _abi.check(lib.blk_check_device_status(stream), "blk_check_device_status")


def test_noalloc_mlp_rejects_oversize():
    build.build()
    lib = _abi.load()
    desc = _abi.MlpDesc(8192, 2048, 5632, _abi.BLK_ACT_SWIGLU)   # 92 MB of activation
    fake = 0x100000
    st = lib.blk_mlp_noalloc(C.byref(desc), fake, fake, fake, None, fake, None, None, None, fake,
                             _abi.BLK_BF16, None)
    assert st == _abi.BLK_EWORKSPACE
    assert b"exceeds" in lib.blk_last_error()
