"""Failure detection without a GPU fault: a bounded in-kernel wait that runs
out reports BLK_ETIMEOUT through the device error word, and the context stays
usable for the next launch."""
import ctypes as C

import pytest
import torch

import alibi_attention_block_gb300 as blk
from alibi_attention_block_gb300 import _abi, build
from tests.parity import check, f64, to_dev
from workloads import draw

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_is_reported_and_cleared():
    build.build()
    lib = _abi.load()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.blk_check_device_status(stream) == _abi.BLK_OK
    assert lib.blk_selftest_bounded_wait(20_000_000, stream) == _abi.BLK_OK   # 20 ms limit
    assert lib.blk_check_device_status(stream) == _abi.BLK_ETIMEOUT
    assert b"gave up" in lib.blk_last_error()
    assert lib.blk_check_device_status(stream) == _abi.BLK_OK                 # cleared
    # the context still runs kernels correctly
    x = draw((64, 1024), "bf16", 3)
    g = draw((1024,), "bf16", 4, "g")
    y = blk.rmsnorm(to_dev(x), to_dev(g), eps=1e-6)
    blk.check_device_status()
    import oracle
    check(y, oracle.rms_norm(f64(x), f64(g), 1e-6), "after timeout", unit_scale=True)


def test_bounded_wait_limits_are_validated():
    lib = _abi.load()
    assert lib.blk_selftest_bounded_wait(10, None) == _abi.BLK_EINVAL
