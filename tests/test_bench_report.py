"""bench.py's roofline bookkeeping on CPU: which measured peak a kernel is
held to, the spec-derived tensor peak's arithmetic, and the per-kernel
rates."""
import pytest

import bench
import workloads

CFG = workloads.BLOCK_CONFIGS["stablelm2_1p6b"]
PEAKS = dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, sm_max_mhz=2070.0,
             source="measured")
SPEC = {"tflops": 152 * 8192 * 2070e6 / 1e12, "derivation": "152 SMs x 8192 x 2070 MHz"}


def _kernel_ms():
    # gate/up dominant at 0.2 ms
    return {"input_norm": 0.02, "qkv": 0.13, "attention": 0.09, "o_proj": 0.06,
            "mlp_norm": 0.02, "mlp_up": 0.2, "mlp_down": 0.14}


def test_short_timed_region_uses_the_burst_peak():
    rep = bench._report(CFG, _kernel_ms(), 0.66, 0.014, PEAKS, SPEC)
    roof = rep["roofline"]
    assert roof["kernel"] == "mlp_up" and roof["bound"] == "tensor"
    flops = 2 * CFG.tokens * CFG.hidden * 2 * CFG.intermediate
    assert roof["achieved"] == pytest.approx(flops / 0.2e-3 / 1e12)
    assert roof["peak"] == 1900.0 and "burst" in roof["peak_source"]
    assert roof["frac"] == pytest.approx(roof["achieved"] / 1900.0)
    assert roof["frac_of_spec_peak"] == pytest.approx(roof["achieved"] / SPEC["tflops"])


def test_long_timed_region_uses_the_sustained_peak():
    roof = bench._report(CFG, _kernel_ms(), 0.66, 2.5, PEAKS, SPEC)["roofline"]
    assert roof["peak"] == 1700.0 and "sustained" in roof["peak_source"]


def test_attention_fractions_and_spec_peak():
    rep = bench._report(CFG, _kernel_ms(), 0.66, 0.014, PEAKS, SPEC)
    at = 4 * CFG.batch * CFG.n_heads * CFG.head_dim * CFG.seq * (CFG.seq + 1) // 2 / 0.09e-3 / 1e12
    assert rep["attention"]["tflops"] == pytest.approx(at)
    assert rep["attention"]["frac_of_spec_peak"] == pytest.approx(at / SPEC["tflops"])
    assert SPEC["tflops"] == pytest.approx(2577.6, rel=1e-3)
    assert rep["kernels"]["input_norm"]["gbs"] == pytest.approx(2 * CFG.tokens * CFG.hidden * 2 / 0.02e-3 / 1e9, rel=1e-3)
