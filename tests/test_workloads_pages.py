"""The workload table against facts the pages print (tests/golden/*.txt)."""
import os

import pytest

from workloads import ATTN_CONFIGS, BLOCK_CONFIGS, weight_shapes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read(name):
    out = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            out[k] = v
    return out


def test_stablelm2_1p6b_matches_printout_and_config():
    g = _read("stablelm2_1p6b_shapes.txt")
    c = BLOCK_CONFIGS["stablelm2_1p6b"]
    assert c.hidden == int(g["hidden_size"])
    assert c.n_heads == int(g["num_attention_heads"])
    assert c.n_kv_heads == int(g["num_key_value_heads"])
    assert c.head_dim == int(g["head_dim"])
    assert c.intermediate == int(g["intermediate_size"])
    assert c.eps == float(g["layer_norm_eps"])
    assert c.rotary_span == int(g["rotary_dims"])
    assert c.rope_base == float(g["rope_theta"])
    assert c.qkv_bias == (g["q_proj_bias"] == "True")
    assert c.o_bias == (g["o_proj_bias"] == "True")
    assert c.mlp_bias == (g["mlp_bias"] == "True")
    assert (c.residual == "parallel") == (g["use_parallel_residual"] == "True")
    assert (c.qk_norm != "none") == (g["qk_layernorm"] == "True")
    assert c.act == "swiglu" and g["hidden_act"] == "silu"
    assert c.norm == "layernorm" and c.norm_place == "pre"
    s = weight_shapes(c)
    assert "b_qkv" in s and "b_o" not in s and "b_up" not in s


def test_stablelm2_12b_facts():
    g = _read("stablelm2_12b_shapes.txt")
    c = BLOCK_CONFIGS["stablelm2_12b"]
    assert c.n_heads == int(g["num_attention_heads"]) and c.n_kv_heads == int(g["num_key_value_heads"])
    assert (c.residual == "parallel") == (g["use_parallel_residual"] == "True")
    assert c.qk_norm == "ln_per_head" and g["qk_layernorm"] == "True"
    assert c.qkv_bias == (g["qkv_bias"] == "True")
    s = weight_shapes(c)
    assert s["q_norm_w"][0] == (32, 160) and s["k_norm_w"][0] == (8, 160)
    assert "mlp_norm_w" not in s and "attn_norm_b" in s
    assert ATTN_CONFIGS["attn_12b"].n_kv_heads == 8


def test_olmo2_facts():
    g = _read("olmo2_block.txt")
    c = BLOCK_CONFIGS["olmo2_1b"]
    assert c.norm_place == g["norm_place"] and c.qk_norm == g["qk_norm"]
    s = weight_shapes(c)
    assert "attn_norm_w" not in s and g["input_norm"] == "False"
    assert s["q_norm_w"][0] == (c.n_heads * c.head_dim,)


@pytest.mark.parametrize("name", sorted(BLOCK_CONFIGS))
def test_slots_are_distinct(name):
    s = weight_shapes(BLOCK_CONFIGS[name])
    assert len(set(s)) == len(s)
