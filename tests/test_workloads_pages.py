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


def test_stablelm2_1p6b_model_facts_match_the_model_bench_and_oracle():
    """bench.py --model and the model wrap use the printed model shape: 24
    layers, a 100352-token vocabulary, an untied bias-free lm_head and a
    final LayerNorm with bias."""
    import inspect

    import bench
    import workloads
    g = _read("stablelm2_1p6b_model.txt")
    src = inspect.getsource(bench.run_model)
    assert f"n_layers, vocab = {int(g['num_hidden_layers'])}, {int(g['vocab_size'])}" in src
    c = BLOCK_CONFIGS["stablelm2_1p6b"]
    assert c.hidden == int(g["embed_dim"]) and c.eps == float(g["final_norm_eps"])
    assert g["tie_word_embeddings"] == "False" and g["lm_head_bias"] == "False"
    # the model inputs draw separate embedding and lm_head tables, a final
    # LayerNorm with a bias, and no lm_head bias slot
    _, mw = workloads.model_inputs(workloads.BLOCK_CONFIGS["tiny_stablelm2"], 1, 64)
    assert mw["embed"].data_ptr() != mw["lm_head"].data_ptr()
    assert ("final_norm_b" in mw) == (g["final_norm_bias"] == "True")
    assert not any(k.startswith("lm_head_b") for k in mw)


def test_bloom_facts():
    """The Bloom workload follows its page: ALiBi without rotary, the fused
    QKV in per-head interleaved order, f16, and the embedding LayerNorm in
    the model wrap's inputs."""
    import workloads
    g = _read("bloom_block.txt")
    c = BLOCK_CONFIGS["bloom_560m"]
    assert c.alibi == (g["alibi"] == "True")
    assert (c.rotary_span > 0) == (g["rotary"] == "True")
    assert (c.qkv_layout == "head_interleaved") == (g["fused_qkv_deinterleave"] == "True")
    assert c.dtype == "fp16" and g["precision"] == "f16"
    _, mw = workloads.model_inputs(c, 0, 64, embed_norm=g["embedding_layernorm"] == "True")
    assert "embed_norm_w" in mw and "embed_norm_b" in mw

