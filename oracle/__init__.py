"""fp64 CPU oracle for the prefill forward of one decoder block.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` import this package. The CUDA
path (``alibi_attention_block_gb300``) never imports, links or calls it, and
it never imports the CUDA path.

Every function is the plain definition of one step of the block, written out
in NumPy float64 from storage-rounded inputs, with no intermediate rounding,
no tiling and no fusion. Each cites the passage of the pages it follows.

Parity pins (tests/test_oracle_*.py) hold every function to closed forms,
invariants, library special cases and a loop-only brute force. One reading
is not fixed by the pages: the sign of ``rotate_half`` (the pages name the
operation but do not define it). Relative-position invariance holds for
either sign; the standard ``[-x2, x1]`` is taken. That sign is parity
unpinned by the pages.
"""
from .block import (  # noqa: F401
    as_f64, layer_norm, rms_norm, linear, split_qkv, split_heads, merge_heads,
    qk_norm_full_rms, qk_norm_per_head_ln, rope_inv_freq, rope, alibi_slopes,
    attention, attention_decode, silu, gelu_tanh, mlp, block_forward, attention_forward,
)
from .model import model_forward  # noqa: F401
from .quant import q8_0_quantize, q8_0_dequantize, linear_q8_0  # noqa: F401
from .decode_step import block_decode_step  # noqa: F401
