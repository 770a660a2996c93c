"""fp64 oracle of the q8 weight path (test infrastructure, like the rest of
``oracle``; the CUDA path never imports it).

The pages report q8/int8 weights only as a secondary precision ("StableLM-2
...", Results: q8 cosine 0.998910; "OLMo-2 ...", section 4: int8 cosine
0.998700) and never define the format; the one format they name is Q8_0
("RoFormer HIP FP32 layout optimization": BS-RoFormer ep368 Q8_0). Reading:
Q8_0 as published with GGML. Each row of W[out, in] is cut into blocks of 32
consecutive input elements. Per block, in float32 arithmetic (GGML quantizes
float32 weights): the scale d = absmax / 127, its reciprocal 1 / d (0 when
d = 0), and the codes q = round(w * (1 / d)) as int8, rounded half away from
zero. Only then is d stored, rounded to fp16; the weight the linear uses is
that stored fp16 d times q. The codes therefore come from the float32 scale,
not from the stored fp16 one. The integer decision is taken in float32 on
both sides (oracle and kernel), so codes compare bit for bit. The linear
itself is float64. Parity of these functions is pinned by closed forms (the
error bound, exact round trips, exact rational arithmetic away from
half-steps) and not by any value the pages print.
"""
from __future__ import annotations

import numpy as np

from .block import as_f64

BLOCK = 32


def q8_0_quantize(w):
    """(q int8 [out, in], d float16 [out, in / 32]) of a weight W[out, in]
    (in a multiple of 32). The weight is taken as float32, as GGML takes it."""
    w32 = np.asarray(as_f64(w), dtype=np.float32)
    out_f, in_f = w32.shape
    if in_f % BLOCK:
        raise ValueError("the input width must be a multiple of 32")
    blocks = w32.reshape(out_f, in_f // BLOCK, BLOCK)
    amax = np.abs(blocks).max(axis=-1)                       # float32
    d32 = amax / np.float32(127.0)                           # float32 division
    with np.errstate(divide="ignore"):
        inv = np.where(d32 > 0, np.float32(1.0) / d32, np.float32(0.0)).astype(np.float32)
    r = (blocks * inv[..., None]).astype(np.float64)         # float32 product, exact in f64
    q = np.sign(r) * np.floor(np.abs(r) + 0.5)               # half away from zero
    if np.abs(q).max(initial=0) > 127:
        raise AssertionError("a Q8_0 code left [-127, 127]")
    return q.astype(np.int8).reshape(out_f, in_f), d32.astype(np.float16)


def q8_0_dequantize(q, d):
    """W ≈ d * q, block by block, in float64."""
    q = np.asarray(q, dtype=np.float64)
    out_f, in_f = q.shape
    df = np.asarray(d, dtype=np.float64)
    return (q.reshape(out_f, in_f // BLOCK, BLOCK) * df[..., None]).reshape(out_f, in_f)


def linear_q8_0(x, q, d, b=None):
    """x W^T (+ b) with the Q8_0 weight: the plain linear on d * q."""
    y = as_f64(x) @ q8_0_dequantize(q, d).T
    return y if b is None else y + as_f64(b)
