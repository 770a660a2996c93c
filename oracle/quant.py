"""fp64 oracle of the q8 weight path (test infrastructure, like the rest of
``oracle``; the CUDA path never imports it).

The pages report q8/int8 weights only as a secondary precision ("StableLM-2
...", Results: q8 cosine 0.998910; "OLMo-2 ...", section 4: int8 cosine
0.998700) and never define the format; the one format they name is Q8_0
("RoFormer HIP FP32 layout optimization": BS-RoFormer ep368 Q8_0). Reading:
Q8_0 as published with GGML — each row of W[out, in] in blocks of 32
consecutive input elements; per block one scale d = absmax / 127 rounded to
fp16, and q = round(w / d) as int8 (round half away from zero; d = 0 gives
q = 0); the weight used is d * q. Parity of this function is pinned by
closed forms (the error bound, exact round trips) and not by any value the
pages print.
"""
from __future__ import annotations

import numpy as np

from .block import as_f64

BLOCK = 32


def q8_0_quantize(w):
    """(q int8 [out, in], d float16 [out, in / 32]) of a weight W[out, in]
    (in a multiple of 32)."""
    w = as_f64(w)
    out_f, in_f = w.shape
    if in_f % BLOCK:
        raise ValueError("the input width must be a multiple of 32")
    blocks = w.reshape(out_f, in_f // BLOCK, BLOCK)
    amax = np.abs(blocks).max(axis=-1)
    d = (amax / 127.0).astype(np.float16)
    df = d.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(df[..., None] > 0, blocks / df[..., None], 0.0)
    q = np.sign(r) * np.floor(np.abs(r) + 0.5)      # half away from zero
    q = np.clip(q, -127, 127).astype(np.int8)
    return q.reshape(out_f, in_f), d


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
