"""Parity helpers: GPU result vs fp64 oracle.

Gate (per output tensor):
  - per-row cosine >= 0.9999 (rows = the last axis);
  - max |gpu - ref| <= 2e-2 * scale, scale = max(1, rms(ref)) for outputs of
    unit scale or larger (block outputs: the residual stream carries
    x ~ N(0, 1), and the blocks add sublayer outputs of rms up to ~3 to it)
    and rms(ref) for sub-block outputs of other scales;
  - for an output stored in a 16-bit type (``storage``), each element may in
    addition be off by half an ulp of that type at the reference value: the
    rounding of the stored output itself, which no kernel can avoid (bf16:
    2^-9 |ref|, i.e. above 2e-2 wherever |ref| > 10.24).
"""
import numpy as np
import torch

COS_MIN = 0.9999
ABS_TOL = 2e-2


def to_dev(t, device="cuda"):
    return t.to(device).contiguous() if t is not None else None


def f64(t):
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def row_cosine(a, b):
    a = a.reshape(-1, a.shape[-1])
    b = b.reshape(-1, b.shape[-1])
    na = np.linalg.norm(a, axis=-1)
    nb = np.linalg.norm(b, axis=-1)
    both_zero = (na == 0) & (nb == 0)
    cos = (a * b).sum(-1) / np.maximum(na * nb, 1e-300)
    return np.where(both_zero, 1.0, cos)


_SIGNIFICANT_BITS = {"bf16": 8, "fp16": 11}


def half_ulp(ref, storage):
    """Half an ulp of the 16-bit storage type at |ref| (normal range)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 1e-30)))
    return np.where(a > 0, np.exp2(e - _SIGNIFICANT_BITS[storage]), 0.0)


def check(gpu, ref, name="", unit_scale=False, cos_min=COS_MIN, abs_tol=ABS_TOL, storage=None):
    g = f64(gpu)
    r = f64(ref)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{name}: non-finite GPU output"
    rms = float(np.sqrt((r * r).mean())) if r.size else 0.0
    scale = max(1.0, rms) if unit_scale else rms
    diff = np.abs(g - r)
    err = float(diff.max()) if g.size else 0.0
    cos = float(row_cosine(g, r).min()) if g.size else 1.0
    if storage is not None:
        # the part of each element's error beyond its own output rounding
        excess = float((diff - half_ulp(r, storage)).max()) if g.size else 0.0
        assert excess <= abs_tol * scale, (
            f"{name}: max abs err beyond half an {storage} ulp {excess:.3e} > {abs_tol}*{scale:.3e} "
            f"(max abs err {err:.3e}, min cos {cos:.6f})")
        assert cos >= cos_min, f"{name}: min per-row cosine {cos:.6f} < {cos_min} (max err {err:.3e})"
        return err, cos
    assert err <= abs_tol * scale, f"{name}: max abs err {err:.3e} > {abs_tol}*{scale:.3e} (min cos {cos:.6f})"
    assert cos >= cos_min, f"{name}: min per-row cosine {cos:.6f} < {cos_min} (max err {err:.3e})"
    return err, cos
