"""Parity helpers: GPU result vs fp64 oracle.

Gate (per output tensor):
  - per-row cosine >= 0.9999 (rows = the last axis);
  - max |gpu - ref| <= 2e-2 * scale, scale = 1 for block outputs (unit
    scale: the residual stream carries x ~ N(0, 1)) and rms(ref) for
    sub-block outputs of other scales.
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


def check(gpu, ref, name="", unit_scale=False, cos_min=COS_MIN, abs_tol=ABS_TOL):
    g = f64(gpu)
    r = f64(ref)
    assert g.shape == r.shape, (name, g.shape, r.shape)
    assert np.isfinite(g).all(), f"{name}: non-finite GPU output"
    scale = 1.0 if unit_scale else float(np.sqrt((r * r).mean()))
    err = float(np.abs(g - r).max()) if g.size else 0.0
    cos = float(row_cosine(g, r).min()) if g.size else 1.0
    assert err <= abs_tol * scale, f"{name}: max abs err {err:.3e} > {abs_tol}*{scale:.3e} (min cos {cos:.6f})"
    assert cos >= cos_min, f"{name}: min per-row cosine {cos:.6f} < {cos_min} (max err {err:.3e})"
    return err, cos
