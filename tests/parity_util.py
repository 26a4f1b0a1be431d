"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances are the ones the method's accuracy target states: for bf16
operands max-abs <= 2e-2 AND rel-L2 <= 5e-3 (rel-L2 = |x - ref|_2 / |ref|_2 over
the whole tensor, with the worst head's rel-L2 reported on a failure); for
the fp32 path both <= 1e-4.
"""
from __future__ import annotations

import numpy as np

TOL_BF16 = dict(max_abs=2e-2, rel_l2=5e-3)
TOL_F32 = dict(max_abs=1e-4, rel_l2=1e-4)


def to_np(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().float().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def errors(x, ref):
    x, ref = to_np(x), to_np(ref)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    assert np.all(np.isfinite(x)), "non-finite values in the GPU result"
    d = x - ref
    max_abs = float(np.max(np.abs(d))) if d.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(d) / den) if den > 0 else float(np.linalg.norm(d))
    return max_abs, rel


def per_head_rel(x, ref, axis=1):
    """rel-L2 of each head (axis 1 of [T, H, d] outputs and [N, H, d, d] states)."""
    x, ref = to_np(x), to_np(ref)
    if x.ndim < 3:
        return np.array([errors(x, ref)[1]])
    xs, rs = np.moveaxis(x, axis, 0), np.moveaxis(ref, axis, 0)
    out = []
    for a, b in zip(xs, rs):
        den = float(np.linalg.norm(b))
        out.append(float(np.linalg.norm(a - b) / den) if den > 0 else float(np.linalg.norm(a - b)))
    return np.array(out)


def assert_close(x, ref, tol, what=""):
    max_abs, rel = errors(x, ref)
    if not (max_abs <= tol["max_abs"] and rel <= tol["rel_l2"]):
        ph = per_head_rel(x, ref)
        raise AssertionError(
            f"{what}: max_abs={max_abs:.3e} (tol {tol['max_abs']:.0e}), "
            f"rel_l2={rel:.3e} (tol {tol['rel_l2']:.0e}); per head rel_l2 max "
            f"{ph.max():.3e} at head {int(ph.argmax())}")
    return max_abs, rel
