"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances are the ones the method's accuracy target states: for bf16
operands max-abs <= 2e-2 AND rel-L2 <= 5e-3 (rel-L2 = |x - ref|_2 / |ref|_2 over
the whole tensor, with the worst head's rel-L2 reported on a failure); for
the fp32 path both <= 1e-4.

A result stored in bf16 carries its own rounding, half a unit in the last
place: at most 1/64 below magnitude 8, which the 2e-2 bound covers, but 1/32
for magnitudes in [8, 16), more than the bound by itself.  So for bf16 results
an element of magnitude >= 8 is allowed the part of its rounding beyond 1/64
on top of 2e-2: the same margin for the arithmetic as an element just below 8.
Below magnitude 8 (and for every fp32 result) the bound is 2e-2 exactly.
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


def _is_bf16(x) -> bool:
    try:
        import torch
        return isinstance(x, torch.Tensor) and x.dtype == torch.bfloat16
    except ImportError:  # pragma: no cover
        return False


def bf16_excess_rounding(ref):
    """Half a bf16 unit in the last place at |ref| (8 significant bits) beyond
    the 1/64 it reaches just below magnitude 8; zero below 8."""
    _, e = np.frexp(np.abs(ref))
    half_ulp = np.ldexp(1.0, e - 9)
    return np.maximum(half_ulp - 2.0 ** -6, 0.0)


def errors(x, ref):
    """(max-abs error, rel-L2 error).  For a bf16 result the max-abs error of an
    element of magnitude >= 8 is counted net of its rounding beyond 1/64 (see
    the module docstring)."""
    bf16 = _is_bf16(x)
    x, ref = to_np(x), to_np(ref)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    assert np.all(np.isfinite(x)), "non-finite values in the GPU result"
    d = x - ref
    ad = np.abs(d)
    if bf16 and d.size:
        ad = np.maximum(ad - bf16_excess_rounding(ref), 0.0)
    max_abs = float(np.max(ad)) if d.size else 0.0
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
        xa, ra = to_np(x), to_np(ref)
        d = np.abs(xa - ra)
        if _is_bf16(x):
            d = np.maximum(d - bf16_excess_rounding(ra), 0.0)
        at = np.unravel_index(int(np.argmax(d)), d.shape)
        n_over = int((d > tol["max_abs"]).sum())
        raise AssertionError(
            f"{what}: max_abs={max_abs:.3e} (tol {tol['max_abs']:.0e}), "
            f"rel_l2={rel:.3e} (tol {tol['rel_l2']:.0e}); per head rel_l2 max "
            f"{ph.max():.3e} at head {int(ph.argmax())}; worst at {tuple(int(i) for i in at)}: "
            f"got {xa[at]:.6g}, oracle {ra[at]:.6g}; {n_over} of {d.size} elements over "
            f"max_abs; largest |oracle| {np.abs(ra).max():.4g}")
    return max_abs, rel
