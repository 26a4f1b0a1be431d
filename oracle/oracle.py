"""ctypes front-end of the CPU oracle (test infrastructure only).

The functions below marshal CPU tensors / arrays into the C oracle in
``kda_oracle.c`` and return fp64 numpy arrays.  Nothing here does any of the
method's arithmetic; see the C file for what is computed and where the pages
state it.  Only the tests, the smoke check and the benchmark's CPU-baseline
leg import this module.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_F32, _BF16, _F64 = 0, 1, 2


class _Opts(ctypes.Structure):
    _fields_ = [
        ("l2norm_qk", ctypes.c_int),
        ("beta_is_logit", ctypes.c_int),
        ("g_min", ctypes.c_double),
        ("q_scale", ctypes.c_double),
        ("eps_l2", ctypes.c_double),
        ("decay_from_logit", ctypes.c_int),
        ("decay_scale", ctypes.c_void_p),
        ("decay_bias", ctypes.c_void_p),
        ("conv_weight", ctypes.c_void_p),
    ]


def _as_buffer(x):
    """Return (contiguous numpy array, dtype code) without changing any value.

    bf16 tensors are passed as their raw 16-bit patterns.
    """
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach()
        if x.device.type != "cpu":
            x = x.cpu()
        x = x.contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), _BF16
        if x.dtype == torch.float32:
            return x.numpy(), _F32
        if x.dtype == torch.float64:
            return x.numpy(), _F64
        raise TypeError(f"oracle: unsupported tensor dtype {x.dtype}")
    a = np.ascontiguousarray(x)
    if a.dtype == np.float32:
        return a, _F32
    if a.dtype == np.float64:
        return a, _F64
    raise TypeError(f"oracle: unsupported array dtype {a.dtype}")


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """Handle on one build of the oracle library (default: the faithful one)."""

    def __init__(self, path: str | None = None):
        self.path = path or _build.build()
        lib = ctypes.CDLL(self.path)
        vp, ci, cd = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.kda_oracle_prefill.argtypes = [vp, vp, vp, ci, vp, ci, vp, ci, vp, vp,
                                           ci, ci, ci, ci, ci, ci, ci,
                                           ctypes.POINTER(_Opts), vp, vp, vp]
        lib.kda_oracle_prefill.restype = ci
        lib.kda_oracle_decode_step.argtypes = [vp, vp, vp, ci, vp, ci, vp, ci, vp,
                                               ci, ci, ci, ci,
                                               ctypes.POINTER(_Opts), vp, vp]
        lib.kda_oracle_decode_step.restype = ci
        lib.kda_oracle_gated_rmsnorm.argtypes = [vp, ci, ci, ci, vp, ci, ci, ci,
                                                 vp, cd, vp]
        lib.kda_oracle_gated_rmsnorm.restype = ci
        lib.kda_oracle_mutation.restype = ci
        self.lib = lib
        self.mutation = lib.kda_oracle_mutation()

    @staticmethod
    def _opts(l2norm_qk, beta_is_logit, g_min, q_scale, eps_l2, decay_from_logit=False,
              decay_scale=None, decay_bias=None, conv_weight=None):
        """The options struct and the fp64 arrays it points to (keep both alive
        for the call)."""
        keep = [None if a is None else _f64(a) for a in (decay_scale, decay_bias, conv_weight)]
        opts = _Opts(int(bool(l2norm_qk)), int(bool(beta_is_logit)), float(g_min),
                     float(q_scale), float(eps_l2), int(bool(decay_from_logit)),
                     *[None if a is None else a.ctypes.data for a in keep])
        return opts, keep

    def prefill(self, q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, *,
                N: int | None = None, heads: tuple[int, int] | None = None,
                l2norm_qk: bool = True, beta_is_logit: bool = False,
                g_min: float = -5.0, q_scale: float = 1.0, eps_l2: float = 1e-6,
                decay_from_logit: bool = False, decay_scale=None, decay_bias=None,
                conv_weight=None, conv_state=None, want_state: bool = True):
        """Token-by-token prefill.

        Shapes: q, k, log_alpha [T, H, dk]; v [T, H, dv]; beta [T, H];
        S0 [N, H, dk, dv] (or None = zeros); cu_seqlens [N+1] int (or None = N
        equal sequences, N defaults to 1).  ``heads`` = (h0, nh) restricts the
        computation to a head range.  With ``decay_from_logit`` log_alpha holds
        decay logits z and log alpha = g_min * sigmoid(A_h (z + b)), A =
        ``decay_scale`` [H] (None = ones), b = ``decay_bias`` [H, dk] (None =
        zeros).  ``conv_weight`` [3, H, d, 4] turns on the short convolution +
        Swish of q, k, v, with ``conv_state`` [N, 3, 3, H, d] the raw rows
        before each sequence (None = zeros).  Returns (o [T, nh, dv],
        S_T [N, nh, dk, dv]).
        """
        qa, qd = _as_buffer(q)
        ka, kd_ = _as_buffer(k)
        va, vd = _as_buffer(v)
        if not (qd == kd_ == vd):
            raise TypeError("oracle: q, k, v must share one dtype")
        la, lad = _as_buffer(log_alpha)
        ba, bd = _as_buffer(beta)
        T, H, dk = qa.shape
        dv = va.shape[2]
        if cu_seqlens is not None:
            cu = np.ascontiguousarray(np.asarray(
                cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                dtype=np.int32))
            N = cu.shape[0] - 1
            cu_p = _ptr(cu)
        else:
            N = N or 1
            cu, cu_p = None, None
        h0, nh = heads if heads is not None else (0, H)
        s0 = _f64(S0) if S0 is not None else None
        cs = _f64(conv_state) if conv_state is not None else None
        o = np.empty((T, nh, dv), dtype=np.float64)
        st = np.empty((N, nh, dk, dv), dtype=np.float64) if want_state else None
        opts, keep = self._opts(l2norm_qk, beta_is_logit, g_min, q_scale, eps_l2,
                                decay_from_logit, decay_scale, decay_bias, conv_weight)
        rc = self.lib.kda_oracle_prefill(
            _ptr(qa), _ptr(ka), _ptr(va), qd, _ptr(la), lad, _ptr(ba), bd,
            _ptr(s0) if s0 is not None else None, cu_p, N, T, H, dk, dv, h0, nh,
            ctypes.byref(opts), _ptr(o), _ptr(st) if st is not None else None,
            _ptr(cs) if cs is not None else None)
        del keep
        if rc != 0:
            raise ValueError("oracle: kda_oracle_prefill rejected its arguments")
        return o, st

    def decode_step(self, q, k, v, log_alpha, beta, S, *, l2norm_qk=True,
                    beta_is_logit=False, g_min=-5.0, q_scale=1.0, eps_l2=1e-6,
                    decay_from_logit=False, decay_scale=None, decay_bias=None,
                    conv_weight=None, conv_state=None):
        """One recurrent step for N sequences.  S [N, H, dk, dv] is NOT modified;
        returns (o [N, H, dv], S_new [N, H, dk, dv]), and with ``conv_weight``
        (o, S_new, conv_state_new [N, 3, 3, H, d]) (``conv_state`` None = zeros)."""
        qa, qd = _as_buffer(q)
        ka, _ = _as_buffer(k)
        va, _ = _as_buffer(v)
        la, lad = _as_buffer(log_alpha)
        ba, bd = _as_buffer(beta)
        N, H, dk = qa.shape
        dv = va.shape[2]
        s = _f64(S).copy()
        o = np.empty((N, H, dv), dtype=np.float64)
        cs = None
        if conv_weight is not None:
            cs = (_f64(conv_state).copy() if conv_state is not None
                  else np.zeros((N, 3, 3, H, dk), dtype=np.float64))
        opts, keep = self._opts(l2norm_qk, beta_is_logit, g_min, q_scale, eps_l2,
                                decay_from_logit, decay_scale, decay_bias, conv_weight)
        rc = self.lib.kda_oracle_decode_step(
            _ptr(qa), _ptr(ka), _ptr(va), qd, _ptr(la), lad, _ptr(ba), bd,
            _ptr(s), N, H, dk, dv, ctypes.byref(opts), _ptr(o),
            _ptr(cs) if cs is not None else None)
        del keep
        if rc != 0:
            raise ValueError("oracle: kda_oracle_decode_step rejected its arguments")
        if conv_weight is not None:
            return o, s, cs
        return o, s

    def gated_rmsnorm(self, o, gate, w=None, eps: float = 1e-6, h0: int = 0):
        """y = o / sqrt(mean(o^2) + eps) * w * sigmoid(gate), per (row, head).

        o [rows, nh, dv] fp64; gate [rows, H, dv] (heads h0..h0+nh-1 used)."""
        oa = _f64(o)
        rows, nh, dv = oa.shape
        ga, gd = _as_buffer(gate)
        H = ga.shape[1]
        wa = _f64(w) if w is not None else None
        y = np.empty_like(oa)
        rc = self.lib.kda_oracle_gated_rmsnorm(
            _ptr(oa), rows, nh, dv, _ptr(ga), gd, H, h0,
            _ptr(wa) if wa is not None else None, float(eps), _ptr(y))
        if rc != 0:
            raise ValueError("oracle: kda_oracle_gated_rmsnorm rejected its arguments")
        return y


_DEFAULT: Oracle | None = None


def default() -> Oracle:
    """The faithful oracle build (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        _DEFAULT = Oracle()
    return _DEFAULT


def prefill(*a, **kw):
    return default().prefill(*a, **kw)


def decode_step(*a, **kw):
    return default().decode_step(*a, **kw)


def gated_rmsnorm(*a, **kw):
    return default().gated_rmsnorm(*a, **kw)
