"""Thin ctypes binding of libkda.so (the C ABI in ``include/kda.h``).

The functions carry the C entry points' names and do argument marshalling
only: shapes are read off the tensors, outputs and the workspace are
allocated with PyTorch when the caller does not pass them, and the call goes
to the library on the current CUDA stream.  Every step of the computation runs
in the library's CUDA kernels; there is no Python or CPU fallback, and a
missing or unloadable library raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

KDA_OK = 0
KDA_ERR_ARG = -1
KDA_ERR_SHAPE = -2
KDA_ERR_DTYPE = -3
KDA_ERR_ALIGN = -4
KDA_ERR_UNSUPPORTED = -5
KDA_ERR_CUDA = -6
KDA_ERR_TIMEOUT = -7
KDA_ERR_WORKSPACE = -8

KDA_F32 = 0
KDA_BF16 = 1

IMPLS = {"auto": 0, "simt": 1, "tc": 2}
# KDA_DECAY_*: log_alpha [T, H, d_k] per key channel (KDA), [T, H] per head
# (Gated DeltaNet), or none (DeltaNet, log_alpha may be None)
DECAY_MODES = {"channel": 0, "head": 1, "none": 2}


class kda_options(ctypes.Structure):
    """Mirror of ``struct kda_options`` (field order and types as in kda.h)."""
    _fields_ = [
        ("chunk", ctypes.c_int),
        ("l2norm_qk", ctypes.c_int),
        ("beta_is_logit", ctypes.c_int),
        ("g_min", ctypes.c_float),
        ("q_scale", ctypes.c_float),
        ("eps_l2", ctypes.c_float),
        ("eps_norm", ctypes.c_float),
        ("gate", ctypes.c_void_p),
        ("norm_weight", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("max_seqlen", ctypes.c_int),
        ("impl", ctypes.c_int),
        ("debug_timeout", ctypes.c_int),
        ("timeout_spins", ctypes.c_longlong),
        ("phase_events", ctypes.c_void_p),
        ("decay_mode", ctypes.c_int),
        ("snapshot_every", ctypes.c_int),
        ("snapshots", ctypes.c_void_p),
        ("decay_from_logit", ctypes.c_int),
        ("decay_scale", ctypes.c_void_p),
        ("decay_bias", ctypes.c_void_p),
        ("conv_weight", ctypes.c_void_p),
        ("conv_state", ctypes.c_void_p),
    ]


class KdaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kda_status_string(status)} ({status})")


_LIB = None
EXPORTS = ("kda_options_init", "kda_prefill", "kda_prefill_noalloc",
           "kda_prefill_workspace_size", "kda_prefill_path",
           "kda_decode_step", "kda_gated_rmsnorm", "kda_get_last_error", "kda_status_string",
           "kda_abi_version")
PATH_NAMES = {1: "simt", 2: "tc"}


def lib_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libkda.so (building it first if it is missing or stale)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    if path is None:
        path = _build.build()
    lib = ctypes.CDLL(path)
    vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    po = ctypes.POINTER(kda_options)
    lib.kda_options_init.argtypes = [po]
    lib.kda_options_init.restype = None
    lib.kda_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, vp, vp, ci, ci, ci, ci, ci, po, vp]
    lib.kda_prefill.restype = ci
    lib.kda_prefill_workspace_size.argtypes = [ci, ci, ci, ci, ci, po]
    lib.kda_prefill_workspace_size.restype = ctypes.c_size_t
    pi = ctypes.POINTER(ctypes.c_int)
    lib.kda_prefill_path.argtypes = [ci, ci, ci, ci, ci, ci, po, pi, pi]
    lib.kda_prefill_path.restype = ci
    lib.kda_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, po, vp]
    lib.kda_decode_step.restype = ci
    lib.kda_gated_rmsnorm.argtypes = [vp, vp, vp, vp, ci, ci, ci, cf, ci, vp]
    lib.kda_gated_rmsnorm.restype = ci
    lib.kda_get_last_error.argtypes = [vp]
    lib.kda_get_last_error.restype = ci
    lib.kda_status_string.argtypes = [ci]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_abi_version.restype = ci
    lib.kda_prefill_noalloc.argtypes = lib.kda_prefill.argtypes
    lib.kda_prefill_noalloc.restype = ci
    if path == _build.LIB or _LIB is None:
        _LIB = lib
    return lib


def kda_status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def kda_abi_version() -> int:
    return load().kda_abi_version()


def kda_options_init(**overrides) -> kda_options:
    """Default options (C kda_options_init), then keyword overrides."""
    opt = kda_options()
    load().kda_options_init(ctypes.byref(opt))
    for key, val in overrides.items():
        if key == "impl" and isinstance(val, str):
            val = IMPLS[val]
        if key == "decay_mode" and isinstance(val, str):
            val = DECAY_MODES[val]
        setattr(opt, key, val)
    return opt


# ---------------------------------------------------------------- marshalling
def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use bfloat16 or float32")


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libkda takes CUDA tensors (device memory)")
        if not t.is_contiguous():
            raise ValueError("libkda takes contiguous tensors")


def _opts(gate, norm_weight, chunk, l2norm_qk, beta_is_logit, g_min, q_scale, eps_l2,
          eps_norm, workspace, workspace_bytes, max_seqlen, impl, debug_timeout,
          timeout_spins, decay_mode="channel", decay_from_logit=False, decay_scale=None,
          decay_bias=None, conv_weight=None, conv_state=None) -> kda_options:
    _check_cuda(decay_scale, decay_bias, conv_weight, conv_state)
    return kda_options_init(
        decay_mode=decay_mode,
        chunk=int(chunk), l2norm_qk=int(bool(l2norm_qk)), beta_is_logit=int(bool(beta_is_logit)),
        g_min=float(g_min), q_scale=float(q_scale), eps_l2=float(eps_l2),
        eps_norm=float(eps_norm), gate=_ptr(gate), norm_weight=_ptr(norm_weight),
        workspace=_ptr(workspace), workspace_bytes=int(workspace_bytes),
        max_seqlen=int(max_seqlen), impl=impl, debug_timeout=int(bool(debug_timeout)),
        timeout_spins=int(timeout_spins), decay_from_logit=int(bool(decay_from_logit)),
        decay_scale=_ptr(decay_scale), decay_bias=_ptr(decay_bias),
        conv_weight=_ptr(conv_weight), conv_state=_ptr(conv_state))


def kda_prefill_workspace_size(T_total: int, N: int, H: int, d_k: int, d_v: int,
                               opt: kda_options | None = None) -> int:
    o = opt if opt is not None else kda_options_init()
    return int(load().kda_prefill_workspace_size(T_total, N, H, d_k, d_v, ctypes.byref(o)))


def kda_prefill_path(T_total: int, N: int, H: int, d_k: int, d_v: int, dtype: int = KDA_BF16,
                     opt: kda_options | None = None) -> tuple[str, int, int]:
    """(path name, kernels per call, chunk) that kda_prefill uses for these sizes."""
    o = opt if opt is not None else kda_options_init()
    launches, chunk = ctypes.c_int(0), ctypes.c_int(0)
    rc = load().kda_prefill_path(T_total, N, H, d_k, d_v, dtype, ctypes.byref(o),
                                 ctypes.byref(launches), ctypes.byref(chunk))
    if rc < 0:
        raise KdaError(rc, "kda_prefill_path")
    return PATH_NAMES[rc], launches.value, chunk.value


def kda_prefill(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, N: int | None = None,
                o=None, S_T=None, *, gate=None, norm_weight=None, chunk: int = 0,
                l2norm_qk: bool = True, beta_is_logit: bool = False, g_min: float = -5.0,
                q_scale: float = 1.0, eps_l2: float = 1e-6, eps_norm: float = 1e-6,
                workspace=None, max_seqlen: int = 0, impl="auto", debug_timeout: bool = False,
                timeout_spins: int = 0, phase_events=None, decay_mode="channel",
                snapshot_every: int = 0, snapshots=None, decay_from_logit: bool = False,
                decay_scale=None, decay_bias=None, conv_weight=None, conv_state=None,
                stream=None):
    """Chunked prefill (C ``kda_prefill``).

    q, k, log_alpha [T, H, d_k]; v [T, H, d_v]; beta [T, H]; S0 [N, H, d_k, d_v]
    fp32 or None; cu_seqlens [N+1] int32 (device) or None.  Returns (o, S_T);
    o holds y = RMSNorm(o) * w * sigmoid(gate) when ``gate`` is given.
    ``decay_mode`` "head" takes log_alpha [T, H]; "none" ignores it (None is fine).
    With ``snapshot_every`` (a multiple of 64) it returns (o, S_T, snapshots),
    snapshots [N, L // snapshot_every, H, d_k, d_v] fp32 with L = max_seqlen
    (T // N without cu_seqlens, T with them): slot m holds the state after
    (m + 1) * snapshot_every tokens of the sequence (zeros, or the given
    buffer's contents, past its length).
    The prologue from raw projections: ``decay_from_logit`` takes log_alpha as
    decay logits z and forms g_min * sigmoid(A_h (z + b)) with ``decay_scale``
    A [H] and ``decay_bias`` b [H, d_k] (fp32, None = ones / zeros);
    ``conv_weight`` [3, H, d, 4] fp32 runs q, k, v through the width-4 causal
    short convolution + Swish first, ``conv_state`` [N, 3, 3, H, d] (dtype of
    q) holding the raw rows before each sequence (None = zeros).
    """
    import torch
    _check_cuda(q, k, v, log_alpha, beta, S0, cu_seqlens, gate, norm_weight, o, S_T)
    T, H, d_k = q.shape
    d_v = v.shape[2]
    if cu_seqlens is not None:
        N = cu_seqlens.numel() - 1
    N = N or 1
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty((T, H, d_v), dtype=q.dtype, device=q.device)
    if S_T is None:
        S_T = torch.empty((N, H, d_k, d_v), dtype=torch.float32, device=q.device)
    impl_code = IMPLS[impl] if isinstance(impl, str) else int(impl)
    opt = _opts(gate, norm_weight, chunk, l2norm_qk, beta_is_logit, g_min, q_scale, eps_l2,
                eps_norm, None, 0, max_seqlen, impl_code, debug_timeout, timeout_spins,
                decay_mode, decay_from_logit, decay_scale, decay_bias, conv_weight, conv_state)
    if phase_events is not None:  # list of torch.cuda.Event, (launches + 1) of them
        if any(not e.cuda_event for e in phase_events):
            raise ValueError("phase_events: record each event once first (torch creates "
                             "the CUDA event lazily)")
        ev_arr = (ctypes.c_void_p * len(phase_events))(*[e.cuda_event for e in phase_events])
        opt.phase_events = ctypes.cast(ev_arr, ctypes.c_void_p)
    if snapshot_every:
        L = max_seqlen if max_seqlen > 0 else (T if cu_seqlens is not None else T // N)
        if snapshots is None:
            snapshots = torch.zeros((N, L // snapshot_every, H, d_k, d_v), dtype=torch.float32,
                                    device=q.device)
        _check_cuda(snapshots)
        opt.snapshot_every = int(snapshot_every)
        opt.snapshots = _ptr(snapshots)
    need = kda_prefill_workspace_size(T, N, H, d_k, d_v, opt)
    if need > 0:
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        opt.workspace = _ptr(workspace)
        opt.workspace_bytes = workspace.numel() * workspace.element_size()
    rc = load().kda_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
                            _ptr(cu_seqlens), N, _ptr(o), _ptr(S_T), T, H, d_k, d_v, dt,
                            ctypes.byref(opt), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill")
    if snapshot_every:
        return o, S_T, snapshots
    return o, S_T


_DECODE_OPTS: dict = {}


def kda_decode_step(q, k, v, log_alpha, beta, S, o=None, *, gate=None, norm_weight=None,
                    l2norm_qk: bool = True, beta_is_logit: bool = False, g_min: float = -5.0,
                    q_scale: float = 1.0, eps_l2: float = 1e-6, eps_norm: float = 1e-6,
                    decay_mode="channel", decay_from_logit: bool = False, decay_scale=None,
                    decay_bias=None, conv_weight=None, conv_state=None, stream=None):
    """One decode step (C ``kda_decode_step``); S [N, H, d_k, d_v] is updated in place.
    Returns o [N, H, d_v].  log_alpha is [N, H] with decay_mode "head".  With
    ``conv_weight``, ``conv_state`` [N, 3, 3, H, d] (the raw q, k, v rows of the
    3 previous tokens) is read and moved on by this token in place."""
    import torch
    _check_cuda(q, k, v, log_alpha, beta, S, o, gate, norm_weight)
    N, H, d_k = q.shape
    d_v = v.shape[2]
    if o is None:
        o = torch.empty((N, H, d_v), dtype=q.dtype, device=q.device)
    # a decode loop calls this once per token: the options struct is built once
    # per distinct setting
    key = (_ptr(gate), _ptr(norm_weight), bool(l2norm_qk), bool(beta_is_logit), float(g_min),
           float(q_scale), float(eps_l2), float(eps_norm), decay_mode, bool(decay_from_logit),
           _ptr(decay_scale), _ptr(decay_bias), _ptr(conv_weight), _ptr(conv_state))
    opt = _DECODE_OPTS.get(key)
    if opt is None:
        opt = _opts(gate, norm_weight, 0, l2norm_qk, beta_is_logit, g_min, q_scale, eps_l2,
                    eps_norm, None, 0, 0, 0, False, 0, decay_mode, decay_from_logit,
                    decay_scale, decay_bias, conv_weight, conv_state)
        if len(_DECODE_OPTS) > 64:
            _DECODE_OPTS.clear()
        _DECODE_OPTS[key] = opt
    rc = load().kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                _ptr(S), _ptr(o), N, H, d_k, d_v, _dtype_code(q),
                                ctypes.byref(opt), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step")
    return o


def kda_gated_rmsnorm(o, gate, w=None, y=None, *, eps: float = 1e-6, stream=None):
    """y = o / sqrt(mean(o^2) + eps) * w * sigmoid(gate) per (row, head)
    (C ``kda_gated_rmsnorm``); o, gate [rows, H, d_v]."""
    import torch
    _check_cuda(o, gate, w, y)
    rows, H, d_v = o.shape
    if y is None:
        y = torch.empty_like(o)
    rc = load().kda_gated_rmsnorm(_ptr(o), _ptr(gate), _ptr(w), _ptr(y), rows, H, d_v,
                                  float(eps), _dtype_code(o), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_gated_rmsnorm")
    return y


def kda_get_last_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(load().kda_get_last_error(_stream(stream)))


NOALLOC_SCRATCH_BYTES = 64 << 20


def kda_prefill_noalloc(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None, N: int | None = None,
                        o=None, S_T=None, *, gate=None, norm_weight=None, l2norm_qk: bool = True,
                        beta_is_logit: bool = False, g_min: float = -5.0, q_scale: float = 1.0,
                        eps_l2: float = 1e-6, eps_norm: float = 1e-6, max_seqlen: int = 0,
                        decay_mode="channel", stream=None):
    """Prefill with the library's built-in scratch (C ``kda_prefill_noalloc``).

    For callers that must not allocate device memory: the library allocates
    nothing for this call (pass ``o`` and ``S_T`` to allocate nothing here
    either).  Same arguments and results as :func:`kda_prefill`; sizes whose
    scratch exceeds 64 MiB raise KdaError(KDA_ERR_WORKSPACE)."""
    import torch
    _check_cuda(q, k, v, log_alpha, beta, S0, cu_seqlens, gate, norm_weight, o, S_T)
    T, H, d_k = q.shape
    d_v = v.shape[2]
    if cu_seqlens is not None:
        N = cu_seqlens.numel() - 1
    N = N or 1
    if o is None:
        o = torch.empty((T, H, d_v), dtype=q.dtype, device=q.device)
    if S_T is None:
        S_T = torch.empty((N, H, d_k, d_v), dtype=torch.float32, device=q.device)
    opt = _opts(gate, norm_weight, 64, l2norm_qk, beta_is_logit, g_min, q_scale, eps_l2,
                eps_norm, None, 0, max_seqlen, IMPLS["tc"], False, 0, decay_mode)
    rc = load().kda_prefill_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                    _ptr(S0), _ptr(cu_seqlens), N, _ptr(o), _ptr(S_T), T, H, d_k,
                                    d_v, _dtype_code(q), ctypes.byref(opt), _stream(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_prefill_noalloc")
    return o, S_T
