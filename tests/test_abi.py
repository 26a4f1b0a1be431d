"""The C-ABI library: it loads, exports every entry point the header declares,
and rejects bad arguments on the host with the documented status codes.

These run without a GPU.  Every call below fails a host-side check before
anything could be launched (the fake device addresses are never touched).
"""
import ctypes
import os
import re

import pytest

from linear_attention_recurrence_prefill_gb300 import kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(kda_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(kda.lib_path() if os.path.exists(kda.lib_path()) else kda.load()._name)
    declared = _declared()
    assert {"kda_prefill", "kda_decode_step", "kda_gated_rmsnorm",
            "kda_prefill_workspace_size", "kda_get_last_error"} <= declared
    missing = [n for n in sorted(declared) if not hasattr(lib, n)]
    assert not missing, f"declared in include/ but not exported: {missing}"


def test_options_defaults():
    o = kda.kda_options_init()
    assert (o.chunk, o.l2norm_qk, o.beta_is_logit, o.impl) == (0, 1, 0, 0)
    assert o.g_min == -5.0 and o.q_scale == 1.0
    assert abs(o.eps_l2 - 1e-6) < 1e-12 and abs(o.eps_norm - 1e-6) < 1e-12
    assert not o.gate and not o.workspace and o.workspace_bytes == 0
    assert o.decay_mode == kda.DECAY_MODES["channel"] == 0
    assert o.snapshot_every == 0 and not o.snapshots
    assert o.decay_from_logit == 0 and not o.decay_scale and not o.decay_bias
    assert not o.conv_weight and not o.conv_state
    # layout of struct kda_options on LP64 (7 x 4-byte fields, 3 pointers,
    # size_t, 3 ints, padding, long long, pointer, 2 ints, pointer, int,
    # padding, 4 pointers)
    assert ctypes.sizeof(kda.kda_options) == 152
    assert kda.kda_abi_version() == 3


def test_status_strings():
    for code in range(-8, 1):
        assert kda.kda_status_string(code) != "unknown status"
    assert kda.kda_status_string(5) == "unknown status"


A = 0x10000  # a 16-byte aligned stand-in address; never dereferenced here

# The rejection tests hand the library fake addresses: they only ever run on
# a machine without a GPU, where nothing could be launched even by mistake.
no_gpu = pytest.mark.skipif(
    __import__("torch").cuda.is_available(),
    reason="host-side rejection checks use fake addresses; run them without a GPU")


def _prefill(**kw):
    lib = kda.load()
    args = dict(q=A, k=A, v=A, la=A, beta=A, S0=None, cu=None, N=1, o=A, S_T=A, T=64, H=2,
                dk=64, dv=64, dtype=kda.KDA_BF16, opt=None)
    args.update(kw)
    opt = args["opt"] if args["opt"] is not None else kda.kda_options_init()
    return lib.kda_prefill(args["q"], args["k"], args["v"], args["la"], args["beta"], args["S0"],
                           args["cu"], args["N"], args["o"], args["S_T"], args["T"], args["H"],
                           args["dk"], args["dv"], args["dtype"], ctypes.byref(opt), None)


@no_gpu
@pytest.mark.parametrize("kw,code", [
    (dict(q=None), kda.KDA_ERR_ARG),
    (dict(o=None), kda.KDA_ERR_ARG),
    (dict(S_T=None), kda.KDA_ERR_ARG),
    (dict(N=0), kda.KDA_ERR_SHAPE),
    (dict(H=0), kda.KDA_ERR_SHAPE),
    (dict(T=-1), kda.KDA_ERR_SHAPE),
    (dict(T=65, N=2), kda.KDA_ERR_SHAPE),
    (dict(dtype=7), kda.KDA_ERR_DTYPE),
    (dict(dk=48, dv=48), kda.KDA_ERR_UNSUPPORTED),
    (dict(dk=64, dv=128), kda.KDA_ERR_UNSUPPORTED),
    (dict(q=A + 8), kda.KDA_ERR_ALIGN),
    (dict(S0=A + 4), kda.KDA_ERR_ALIGN),
    (dict(cu=A + 2, N=1), kda.KDA_ERR_ALIGN),
])
def test_prefill_rejects(kw, code):
    assert _prefill(**kw) == code


@no_gpu
@pytest.mark.parametrize("opt_kw,code", [
    (dict(g_min=-6.0), kda.KDA_ERR_ARG),
    (dict(g_min=0.5), kda.KDA_ERR_ARG),
    (dict(chunk=32), kda.KDA_ERR_ARG),
    (dict(l2norm_qk=2), kda.KDA_ERR_ARG),
    (dict(eps_l2=-1.0), kda.KDA_ERR_ARG),
    (dict(max_seqlen=1000), kda.KDA_ERR_SHAPE),
    (dict(impl=9), kda.KDA_ERR_UNSUPPORTED),
    (dict(gate=A + 2), kda.KDA_ERR_ALIGN),
    (dict(decay_mode=3), kda.KDA_ERR_ARG),
    (dict(decay_mode=-1), kda.KDA_ERR_ARG),
    (dict(snapshot_every=32, snapshots=A), kda.KDA_ERR_ARG),
    (dict(snapshot_every=-64, snapshots=A), kda.KDA_ERR_ARG),
    (dict(snapshot_every=64), kda.KDA_ERR_ARG),
    (dict(snapshot_every=64, snapshots=A + 4), kda.KDA_ERR_ALIGN),
    (dict(decay_from_logit=2), kda.KDA_ERR_ARG),
    (dict(decay_from_logit=1, decay_mode=1), kda.KDA_ERR_ARG),
    (dict(decay_from_logit=1, decay_scale=A + 2), kda.KDA_ERR_ALIGN),
    (dict(decay_from_logit=1, decay_bias=A + 1), kda.KDA_ERR_ALIGN),
    (dict(conv_weight=A + 4), kda.KDA_ERR_ALIGN),
    (dict(conv_weight=A, conv_state=A + 8), kda.KDA_ERR_ALIGN),
])
def test_prefill_rejects_options(opt_kw, code):
    assert _prefill(opt=kda.kda_options_init(**opt_kw)) == code


@no_gpu
def test_log_alpha_requirements_follow_the_decay_mode():
    # per channel: required and 16-byte aligned; per head: 4-byte alignment
    assert _prefill(la=None) == kda.KDA_ERR_ARG
    assert _prefill(la=A + 4) == kda.KDA_ERR_ALIGN
    assert _prefill(la=None, opt=kda.kda_options_init(decay_mode="head")) == kda.KDA_ERR_ARG
    assert _prefill(la=A + 2, opt=kda.kda_options_init(decay_mode="head")) == kda.KDA_ERR_ALIGN
    # a 4-byte aligned per-head array, and no array without decay, pass the
    # pointer and alignment checks: the option check that follows them (a floor
    # below -5) is what stops these calls, before anything could launch
    assert _prefill(la=A + 4, opt=kda.kda_options_init(decay_mode="head", g_min=-6.0)) == \
        kda.KDA_ERR_ARG
    assert _prefill(la=A + 4, opt=kda.kda_options_init(g_min=-6.0)) == kda.KDA_ERR_ALIGN
    assert _prefill(la=None, opt=kda.kda_options_init(decay_mode="none", g_min=-6.0)) == \
        kda.KDA_ERR_ARG
    assert _prefill(la=None, dtype=7, opt=kda.kda_options_init(decay_mode="none")) == \
        kda.KDA_ERR_DTYPE


@no_gpu
def test_decode_and_norm_reject():
    lib = kda.load()
    opt = kda.kda_options_init()
    assert lib.kda_decode_step(A, A, A, A, A, None, A, 4, 2, 64, 64, kda.KDA_BF16,
                               ctypes.byref(opt), None) == kda.KDA_ERR_ARG
    assert lib.kda_decode_step(A, A, A, A, A, A, A, 0, 2, 64, 64, kda.KDA_BF16,
                               ctypes.byref(opt), None) == kda.KDA_ERR_SHAPE
    assert lib.kda_decode_step(A, A, A, A, A, A, A, 4, 2, 96, 96, kda.KDA_BF16,
                               ctypes.byref(opt), None) == kda.KDA_ERR_UNSUPPORTED
    assert lib.kda_decode_step(A, A, A + 4, A, A, A, A, 4, 2, 64, 64, kda.KDA_F32,
                               ctypes.byref(opt), None) == kda.KDA_ERR_ALIGN
    assert lib.kda_gated_rmsnorm(A, None, None, A, 4, 2, 64, 1e-6, kda.KDA_BF16,
                                 None) == kda.KDA_ERR_ARG
    assert lib.kda_gated_rmsnorm(A, A, None, A, 4, 2, 64, -1.0, kda.KDA_BF16,
                                 None) == kda.KDA_ERR_ARG
    assert lib.kda_gated_rmsnorm(A, A, None, A, 4, 2, 64, 1e-6, 3, None) == kda.KDA_ERR_DTYPE


def test_prefill_path_query():
    assert kda.kda_prefill_path(128, 1, 2, 32, 32, kda.KDA_F32,
                                kda.kda_options_init(impl="simt")) == ("simt", 1, 16)
    with pytest.raises(kda.KdaError):
        kda.kda_prefill_path(128, 1, 2, 48, 48)
    with pytest.raises(kda.KdaError):
        kda.kda_prefill_path(128, 1, 2, 64, 64, kda.KDA_BF16, kda.kda_options_init(g_min=-7.0))


def test_workspace_size_is_zero_for_simt():
    assert kda.kda_prefill_workspace_size(4096, 1, 96, 128, 128,
                                          kda.kda_options_init(impl="simt")) == 0
    assert kda.kda_prefill_workspace_size(4096, 1, 96, 48, 48) == 0


def _noalloc(**kw):
    lib = kda.load()
    args = dict(q=A, k=A, v=A, la=A, beta=A, S0=None, cu=None, N=1, o=A, S_T=A, T=64, H=2,
                dk=128, dv=128, dtype=kda.KDA_BF16, opt=None)
    args.update(kw)
    opt = args["opt"] if args["opt"] is not None else kda.kda_options_init()
    return lib.kda_prefill_noalloc(args["q"], args["k"], args["v"], args["la"], args["beta"],
                                   args["S0"], args["cu"], args["N"], args["o"], args["S_T"],
                                   args["T"], args["H"], args["dk"], args["dv"], args["dtype"],
                                   ctypes.byref(opt), None)


@no_gpu
@pytest.mark.parametrize("kw,code", [
    # what the tensor-core path does not take
    (dict(opt=kda.kda_options_init(chunk=16)), kda.KDA_ERR_UNSUPPORTED),
    (dict(opt=kda.kda_options_init(impl="simt")), kda.KDA_ERR_UNSUPPORTED),
    (dict(dtype=kda.KDA_F32), kda.KDA_ERR_UNSUPPORTED),
    (dict(dk=64, dv=64), kda.KDA_ERR_UNSUPPORTED),
    # kda_prefill's argument checks come before the scratch size, even for sizes
    # far beyond the scratch
    (dict(q=None, T=1 << 20, H=96), kda.KDA_ERR_ARG),
    (dict(q=A + 8, T=1 << 20, H=96), kda.KDA_ERR_ALIGN),
    (dict(dtype=7, T=1 << 20, H=96), kda.KDA_ERR_DTYPE),
    (dict(opt=kda.kda_options_init(chunk=32)), kda.KDA_ERR_UNSUPPORTED),
    # a valid call whose scratch exceeds the array
    (dict(T=4096, H=96), kda.KDA_ERR_WORKSPACE),
])
def test_noalloc_rejects(kw, code):
    assert _noalloc(**kw) == code
