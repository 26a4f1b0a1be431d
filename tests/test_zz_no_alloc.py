"""kda_prefill_noalloc: the prefill for callers that cannot allocate device
memory (it uses a fixed scratch array built into the library instead of a
caller-provided workspace).

Called through the C ABI on two calls in a row and checked against kda_prefill
(the entry point with a caller-allocated workspace): both run the same kernels
with the same arithmetic, so the results must be equal bit for bit.  The second
call uses different inputs and sizes, so a result that leaned on the first
call's leftovers in the shared scratch would show up.  The first case is also
compared with the CPU oracle, within the bf16 tolerance of the parity tests.
This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import oracle
from linear_attention_recurrence_prefill_gb300 import inputs, kda
from tests.parity_util import TOL_BF16, assert_close

pytestmark = pytest.mark.gpu


def _noalloc_c(inp, o, S_T, max_seqlen=0):
    """Raw C-ABI call; returns the status code."""
    lib = kda.load()
    opt = kda.kda_options_init(gate=inp.gate.data_ptr(), max_seqlen=max_seqlen)
    p = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    return lib.kda_prefill_noalloc(p(inp.q), p(inp.k), p(inp.v), p(inp.log_alpha), p(inp.beta),
                                   p(inp.S0), p(inp.cu_seqlens), inp.N, p(o), p(S_T), inp.T,
                                   inp.H, 128, 128, kda.KDA_BF16, ctypes.byref(opt),
                                   torch.cuda.current_stream().cuda_stream)


def _reference(inp):
    o, S_T = kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0,
                             inp.cu_seqlens, N=inp.N, gate=inp.gate, impl="tc")
    torch.cuda.synchronize()
    return o, S_T


def test_noalloc_matches_kda_prefill_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    cases = [inputs.k3(dev, H=4, T=700, seed=31),
             inputs.varlen(dev, H=3, lengths=[130, 0, 257, 64])]
    cases[1].S0 = torch.randn((4, 3, 128, 128), device=dev) * 0.05
    for i, inp in enumerate(cases):
        o = torch.empty_like(inp.q)
        S_T = torch.empty((inp.N, inp.H, 128, 128), dtype=torch.float32, device=dev)
        assert _noalloc_c(inp, o, S_T) == kda.KDA_OK
        torch.cuda.synchronize()
        assert kda.kda_get_last_error() == kda.KDA_OK
        o_ref, S_ref = _reference(inp)
        assert torch.equal(o, o_ref), f"{inp.name}: noalloc y differs from kda_prefill"
        assert torch.equal(S_T, S_ref), f"{inp.name}: noalloc S_T differs from kda_prefill"
        if i == 0:
            o_orc, S_orc = oracle.prefill(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(),
                                          inp.log_alpha.cpu(), inp.beta.cpu(), inp.S0.cpu())
            y_orc = oracle.gated_rmsnorm(o_orc, inp.gate.cpu())
            assert_close(o, y_orc, TOL_BF16, f"{inp.name} noalloc y vs oracle")
            assert_close(S_T, S_orc, TOL_BF16, f"{inp.name} noalloc S_T vs oracle")


def test_noalloc_refuses_sizes_beyond_the_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    inp = inputs.k3(dev, H=96, T=4096, seed=32)   # needs ~456 MB of scratch
    need = kda.kda_prefill_workspace_size(inp.T, 1, inp.H, 128, 128)
    assert need > kda.NOALLOC_SCRATCH_BYTES
    o = torch.zeros_like(inp.q)
    S_T = torch.zeros((1, 96, 128, 128), dtype=torch.float32, device=dev)
    assert _noalloc_c(inp, o, S_T) == kda.KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not o.any() and not S_T.any()          # nothing was launched
    with pytest.raises(kda.KdaError):
        kda.kda_prefill_noalloc(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0)


def test_noalloc_at_the_size_limit():
    """The largest size whose scratch fits the array runs (and equals
    kda_prefill bit for bit); one chunk more is refused before anything runs."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = torch.device("cuda")
    H = 8
    # scratch = header + H * (T / 64 + N) blocks: the largest T (a multiple of 64)
    # that fits, and the next one
    T = 64
    while kda.kda_prefill_workspace_size(T + 64, 1, H, 128, 128) <= kda.NOALLOC_SCRATCH_BYTES:
        T += 64
    assert kda.kda_prefill_workspace_size(T, 1, H, 128, 128) <= kda.NOALLOC_SCRATCH_BYTES
    inp = inputs.k3(dev, H=H, T=T, seed=33)
    o = torch.empty_like(inp.q)
    S_T = torch.empty((1, H, 128, 128), dtype=torch.float32, device=dev)
    assert _noalloc_c(inp, o, S_T) == kda.KDA_OK
    torch.cuda.synchronize()
    assert kda.kda_get_last_error() == kda.KDA_OK
    o_ref, S_ref = _reference(inp)
    assert torch.equal(o, o_ref) and torch.equal(S_T, S_ref)
    big = inputs.k3(dev, H=H, T=T + 64, seed=34)
    o2 = torch.zeros_like(big.q)
    S2 = torch.zeros((1, H, 128, 128), dtype=torch.float32, device=dev)
    assert _noalloc_c(big, o2, S2) == kda.KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert not o2.any() and not S2.any()
