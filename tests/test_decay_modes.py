"""Gated DeltaNet and DeltaNet modes (one decay per token and head, or none)
against the fp64 oracle.

KDA's per-channel decay reduces to Gated DeltaNet when every channel of a head
shares the decay, and to DeltaNet when there is none ("Kimi K3", section
"Forgetting different features at different rates"; "Kimi K3's hybrid block,
from first principles", section "From linear attention to the delta rule").
So the oracle runs its usual per-channel recurrence on the decay broadcast over
the channels (or on zeros), and the library runs with ``decay_mode`` "head"
(log_alpha [T, H]) or "none" (no log_alpha at all).
"""
from __future__ import annotations

import pytest
import torch

import oracle
from linear_attention_recurrence_prefill_gb300 import inputs, kda
from tests.parity_util import TOL_BF16, TOL_F32, assert_close

pytestmark = pytest.mark.gpu


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


def _head_decay(inp, seed):
    """A per-(token, head) log decay with the workload's distribution."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    z = torch.randn((inp.T, inp.H), generator=g) * 1.5
    return (-5.0 * torch.sigmoid(z)).to(inp.q.device)


def _expanded(inp, mode, la_head):
    """The per-channel log decay the oracle sees for this mode."""
    if mode == "head":
        return la_head[:, :, None].expand(inp.T, inp.H, inp.d).contiguous()
    return torch.zeros((inp.T, inp.H, inp.d), dtype=torch.float32, device=inp.q.device)


def _oracle(inp, la_full, gate=True):
    cu = inp.cu_seqlens.cpu() if inp.cu_seqlens is not None else None
    S0 = inp.S0.cpu() if inp.S0 is not None else None
    o, S_T = oracle.prefill(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(), la_full.cpu(),
                            inp.beta.cpu(), S0, cu, N=inp.N)
    if gate and inp.gate is not None:
        o = oracle.gated_rmsnorm(o, inp.gate.cpu())
    return o, S_T


@pytest.mark.parametrize("impl", ["simt", "tc"])
@pytest.mark.parametrize("mode", ["head", "none"])
@pytest.mark.parametrize("T", [64, 200])
def test_prefill_decay_modes(impl, mode, T):
    dev = _cuda()
    inp = inputs.k3(dev, H=3, T=T, seed=70 + T)
    la_head = _head_decay(inp, 90 + T)
    la_arg = la_head if mode == "head" else None
    o, S_T = kda.kda_prefill(inp.q, inp.k, inp.v, la_arg, inp.beta, inp.S0, N=1,
                             gate=inp.gate, impl=impl, decay_mode=mode)
    torch.cuda.synchronize()
    assert kda.kda_get_last_error() == kda.KDA_OK
    o_ref, S_ref = _oracle(inp, _expanded(inp, mode, la_head))
    assert_close(o, o_ref, TOL_BF16, f"{mode} {impl} y")
    assert_close(S_T, S_ref, TOL_BF16, f"{mode} {impl} S_T")


def test_prefill_head_mode_matches_its_channel_broadcast_on_the_gpu():
    """The per-head mode gives the per-channel path's result on the broadcast
    decay (same kernels, so up to rounding order only)."""
    dev = _cuda()
    inp = inputs.k3(dev, H=4, T=300, seed=77)
    la_head = _head_decay(inp, 78)
    o1, S1 = kda.kda_prefill(inp.q, inp.k, inp.v, la_head, inp.beta, inp.S0, N=1,
                             gate=inp.gate, impl="tc", decay_mode="head")
    o2, S2 = kda.kda_prefill(inp.q, inp.k, inp.v, _expanded(inp, "head", la_head), inp.beta,
                             inp.S0, N=1, gate=inp.gate, impl="tc")
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


@pytest.mark.parametrize("mode", ["head", "none"])
def test_prefill_decay_modes_fp32_varlen(mode):
    dev = _cuda()
    inp = inputs.k3(dev, H=2, T=150, d=32, dtype=torch.float32, seed=81)
    inp.cu_seqlens = torch.tensor([0, 40, 40, 150], dtype=torch.int32, device=dev)
    inp.N = 3
    inp.S0 = torch.randn((3, 2, 32, 32), device=dev) * 0.05
    la_head = _head_decay(inp, 82)
    la_arg = la_head if mode == "head" else None
    o, S_T = kda.kda_prefill(inp.q, inp.k, inp.v, la_arg, inp.beta, inp.S0, inp.cu_seqlens,
                             gate=inp.gate, impl="simt", decay_mode=mode)
    torch.cuda.synchronize()
    o_ref, S_ref = _oracle(inp, _expanded(inp, mode, la_head))
    assert_close(o, o_ref, TOL_F32, f"{mode} fp32 y")
    assert_close(S_T, S_ref, TOL_F32, f"{mode} fp32 S_T")


@pytest.mark.parametrize("mode", ["head", "none"])
def test_decode_decay_modes(mode):
    dev = _cuda()
    d = inputs.decode(dev, N=4, H=3, steps=2, seed=83)
    g = torch.Generator(device="cpu").manual_seed(84)
    la_head = (-5.0 * torch.sigmoid(torch.randn((4, 3), generator=g))).to(dev)
    S = d.S.clone()
    la_arg = la_head if mode == "head" else None
    o = kda.kda_decode_step(d.q[0], d.k[0], d.v[0], la_arg, d.beta[0], S, decay_mode=mode)
    torch.cuda.synchronize()
    la_full = (la_head[:, :, None].expand(4, 3, 128) if mode == "head"
               else torch.zeros((4, 3, 128), device=dev))
    o_ref, S_ref = oracle.decode_step(d.q[0].cpu(), d.k[0].cpu(), d.v[0].cpu(),
                                      la_full.contiguous().cpu(), d.beta[0].cpu(), d.S.cpu())
    assert_close(o, o_ref, TOL_BF16, f"{mode} decode o")
    assert_close(S, S_ref, TOL_BF16, f"{mode} decode S")
