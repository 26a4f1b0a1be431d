"""State snapshots during prefill (prefix caching).

A KDA prefix can be resumed only where its state was saved ("What's new in
Kimi K3", section "What it costs to serve").  With ``snapshot_every`` the
prefill also writes the state after every m * snapshot_every tokens of each
sequence.  Each snapshot must equal the final state of a prefill over that
prefix: checked against the fp64 oracle (tolerance) and against the library's
own prefill of the prefix (same kernels, so exactly).
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


def _prefix(inp, t0, n):
    """Tokens t0 .. t0 + n - 1 of the inputs (all heads)."""
    sl = lambda x: x[t0:t0 + n].contiguous()  # noqa: E731
    return sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.log_alpha), sl(inp.beta)


@pytest.mark.parametrize("impl", ["simt", "tc"])
@pytest.mark.parametrize("every", [64, 128])
def test_snapshots_equal_prefix_states(impl, every):
    dev = _cuda()
    inp = inputs.k3(dev, H=3, T=300, seed=101)
    o, S_T, snaps = kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0, N=1,
                                    gate=inp.gate, impl=impl, snapshot_every=every)
    torch.cuda.synchronize()
    assert kda.kda_get_last_error() == kda.KDA_OK
    assert snaps.shape == (1, 300 // every, 3, 128, 128)
    for m in range(300 // every):
        n = (m + 1) * every
        q, k, v, la, beta = _prefix(inp, 0, n)
        _, S_gpu = kda.kda_prefill(q, k, v, la, beta, inp.S0, N=1, impl=impl)
        torch.cuda.synchronize()
        assert torch.equal(snaps[0, m], S_gpu[0]), f"snapshot {m} != prefix prefill"
        _, S_ref = oracle.prefill(q.cpu(), k.cpu(), v.cpu(), la.cpu(), beta.cpu(),
                                  inp.S0.cpu(), N=1)
        assert_close(snaps[0, m], S_ref[0], TOL_BF16, f"snapshot {m}")
    # the snapshots change nothing else
    o2, S2 = kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0, N=1,
                             gate=inp.gate, impl=impl)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(S_T, S2)


@pytest.mark.parametrize("impl", ["simt", "tc"])
def test_snapshots_varlen(impl):
    """Packed sequences of 100, 128, 0 and 192 tokens, a snapshot every 64
    tokens, room for 3 per sequence (max_seqlen 192): each sequence fills the
    slots its length reaches, including one at its very end, and no others."""
    dev = _cuda()
    lengths = [100, 128, 0, 192]
    T = sum(lengths)
    inp = inputs.k3(dev, H=2, T=T, seed=102)
    cu = torch.tensor([0, 100, 228, 228, 420], dtype=torch.int32, device=dev)
    S0 = torch.randn((4, 2, 128, 128), device=dev) * 0.02
    snaps = torch.full((4, 3, 2, 128, 128), 7.0, device=dev)
    o, S_T, snaps = kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, S0, cu,
                                    gate=inp.gate, impl=impl, max_seqlen=192,
                                    snapshot_every=64, snapshots=snaps)
    torch.cuda.synchronize()
    assert kda.kda_get_last_error() == kda.KDA_OK
    starts = [0, 100, 228, 228]
    for n, (t0, L) in enumerate(zip(starts, lengths)):
        for m in range(3):
            if (m + 1) * 64 > L:
                assert bool((snaps[n, m] == 7.0).all()), f"seq {n} slot {m} written"
                continue
            q, k, v, la, beta = _prefix(inp, t0, (m + 1) * 64)
            _, S_ref = oracle.prefill(q.cpu(), k.cpu(), v.cpu(), la.cpu(), beta.cpu(),
                                      S0[n:n + 1].cpu(), N=1)
            assert_close(snaps[n, m], S_ref[0], TOL_BF16, f"seq {n} slot {m}")
        if L % 64 == 0 and L > 0:
            assert torch.equal(snaps[n, L // 64 - 1], S_T[n])


def test_snapshots_fp32_path():
    dev = _cuda()
    inp = inputs.k3(dev, H=2, T=256, d=64, dtype=torch.float32, seed=103)
    o, S_T, snaps = kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0, N=1,
                                    impl="simt", snapshot_every=128)
    torch.cuda.synchronize()
    q, k, v, la, beta = _prefix(inp, 0, 128)
    _, S_ref = oracle.prefill(q.cpu(), k.cpu(), v.cpu(), la.cpu(), beta.cpu(), inp.S0.cpu(), N=1)
    assert_close(snaps[0, 0], S_ref[0], TOL_F32, "fp32 snapshot 0")
    assert torch.equal(snaps[0, 1], S_T[0])
