"""GPU parity: libkda.so (through its C ABI) against the fp64 CPU oracle.

Both sides get the same seeded inputs (``inputs``).  Small cases are compared
element by element over whole tensors; the full-size workloads too (every head
of the K3-shaped and varlen prefills, every other head of the decay-extreme
prefill, 16 of the 64 decode sequences), the oracle running over groups of
heads.  Tolerances:
max-abs <= 2e-2 and rel-L2 <= 5e-3 for bf16 operands, 1e-4 for the fp32 path.
"""
from __future__ import annotations

import random

import numpy as np
import pytest
import torch

import oracle
from linear_attention_recurrence_prefill_gb300 import inputs, kda
from tests.parity_util import TOL_BF16, TOL_F32, assert_close

pytestmark = pytest.mark.gpu

IMPLS = ["simt", "tc"]


def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda")


def _oracle_prefill(inp, heads=None, gate=True):
    """Oracle o (or y) and S_T for the given head indices (all by default)."""
    idx = list(range(inp.H)) if heads is None else list(heads)
    sl = lambda t: t[:, idx].cpu() if t is not None else None  # noqa: E731
    S0 = inp.S0[:, idx].cpu() if inp.S0 is not None else None
    cu = inp.cu_seqlens.cpu() if inp.cu_seqlens is not None else None
    o, S_T = oracle.prefill(sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.log_alpha), sl(inp.beta),
                            S0, cu, N=inp.N)
    if gate and inp.gate is not None:
        o = oracle.gated_rmsnorm(o, sl(inp.gate))
    return o, S_T, idx


def _gpu_prefill(inp, impl, gate=True, **kw):
    o, S_T = kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0,
                             inp.cu_seqlens, N=inp.N, gate=inp.gate if gate else None,
                             impl=impl, **kw)
    torch.cuda.synchronize()
    assert kda.kda_get_last_error() == kda.KDA_OK
    return o, S_T


def _check(inp, impl, tol, heads=None, gate=True, **kw):
    o, S_T = _gpu_prefill(inp, impl, gate=gate, **kw)
    o_ref, S_ref, idx = _oracle_prefill(inp, heads, gate=gate)
    assert_close(o[:, idx], o_ref, tol, f"{inp.name} o/y")
    assert_close(S_T[:, idx], S_ref, tol, f"{inp.name} S_T")
    return o, S_T


# --------------------------------------------------------------------- small
def test_tiny_fp32():
    """Tiny workload: H=2, T=128, d=32, fp32, chunk 16 (whole tensors)."""
    dev = _cuda()
    inp = inputs.tiny(dev)
    _check(inp, "simt", TOL_F32)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("T", [1, 15, 64, 200, 1000])
def test_k3_shaped_small(impl, T):
    """K3-shaped distributions, 4 heads, ragged lengths, gated output."""
    dev = _cuda()
    inp = inputs.k3(dev, H=4, T=T, seed=11 + T)
    _check(inp, impl, TOL_BF16)


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("la", [-5.0, -7.0, 0.0])
def test_constant_decay_edges(impl, la):
    """Every channel at the floor (log alpha = -5, and -7 which the floor clamps to
    -5): over 16 tokens the running log-decay moves by 80, so the rescaled
    factors inside a chunk reach e^+-80 on both sides of a row; and no decay at
    all (log alpha = 0).  T = 200: three full chunks and a ragged tail."""
    dev = _cuda()
    inp = inputs.k3(dev, H=3, T=200, seed=41)
    inp.log_alpha = torch.full_like(inp.log_alpha, la)
    _check(inp, impl, TOL_BF16)


@pytest.mark.parametrize("d", [32, 64, 128])
def test_fp32_path_head_sizes(d):
    dev = _cuda()
    inp = inputs.k3(dev, H=3, T=100, d=d, dtype=torch.float32, seed=5)
    _check(inp, "simt", TOL_F32)


def test_varlen_small_edges():
    """Packed sequences with empty, single-token and ragged members."""
    dev = _cuda()
    lens = [0, 1, 17, 64, 65, 0, 130, 3]
    inp = inputs.varlen(dev, H=3, lengths=lens)
    inp.S0 = torch.randn((len(lens), 3, 128, 128), device=dev) * 0.05
    for impl in IMPLS:
        o, S_T = _check(inp, impl, TOL_BF16)
        # empty sequences hand back their initial state
        torch.testing.assert_close(S_T[0], inp.S0[0], rtol=0, atol=0)
        torch.testing.assert_close(S_T[5], inp.S0[5], rtol=0, atol=0)


@pytest.mark.parametrize("impl", IMPLS)
def test_many_short_sequences(impl):
    """2,500 packed sequences of 0..12 tokens (many empty, none a full chunk):
    the chunk-base prefix sum runs over several blocks of sequences and each
    chunk finds its sequence by search; every sequence starts from its own
    state."""
    dev = _cuda()
    g = torch.Generator().manual_seed(47)
    lens = torch.randint(0, 13, (2500,), generator=g).tolist()
    inp = inputs.varlen(dev, H=2, lengths=lens)
    inp.S0 = torch.randn((len(lens), 2, 128, 128), device=dev) * 0.05
    o, S_T = _check(inp, impl, TOL_BF16, max_seqlen=max(lens))
    empty = [n for n, L in enumerate(lens) if L == 0]
    assert empty and torch.equal(S_T[empty], inp.S0[empty])


@pytest.mark.parametrize("impl", IMPLS)
@pytest.mark.parametrize("case", range(16))
def test_random_shapes(impl, case):
    """Seeded random shapes against the oracle: head counts that do not divide
    the SM count, equal-length batches given with and without cu_seqlens, and
    packed sequences with empty, single-token and ragged members, with and
    without the gate."""
    dev = _cuda()
    rng = random.Random(1000 + case)
    H = rng.choice([1, 2, 3, 5, 7, 33])
    if rng.random() < 0.5:
        N = rng.choice([1, 2, 3])
        L = rng.choice([1, 17, 63, 64, 65, 127, 200])
        inp = inputs.k3(dev, H=H, T=N * L, seed=2000 + case)
        inp.N = N
        if N > 1 and rng.random() < 0.5:
            inp.cu_seqlens = torch.arange(0, N + 1, dtype=torch.int32, device=dev) * L
    else:
        lens = [rng.choice([0, 1, 5, 63, 64, 65, 130, 300]) for _ in range(rng.choice([2, 4, 9]))]
        lens[rng.randrange(len(lens))] = max(1, lens[0])
        inp = inputs.varlen(dev, H=H, lengths=lens, seed=2000 + case)
    inp.S0 = torch.randn((inp.N, H, 128, 128), device=dev) * 0.02
    _check(inp, impl, TOL_BF16, gate=rng.random() < 0.5)


def test_chain_order_longest_first():
    """With packed sequences the chunk-base kernel leaves, behind the N + 1 chunk
    bases at the head of the workspace, the order in which the chain grid takes
    the sequences: a permutation by descending chunk count, ties by index (the
    results themselves do not depend on it: each chain CTA is one sequence and
    head)."""
    dev = _cuda()
    lens = [70, 0, 640, 33, 64, 65, 129, 640, 1, 200]
    inp = inputs.varlen(dev, H=2, lengths=lens)
    need = kda.kda_prefill_workspace_size(inp.T, len(lens), inp.H, 128, 128)
    ws = torch.zeros(need, dtype=torch.uint8, device=dev)
    o, S_T = kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, None,
                             inp.cu_seqlens, len(lens), gate=inp.gate, impl="tc", workspace=ws)
    torch.cuda.synchronize()
    N = len(lens)
    head = ws[: (2 * N + 1) * 4].cpu().view(torch.int32).tolist()
    chunks = [(L + 63) // 64 for L in lens]
    base = [0]
    for c in chunks:
        base.append(base[-1] + c)
    assert head[: N + 1] == base
    assert head[N + 1:] == sorted(range(N), key=lambda n: (-chunks[n], n))
    _check(inp, "tc", TOL_BF16)


@pytest.mark.parametrize("impl", IMPLS)
def test_varlen_equals_separate_calls(impl):
    """Packed sequences give exactly what separate calls on each one give: every
    chunk restarts at its sequence start, and the kernels do the same arithmetic
    in the same order either way."""
    dev = _cuda()
    lens = [70, 0, 128, 33]
    inp = inputs.varlen(dev, H=2, lengths=lens)
    inp.S0 = torch.randn((len(lens), 2, 128, 128), device=dev) * 0.05
    o, S_T = _gpu_prefill(inp, impl)
    t0 = 0
    for n, L in enumerate(lens):
        sl = lambda x: x[t0:t0 + L].contiguous()  # noqa: E731
        if L:
            o1, S1 = kda.kda_prefill(sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.log_alpha),
                                     sl(inp.beta), inp.S0[n:n + 1].contiguous(), N=1,
                                     gate=sl(inp.gate), impl=impl)
            torch.cuda.synchronize()
            assert torch.equal(o[t0:t0 + L], o1), f"sequence {n}: output differs"
            assert torch.equal(S_T[n:n + 1], S1), f"sequence {n}: state differs"
        else:
            assert torch.equal(S_T[n], inp.S0[n])
        t0 += L


@pytest.mark.parametrize("impl", IMPLS)
def test_equal_length_batch(impl):
    """N = 3 sequences of 100 tokens given as N alone (no cu_seqlens): each
    sequence's chunks, the last one ragged, are found by arithmetic.  Checked
    against the oracle, and bit for bit against the same batch with explicit
    cu_seqlens."""
    dev = _cuda()
    inp = inputs.k3(dev, H=2, T=300, seed=43)
    inp.N = 3
    inp.S0 = torch.randn((3, 2, 128, 128), device=dev) * 0.05
    o, S_T = _check(inp, impl, TOL_BF16)
    cu = torch.tensor([0, 100, 200, 300], dtype=torch.int32, device=dev)
    o2, S2 = kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0, cu,
                             gate=inp.gate, impl=impl)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(S_T, S2)


def test_no_tokens():
    dev = _cuda()
    S0 = torch.randn((2, 3, 64, 64), device=dev)
    S_T = torch.empty_like(S0)
    cu = torch.zeros(3, dtype=torch.int32, device=dev)
    lib = kda.load()
    import ctypes
    opt = kda.kda_options_init()
    rc = lib.kda_prefill(None, None, None, None, None, S0.data_ptr(), cu.data_ptr(), 2, None,
                         S_T.data_ptr(), 0, 3, 64, 64, kda.KDA_BF16, ctypes.byref(opt),
                         torch.cuda.current_stream().cuda_stream)
    assert rc == kda.KDA_OK
    torch.cuda.synchronize()
    torch.testing.assert_close(S_T, S0, rtol=0, atol=0)


def test_options_logit_beta_qscale_weight():
    """beta as logit, q_scale and an RMSNorm weight, against the oracle."""
    dev = _cuda()
    inp = inputs.k3(dev, H=2, T=77, seed=3)
    z = torch.randn((inp.T, inp.H), device=dev).to(torch.bfloat16)
    w = torch.linspace(0.5, 1.5, 128, device=dev)
    for impl in IMPLS:
        o, S_T = kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, z, inp.S0, gate=inp.gate,
                                 norm_weight=w, beta_is_logit=True, q_scale=0.5, impl=impl)
        torch.cuda.synchronize()
        o_ref, S_ref = oracle.prefill(inp.q.cpu(), inp.k.cpu(), inp.v.cpu(),
                                      inp.log_alpha.cpu(), z.cpu(), inp.S0.cpu(),
                                      beta_is_logit=True, q_scale=0.5)
        y_ref = oracle.gated_rmsnorm(o_ref, inp.gate.cpu(), w=w.cpu())
        assert_close(o, y_ref, TOL_BF16, "y")
        assert_close(S_T, S_ref, TOL_BF16, "S_T")


def test_split_equals_whole():
    """Prefix caching: prefill(T) == prefill(T1) then prefill(T - T1) from S_T1."""
    dev = _cuda()
    inp = inputs.k3(dev, H=2, T=300, seed=4)
    for impl in IMPLS:
        o, S_T = _gpu_prefill(inp, impl)
        T1 = 100
        sl = lambda t, a, b: t[a:b].contiguous()  # noqa: E731
        o1, S1 = kda.kda_prefill(sl(inp.q, 0, T1), sl(inp.k, 0, T1), sl(inp.v, 0, T1),
                                 sl(inp.log_alpha, 0, T1), sl(inp.beta, 0, T1), inp.S0,
                                 gate=sl(inp.gate, 0, T1), impl=impl)
        o2, S2 = kda.kda_prefill(sl(inp.q, T1, None), sl(inp.k, T1, None), sl(inp.v, T1, None),
                                 sl(inp.log_alpha, T1, None), sl(inp.beta, T1, None), S1,
                                 gate=sl(inp.gate, T1, None), impl=impl)
        torch.cuda.synchronize()
        assert_close(torch.cat([o1, o2]), o.float(), TOL_BF16, "split o")
        assert_close(S2, S_T, TOL_BF16, "split S_T")


def test_gated_rmsnorm_standalone():
    dev = _cuda()
    for dt, tol in ((torch.bfloat16, TOL_BF16), (torch.float32, TOL_F32)):
        o = (torch.randn((50, 3, 128), device=dev) * 0.3).to(dt)
        g = torch.randn((50, 3, 128), device=dev).to(dt)
        w = torch.rand(128, device=dev) + 0.5
        y = kda.kda_gated_rmsnorm(o, g, w)
        torch.cuda.synchronize()
        ref = oracle.gated_rmsnorm(o.cpu().double().numpy(), g.cpu(), w=w.cpu())
        assert_close(y, ref, tol, "rmsnorm")
        y2 = kda.kda_gated_rmsnorm(o, g, w, y=o)       # in place
        torch.cuda.synchronize()
        assert_close(y2, ref, tol, "rmsnorm in place")


def test_tc_and_simt_agree():
    """Chunk 64 on the tensor cores == chunk 16 on CUDA cores (same problem)."""
    dev = _cuda()
    inp = inputs.k3(dev, H=3, T=333, seed=21)
    o1, S1 = _gpu_prefill(inp, "simt")
    o2, S2 = _gpu_prefill(inp, "tc")
    assert_close(o2, o1.float(), TOL_BF16, "tc vs simt y")
    assert_close(S2, S1, TOL_BF16, "tc vs simt S_T")


def test_tc_repeatable():
    """Two identical calls give bit-identical results (no races)."""
    dev = _cuda()
    inp = inputs.k3(dev, H=4, T=500, seed=22)
    o1, S1 = _gpu_prefill(inp, "tc")
    o2, S2 = _gpu_prefill(inp, "tc")
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


def test_tc_timeout_is_reported_and_recoverable():
    """A bounded device wait that gives up comes back as KDA_ERR_TIMEOUT, and
    the next call on the same context runs normally (no GPU fault involved:
    the test hook waits on a barrier nothing completes, before any async work)."""
    dev = _cuda()
    inp = inputs.k3(dev, H=2, T=100, seed=23)
    kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0, gate=inp.gate,
                    impl="tc", debug_timeout=True)
    assert kda.kda_get_last_error() == kda.KDA_ERR_TIMEOUT
    assert kda.kda_get_last_error() == kda.KDA_OK  # cleared
    _check(inp, "tc", TOL_BF16)


def test_tc_workspace_checks():
    dev = _cuda()
    inp = inputs.k3(dev, H=2, T=100, seed=24)
    need = kda.kda_prefill_workspace_size(inp.T, 1, inp.H, 128, 128)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device=dev)
    with pytest.raises(kda.KdaError) as ei:
        kda.kda_prefill(inp.q, inp.k, inp.v, inp.log_alpha, inp.beta, inp.S0, impl="tc",
                        workspace=small)
    assert ei.value.status == kda.KDA_ERR_WORKSPACE


# --------------------------------------------------------------------- decode
def _decode_run(d, steps, N=4, H=3, dtype=torch.bfloat16, gate=False):
    dev = _cuda()
    di = inputs.decode(dev, N=N, H=H, d=d, steps=steps, dtype=dtype)
    S = di.S.clone()
    S_ref = di.S.cpu().double().numpy()
    for t in range(steps):
        g = torch.randn((N, H, d), device=dev).to(dtype) if gate else None
        o = kda.kda_decode_step(di.q[t], di.k[t], di.v[t], di.log_alpha[t], di.beta[t], S, gate=g)
        o_ref, S_ref = oracle.decode_step(di.q[t].cpu(), di.k[t].cpu(), di.v[t].cpu(),
                                          di.log_alpha[t].cpu(), di.beta[t].cpu(), S_ref)
        if g is not None:
            o_ref = oracle.gated_rmsnorm(o_ref, g.cpu())
        torch.cuda.synchronize()
        tol = TOL_BF16 if dtype == torch.bfloat16 else TOL_F32
        assert_close(o, o_ref, tol, f"decode o step {t}")
    assert_close(S, S_ref, TOL_BF16 if dtype == torch.bfloat16 else TOL_F32, "decode S")


@pytest.mark.parametrize("d", [32, 64, 128])
def test_decode_small(d):
    _decode_run(d, steps=5)


def test_decode_fp32_and_gate():
    _decode_run(64, steps=3, dtype=torch.float32)
    _decode_run(128, steps=3, gate=True)


def test_prefill_equals_decode_steps():
    """T decode steps reach the state one prefill of T tokens reaches."""
    dev = _cuda()
    inp = inputs.k3(dev, H=2, T=40, seed=8)
    S = inp.S0.clone()
    outs = []
    for t in range(inp.T):
        outs.append(kda.kda_decode_step(inp.q[t:t + 1], inp.k[t:t + 1], inp.v[t:t + 1],
                                        inp.log_alpha[t:t + 1], inp.beta[t:t + 1], S))
    for impl in IMPLS:
        o, S_T = _gpu_prefill(inp, impl, gate=False)
        assert_close(torch.cat(outs).float(), o.float(), TOL_BF16, "decode vs prefill o")
        assert_close(S, S_T, TOL_BF16, "decode vs prefill S")


# ------------------------------------------------------------ full workloads
def _full_check(inp, heads, group=8, **kw):
    """Both implementations at full size against the oracle on `heads`.

    The GPU results of both are kept on the device; the oracle then runs over
    groups of `group` heads (bounded host memory) and each group is compared
    element by element.  Every group within max-abs and rel-L2 implies the
    whole compared tensor is within them too (the squared errors and norms add
    over groups)."""
    outs = {impl: _gpu_prefill(inp, impl, **kw) for impl in IMPLS}
    for g0 in range(0, len(heads), group):
        idx = list(heads[g0:g0 + group])
        o_ref, S_ref, _ = _oracle_prefill(inp, idx)
        for impl, (o, S_T) in outs.items():
            what = f"{inp.name} {impl} heads {idx[0]}..{idx[-1]}"
            assert_close(o[:, idx], o_ref, TOL_BF16, f"{what} o/y")
            assert_close(S_T[:, idx], S_ref, TOL_BF16, f"{what} S_T")
        del o_ref, S_ref


def test_k3_full():
    """K3-shaped prefill at full size (H=96, T=4096): every head, both paths."""
    dev = _cuda()
    inp = inputs.k3(dev)
    _full_check(inp, range(inp.H), group=16)


def test_varlen_full():
    """8 packed sequences of 1024..16384 tokens: every head, every sequence."""
    dev = _cuda()
    inp = inputs.varlen(dev)
    _full_check(inp, range(inp.H), group=8, max_seqlen=max(inp.meta["lengths"]))


def test_decode_full():
    """64 sequences x 96 heads, 256 steps in place; 16 sequences (all their
    heads) checked every 32 steps and at the end."""
    dev = _cuda()
    di = inputs.decode(dev)
    S = di.S.clone()
    pick = list(range(0, 64, 4))
    S_ref = di.S[pick].cpu().double().numpy()
    for t in range(di.q.shape[0]):
        o = kda.kda_decode_step(di.q[t], di.k[t], di.v[t], di.log_alpha[t], di.beta[t], S)
        o_ref, S_ref = oracle.decode_step(di.q[t, pick].cpu(), di.k[t, pick].cpu(),
                                          di.v[t, pick].cpu(), di.log_alpha[t, pick].cpu(),
                                          di.beta[t, pick].cpu(), S_ref)
        if t % 32 == 31:
            torch.cuda.synchronize()
            assert_close(o[pick], o_ref, TOL_BF16, f"decode o step {t}")
    torch.cuda.synchronize()
    assert_close(S[pick], S_ref, TOL_BF16, "decode S after 256 steps")


def test_extreme_full():
    """Decay-extreme prefill at full size (T=262144): 48 of the 96 heads (every
    other one), both paths."""
    dev = _cuda()
    inp = inputs.extreme(dev)
    _full_check(inp, range(0, inp.H, 2), group=8)
