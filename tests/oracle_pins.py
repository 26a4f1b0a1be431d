"""Pins that tie the CPU oracle to what the pages and the mathematics fix.

Every pin is a function ``pin_*(orc) -> None`` that raises ``AssertionError``
when the oracle build ``orc`` disagrees with something other than itself:
a brute-force unrolled matrix product, an exact invariant of the delta rule,
a worked example or number printed on the pages (``tests/golden``), a closed
form, or a textbook special case.  ``test_oracle.py`` runs them on the faithful
build, and on builds with a planted mistake to show that each mistake is caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _l2(x, eps):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


# ---------------------------------------------------------------- brute force
def brute_force(q, k, v, la, beta, S0, *, g_min=-5.0, l2=True, eps=1e-6):
    """Unrolled product form of S_t = (I - b k k^T) Diag(a) S_{t-1} + b k v^T.

    S_t = (M_t ... M_1) S0 + sum_s (M_t ... M_{s+1}) b_s k_s v_s^T with dense
    M_t = (I - b_t k_t k_t^T) Diag(a_t); o_t = S_t^T q_t.  Single head,
    q, k, la [T, dk], v [T, dv], beta [T], S0 [dk, dv].
    """
    T, dk = q.shape
    if l2:
        q, k = _l2(q, eps), _l2(k, eps)
    a = np.exp(np.minimum(np.maximum(la, g_min), 0.0))
    M = [(np.eye(dk) - beta[t] * np.outer(k[t], k[t])) @ np.diag(a[t]) for t in range(T)]
    B = [beta[t] * np.outer(k[t], v[t]) for t in range(T)]
    o, S_t = [], S0
    for t in range(T):
        P = np.eye(dk)
        acc = np.zeros_like(S0)
        for s in range(t, -1, -1):
            acc = acc + P @ B[s]
            P = P @ M[s]
        S_t = P @ S0 + acc
        o.append(S_t.T @ q[t])
    return np.array(o), S_t


def _run(orc, q, k, v, la, beta, S0=None, **kw):
    """Oracle on [T, H, d] fp64 arrays; returns (o [T, H, dv], S_T [N, H, dk, dv]).

    The L2-norm epsilon defaults to 0 here so that unit keys stay exactly unit."""
    kw.setdefault("eps_l2", 0.0)
    return orc.prefill(q, k, v, la, beta, S0, **kw)


def pin_brute_force(orc):
    """Oracle == unrolled product on tiny random problems (several shapes,
    non-unit keys, clamped and unclamped decays, dk != dv)."""
    for seed, (T, H, dk, dv, l2, eps) in enumerate([(6, 2, 4, 4, True, 1e-6),
                                                    (8, 1, 5, 7, False, 0.0),
                                                    (7, 3, 8, 8, True, 0.0),
                                                    (5, 2, 6, 3, False, 0.0),
                                                    (4, 1, 3, 5, True, 0.5)]):
        r = _rng(100 + seed)
        q = r.normal(size=(T, H, dk))
        k = r.normal(size=(T, H, dk)) * (0.6 if not l2 else 1.0)
        v = r.normal(size=(T, H, dv))
        la = r.uniform(-7.0, 0.2, size=(T, H, dk))
        beta = r.uniform(0.05, 1.0, size=(T, H))
        S0 = r.normal(size=(1, H, dk, dv))
        o, S_T = _run(orc, q, k, v, la, beta, S0, l2norm_qk=l2, eps_l2=eps)
        for h in range(H):
            o_ref, S_ref = brute_force(q[:, h], k[:, h], v[:, h], la[:, h], beta[:, h],
                                       S0[0, h], l2=l2, eps=eps)
            np.testing.assert_allclose(o[:, h], o_ref, rtol=1e-11, atol=1e-11)
            np.testing.assert_allclose(S_T[0, h], S_ref, rtol=1e-11, atol=1e-11)


# ---------------------------------------------------------------- delta rule
def pin_overwrite(orc):
    """beta = 1 and a unit key replace whatever was stored along k with v
    exactly (the delta rule as one gradient step on 1/2 |S^T k - v|^2), and
    leave every direction orthogonal to k with the faded state."""
    r = _rng(7)
    d = 8
    T = 5
    k = _unit(r.normal(size=(T, 1, d)))
    q = k.copy()                       # read back along the key just written
    v = r.normal(size=(T, 1, d))
    la = r.uniform(-3.0, 0.0, size=(T, 1, d))
    beta = np.ones((T, 1))
    S0 = r.normal(size=(1, 1, d, d))
    o, _ = _run(orc, q, k, v, la, beta, S0)
    np.testing.assert_allclose(o[:, 0], v[:, 0], rtol=0, atol=1e-12)
    # one step, check the orthogonal complement keeps Diag(a) S0
    o1, S1 = _run(orc, q[:1], k[:1], v[:1], la[:1], beta[:1], S0)
    faded = np.exp(la[0, 0])[:, None] * S0[0, 0]
    x = r.normal(size=d)
    x = x - (x @ k[0, 0]) * k[0, 0]     # x orthogonal to k
    np.testing.assert_allclose(S1[0, 0].T @ x, faded.T @ x, rtol=0, atol=1e-12)
    np.testing.assert_allclose(S1[0, 0].T @ k[0, 0], v[0, 0], rtol=0, atol=1e-12)


def pin_meeting(orc):
    """The pages' whiteboard example, built exactly: orthonormal rows, alpha = 1,
    beta = 1.  Editing the meeting-day row changes only that row; the board
    keeps three rows."""
    g = golden("meeting.json")
    d = 4
    keys, vals = g["key_rows"], g["value_codes"]
    writes = g["writes"]
    T = len(writes)
    k = np.zeros((T, 1, d))
    v = np.zeros((T, 1, d))
    for t, (row, val) in enumerate(writes):
        k[t, 0, keys[row]] = 1.0
        v[t, 0, vals[val]] = 1.0
    q = k.copy()
    la = np.zeros((T, 1, d))
    beta = np.ones((T, 1))
    _, S_before = _run(orc, q[:3], k[:3], v[:3], la[:3], beta[:3])
    _, S_after = _run(orc, q, k, v, la, beta)
    B0, B1 = S_before[0, 0], S_after[0, 0]
    for row, val in g["expected_board"].items():
        e = np.zeros(d)
        e[vals[val]] = 1.0
        np.testing.assert_array_equal(B1[keys[row]], e)
    for row in ("client", "budget"):           # untouched rows: bit-exact
        np.testing.assert_array_equal(B1[keys[row]], B0[keys[row]])
    assert int((np.abs(B1).sum(1) > 0).sum()) == g["expected_rows"]


# ------------------------------------------------- linear-attention reductions
def pin_linear_attention(orc):
    """alpha = 1 reductions (see the linear-attention paragraph of the pages):
    L0 alpha=1, beta=0: S never changes, o_t = S0^T q_t exactly;
    L1 alpha=1, orthonormal keys, S0=0: o_t = sum_{s<=t} beta_s (q_t.k_s) v_s,
       and with beta = 1 that is plain (unnormalised) linear attention;
    L2 alpha=1, S0=0, generic keys, beta = eps -> 0: o_t/eps -> sum (q_t.k_s) v_s."""
    r = _rng(11)
    T, d = 6, 8
    q = _unit(r.normal(size=(T, 1, d)))
    k = _unit(r.normal(size=(T, 1, d)))
    v = r.normal(size=(T, 1, d))
    la = np.zeros((T, 1, d))
    S0 = r.normal(size=(1, 1, d, d))
    # L0
    o, S_T = _run(orc, q, k, v, la, np.zeros((T, 1)), S0)
    np.testing.assert_array_equal(S_T[0, 0], S0[0, 0])
    np.testing.assert_allclose(o[:, 0], q[:, 0] @ S0[0, 0], rtol=0, atol=1e-13)
    # L1 (orthonormal keys: columns of a random orthogonal matrix)
    Qm, _ = np.linalg.qr(r.normal(size=(d, d)))
    ko = Qm.T[:T].reshape(T, 1, d)
    for beta in (r.uniform(0.1, 1.0, size=(T, 1)), np.ones((T, 1))):
        o, _ = _run(orc, q, ko, v, la, beta)
        ref = np.array([sum(beta[s, 0] * (q[t, 0] @ ko[s, 0]) * v[s, 0] for s in range(t + 1))
                        for t in range(T)])
        np.testing.assert_allclose(o[:, 0], ref, rtol=0, atol=1e-12)
    # L2
    eps = 1e-7
    o, _ = _run(orc, q, k, v, la, np.full((T, 1), eps))
    ref = np.array([sum((q[t, 0] @ k[s, 0]) * v[s, 0] for s in range(t + 1)) for t in range(T)])
    np.testing.assert_allclose(o[:, 0] / eps, ref, rtol=0, atol=1e-5)


# ---------------------------------------------------------------- decay
def pin_half_life(orc):
    """With beta = 0 and S0 = I a channel of constant alpha decays as alpha^n;
    alpha = 0.99 halves it at n = ln 0.5 / ln 0.99 = 68.97, i.e. about 69
    tokens; log alpha = ln 0.5 / n gives exactly one half after n tokens."""
    g = golden("half_life.json")
    alpha = g["alpha"]
    n_half = math.log(0.5) / math.log(alpha)
    assert round(n_half) == g["n_half_about"]
    d, T = 4, 80
    q = np.tile(np.eye(d)[None, None, 0], (T, 1, 1))    # read channel 0
    k = np.tile(np.eye(d)[None, None, 1], (T, 1, 1))
    v = np.zeros((T, 1, d))
    la = np.full((T, 1, d), math.log(alpha))
    S0 = np.eye(d)[None, None]
    o, _ = _run(orc, q, k, v, la, np.zeros((T, 1)), S0, l2norm_qk=False)
    trace = o[:, 0, 0]                                   # alpha^(t+1)
    np.testing.assert_allclose(trace, alpha ** np.arange(1, T + 1), rtol=1e-13)
    first_below = int(np.argmax(trace <= 0.5)) + 1
    assert first_below == g["n_half_about"]
    n = 50
    la2 = np.full((n, 1, d), math.log(0.5) / n)
    o2, _ = _run(orc, q[:n], k[:n], v[:n], la2, np.zeros((n, 1)), S0, l2norm_qk=False)
    assert abs(o2[-1, 0, 0] - 0.5) < 1e-13


def pin_floor(orc):
    """log alpha is floored at -5 (retention >= e^-5 ~ 0.0067) and capped at 0."""
    g = golden("floor.json")
    d = 4
    q = np.eye(d)[None, None, 0]
    k = np.eye(d)[None, None, 1]
    v = np.zeros((1, 1, d))
    S0 = np.eye(d)[None, None]
    o7, _ = _run(orc, q, k, v, np.full((1, 1, d), -7.0), np.zeros((1, 1)), S0, l2norm_qk=False)
    o5, _ = _run(orc, q, k, v, np.full((1, 1, d), g["log_alpha_floor"]), np.zeros((1, 1)), S0,
                 l2norm_qk=False)
    np.testing.assert_array_equal(o7, o5)
    assert round(float(o5[0, 0, 0]), g["decimals"]) == g["retention_floor_about"]
    op, _ = _run(orc, q, k, v, np.full((1, 1, d), 0.5), np.zeros((1, 1)), S0, l2norm_qk=False)
    assert op[0, 0, 0] == 1.0
    # the floor also holds inside a full update
    r = _rng(5)
    T = 6
    qq, kk, vv = r.normal(size=(T, 1, d)), r.normal(size=(T, 1, d)), r.normal(size=(T, 1, d))
    bb = r.uniform(0.2, 0.9, size=(T, 1))
    lo = r.uniform(-12.0, -5.0, size=(T, 1, d))
    a1, s1 = _run(orc, qq, kk, vv, lo, bb)
    a2, s2 = _run(orc, qq, kk, vv, np.full_like(lo, -5.0), bb)
    np.testing.assert_array_equal(a1, a2)
    np.testing.assert_array_equal(s1, s2)


def pin_scalar_decay(orc):
    """All channels equal reduces KDA to Gated DeltaNet (one decay per head):
    S_t = a_t (I - b k k^T) S_{t-1} + b k v^T, here as a separate scalar loop."""
    r = _rng(13)
    T, d = 9, 6
    q, k = _unit(r.normal(size=(T, d))), _unit(r.normal(size=(T, d)))
    v = r.normal(size=(T, d))
    a = r.uniform(0.3, 1.0, size=T)
    b = r.uniform(0.1, 1.0, size=T)
    S = r.normal(size=(d, d))
    S0 = S.copy()
    ref = []
    for t in range(T):
        S = a[t] * (S - b[t] * np.outer(k[t], k[t] @ S)) + b[t] * np.outer(k[t], v[t])
        ref.append(S.T @ q[t])
    la = np.repeat(np.log(a)[:, None, None], d, axis=2)
    o, S_T = _run(orc, q[:, None], k[:, None], v[:, None], la, b[:, None], S0[None, None])
    np.testing.assert_allclose(o[:, 0], np.array(ref), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S_T[0, 0], S, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- prologue
def pin_l2norm(orc):
    """With L2 normalisation on, rescaling q or k by a positive factor changes
    nothing (the layer normalises them; same section as the recurrence)."""
    r = _rng(17)
    T, H, d = 7, 2, 8
    q, k, v = r.normal(size=(T, H, d)), r.normal(size=(T, H, d)), r.normal(size=(T, H, d))
    la = r.uniform(-5, 0, size=(T, H, d))
    b = r.uniform(0.1, 1, size=(T, H))
    o1, s1 = _run(orc, q, k, v, la, b, eps_l2=0.0)
    o2, s2 = _run(orc, 7.0 * q, 3.0 * k, v, la, b, eps_l2=0.0)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s1, s2, rtol=1e-12, atol=1e-12)
    qn = q / np.linalg.norm(q, axis=-1, keepdims=True)
    kn = k / np.linalg.norm(k, axis=-1, keepdims=True)
    o3, _ = _run(orc, qn, kn, v, la, b, l2norm_qk=False)
    np.testing.assert_allclose(o1, o3, rtol=1e-12, atol=1e-12)


def pin_beta_logit(orc):
    """beta given as a logit equals beta given as sigmoid(logit)."""
    r = _rng(19)
    T, H, d = 6, 2, 8
    q, k, v = r.normal(size=(T, H, d)), r.normal(size=(T, H, d)), r.normal(size=(T, H, d))
    la = r.uniform(-5, 0, size=(T, H, d))
    z = r.normal(size=(T, H))
    o1, _ = _run(orc, q, k, v, la, z, beta_is_logit=True)
    o2, _ = _run(orc, q, k, v, la, 1.0 / (1.0 + np.exp(-z)))
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- structure
def pin_split_and_decode(orc):
    """Prefix caching: prefill(T) = prefill(T1) then prefill(rest) from S_T1,
    and = T single-token decode steps; packed sequences = separate calls;
    a zero-length sequence returns its S0."""
    r = _rng(23)
    T, H, d = 11, 2, 6
    q, k, v = r.normal(size=(T, H, d)), r.normal(size=(T, H, d)), r.normal(size=(T, H, d))
    la = r.uniform(-5, 0, size=(T, H, d))
    b = r.uniform(0.1, 1, size=(T, H))
    S0 = r.normal(size=(1, H, d, d))
    o, S_T = _run(orc, q, k, v, la, b, S0)
    T1 = 4
    oa, Sa = _run(orc, q[:T1], k[:T1], v[:T1], la[:T1], b[:T1], S0)
    ob, Sb = _run(orc, q[T1:], k[T1:], v[T1:], la[T1:], b[T1:], Sa)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(Sb, S_T, rtol=1e-13, atol=1e-13)
    S = S0.copy()
    for t in range(T):
        ot, S = orc.decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], la[t:t + 1], b[t:t + 1], S,
                                eps_l2=0.0)
        np.testing.assert_allclose(ot[0], o[t], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S, S_T, rtol=1e-13, atol=1e-13)
    # packed: [T1 tokens | 0 tokens | rest]
    cu = np.array([0, T1, T1, T], dtype=np.int32)
    S03 = r.normal(size=(3, H, d, d))
    op, Sp = orc.prefill(q, k, v, la, b, S03, cu, eps_l2=0.0)
    o1, S1 = _run(orc, q[:T1], k[:T1], v[:T1], la[:T1], b[:T1], S03[0:1])
    o3, S3 = _run(orc, q[T1:], k[T1:], v[T1:], la[T1:], b[T1:], S03[2:3])
    np.testing.assert_allclose(op, np.concatenate([o1, o3]), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(Sp[0], S1[0], rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(Sp[1], S03[1])
    np.testing.assert_allclose(Sp[2], S3[0], rtol=1e-13, atol=1e-13)
    # head subset = the same heads of the full run
    o_h, S_h = _run(orc, q, k, v, la, b, S0, heads=(1, 1))
    np.testing.assert_array_equal(o_h[:, 0], o[:, 1])
    np.testing.assert_array_equal(S_h[0, 0], S_T[0, 1])


def pin_gated_rmsnorm(orc):
    """Closed forms of the per-head RMSNorm x sigmoid gate: a constant vector
    c*1 maps to sign(c)*sigmoid(g); a one-hot a*e_j maps to sqrt(dv)*sigmoid(g)
    at j; a weight vector scales channel-wise."""
    dv = 16
    o = np.zeros((3, 2, dv))
    o[0, 0] = 2.5
    o[0, 1] = -0.75
    o[1, 0, 5] = 3.0
    o[1, 1, 0] = -0.1
    o[2] = _rng(29).normal(size=(2, dv))
    gate = _rng(31).normal(size=(3, 2, dv))
    sg = 1.0 / (1.0 + np.exp(-gate))
    y = orc.gated_rmsnorm(o, gate, eps=0.0)
    np.testing.assert_allclose(y[0, 0], sg[0, 0], rtol=1e-14)
    np.testing.assert_allclose(y[0, 1], -sg[0, 1], rtol=1e-14)
    assert abs(y[1, 0, 5] - math.sqrt(dv) * sg[1, 0, 5]) < 1e-13
    assert np.count_nonzero(y[1, 0]) == 1
    assert abs(y[1, 1, 0] + math.sqrt(dv) * sg[1, 1, 0]) < 1e-13
    # rms of the normalised vector is 1 before the gate
    yn = orc.gated_rmsnorm(o[2:3], np.full((1, 2, dv), 50.0), eps=0.0)
    np.testing.assert_allclose(np.sqrt((yn ** 2).mean(-1)), 1.0, rtol=1e-12)
    w = np.linspace(0.5, 2.0, dv)
    yw = orc.gated_rmsnorm(o, gate, w=w, eps=0.0)
    np.testing.assert_allclose(yw, y * w, rtol=1e-14)
    # head offset selects the gate's heads
    y1 = orc.gated_rmsnorm(o[:, 1:2], gate, eps=0.0, h0=1)
    np.testing.assert_allclose(y1[:, 0], y[:, 1], rtol=1e-14)


# ---------------------------------------------------------------- input widening
# bf16 bit patterns with their values written out from the IEEE binary32 layout
# (a bf16 value is the upper half of a binary32 pattern)
BF16_KNOWN = [
    (0x3F80, 1.0),
    (0xC0A0, -5.0),
    (0x3FC0, 1.5),
    (0x0001, 2.0 ** -133),                         # smallest positive subnormal
    (0x8000, -0.0),
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),      # largest finite
    (0x4049, 3.140625),
    (0xBE80, -0.25),
]


def _bf16_tensor(bits, shape=None):
    import torch
    t = torch.from_numpy(np.array(bits, dtype=np.uint16).view(np.int16).copy()).view(
        torch.bfloat16)
    return t.reshape(shape) if shape is not None else t


def _bf16_values(t):
    """fp64 values of a bf16 tensor by the library's own conversion."""
    import torch
    return t.to(torch.float64).numpy()


def pin_input_widening(orc):
    """Inputs stored as bf16 (raw 16-bit patterns) or fp32 are widened exactly.

    Known bf16 patterns pass through exact identity paths of the recurrence
    (S0 = I with beta = 0 returns q; one write with beta = 1 returns v, k and
    beta; the fade of S0 = I returns exp of the clamped log alpha), and through
    the gate of the RMSNorm epilogue.  Random bf16 and fp32 inputs give results
    bit-identical to the fp64 run on the same values, for the prefill, the
    decode step and the gate."""
    import torch
    d = len(BF16_KNOWN)
    bits = [b for b, _ in BF16_KNOWN]
    vals = np.array([x for _, x in BF16_KNOWN])
    row = _bf16_tensor(bits, (1, 1, d))
    eye = np.eye(d)
    z = lambda *s: torch.zeros(s, dtype=torch.bfloat16)  # noqa: E731
    one_hot = lambda c, s: _bf16_tensor([0x3F80 if i == c else 0 for i in range(d)], s)  # noqa: E731
    kw = dict(l2norm_qk=False, eps_l2=0.0)
    # q: S0 = I, beta = 0, no decay -> o = q
    o, _ = orc.prefill(row, z(1, 1, d), z(1, 1, d), np.zeros((1, 1, d)), z(1, 1),
                       eye[None, None], **kw)
    np.testing.assert_array_equal(o[0, 0], vals)
    # v: S0 = 0, beta = 1, k = q = e_0 -> o = v
    e0 = one_hot(0, (1, 1, d))
    o, S = orc.prefill(e0, e0, row, np.zeros((1, 1, d)), _bf16_tensor([0x3F80], (1, 1)), **kw)
    np.testing.assert_array_equal(o[0, 0], vals)
    np.testing.assert_array_equal(S[0, 0, 0], vals)
    # k: head h reads channel h of the key just written (v = e_0): o[h, 0] = k_h
    H = d
    krow = torch.cat([row] * H, dim=1)
    qh = torch.cat([one_hot(h, (1, 1, d)) for h in range(H)], dim=1)
    vh = torch.cat([e0] * H, dim=1)
    o, _ = orc.prefill(qh, krow, vh, np.zeros((1, H, d)), _bf16_tensor([0x3F80] * H, (1, H)),
                       **kw)
    np.testing.assert_array_equal(o[0, :, 0], vals)
    # beta: S0 = 0, k = q = v = e_0 -> o_0 = beta (one head per pattern)
    e0h = torch.cat([e0] * H, dim=1)
    o, _ = orc.prefill(e0h, e0h, e0h, np.zeros((1, H, d)), _bf16_tensor(bits, (1, H)), **kw)
    np.testing.assert_array_equal(o[0, :, 0], vals)
    # log alpha (bf16 and fp32 storage): S0 = I, beta = 0, head h reads channel h
    la32 = np.array([-5.0, -0.25, -1e-4, -3.3, 0.0, -4.99, -0.001, -2.0], dtype=np.float32)
    for la, la64 in ((row.expand(1, H, d).contiguous(), vals),
                     (np.broadcast_to(la32, (1, H, d)).copy(), la32.astype(np.float64))):
        S0 = np.broadcast_to(eye, (1, H, d, d)).copy()
        o, _ = orc.prefill(qh, z(1, H, d), z(1, H, d), la, z(1, H), S0, **kw)
        want = np.exp(np.minimum(np.maximum(la64, -5.0), 0.0))
        np.testing.assert_array_equal(np.diagonal(o[0]), want)
    # the gate: y = sigmoid(g) for a constant unit output
    y = orc.gated_rmsnorm(np.ones((1, 1, d)), row, eps=0.0)
    np.testing.assert_allclose(y[0, 0], 1.0 / (1.0 + np.exp(-vals)), rtol=1e-15, atol=0)
    # random inputs: bf16 / fp32 storage == fp64 of the same values, bit for bit
    r = _rng(37)
    T, H2, dd = 9, 3, 8
    g = torch.Generator().manual_seed(37)
    qb, kb, vb = (torch.randn((T, H2, dd), generator=g).to(torch.bfloat16) for _ in range(3))
    bb = torch.rand((T, H2), generator=g).to(torch.bfloat16)
    lab = (-6.0 * torch.rand((T, H2, dd), generator=g)).to(torch.bfloat16)
    la_f32 = r.uniform(-6.0, 0.1, size=(T, H2, dd)).astype(np.float32)
    S0 = r.normal(size=(1, H2, dd, dd))
    for la_in, la_ref in ((lab, _bf16_values(lab)), (la_f32, la_f32.astype(np.float64))):
        o1, s1 = orc.prefill(qb, kb, vb, la_in, bb, S0)
        o2, s2 = orc.prefill(_bf16_values(qb), _bf16_values(kb), _bf16_values(vb), la_ref,
                             _bf16_values(bb), S0)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(s1, s2)
        d1, n1 = orc.decode_step(qb[:1], kb[:1], vb[:1], la_in[:1], bb[:1], S0)
        d2, n2 = orc.decode_step(_bf16_values(qb[:1]), _bf16_values(kb[:1]), _bf16_values(vb[:1]),
                                 la_ref[:1], _bf16_values(bb[:1]), S0)
        np.testing.assert_array_equal(d1, d2)
        np.testing.assert_array_equal(n1, n2)
    q32, k32, v32 = (r.normal(size=(T, H2, dd)).astype(np.float32) for _ in range(3))
    b32 = r.uniform(0, 1, size=(T, H2)).astype(np.float32)
    o1, s1 = orc.prefill(q32, k32, v32, la_f32, b32, S0)
    o2, s2 = orc.prefill(q32.astype(np.float64), k32.astype(np.float64), v32.astype(np.float64),
                         la_f32.astype(np.float64), b32.astype(np.float64), S0)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(s1, s2)
    gb = torch.randn((T, H2, dd), generator=g).to(torch.bfloat16)
    g32 = r.normal(size=(T, H2, dd)).astype(np.float32)
    for gin, gref in ((gb, _bf16_values(gb)), (g32, g32.astype(np.float64))):
        np.testing.assert_array_equal(orc.gated_rmsnorm(o1, gin), orc.gated_rmsnorm(o1, gref))


# ---------------------------------------------------------------- decay from logits
def _retention(orc, z, *, A=None, b=None, g_min=-5.0):
    """exp(log alpha) for decay logits z [d] (one head per channel reads its
    channel of S0 = I after one step with beta = 0)."""
    d = z.shape[-1]
    H = d
    eye = np.eye(d)
    q = np.broadcast_to(eye[None], (1, H, d)).copy()       # head h reads channel h
    zero = np.zeros((1, H, d))
    la = np.broadcast_to(z, (1, H, d)).copy()
    S0 = np.broadcast_to(eye, (1, H, d, d)).copy()
    Ah = None if A is None else np.full(H, float(A))
    bh = None if b is None else np.broadcast_to(b, (H, d)).copy()
    o, _ = orc.prefill(q, zero, zero, la, np.zeros((1, H)), S0, l2norm_qk=False, eps_l2=0.0,
                       decay_from_logit=True, decay_scale=Ah, decay_bias=bh, g_min=g_min)
    return np.diagonal(o[0])


def pin_decay_logit(orc):
    """log alpha from the decay logit z through the bounded sigmoid with one
    scale A_h per head: every factor lies in [e^g_min, 1] whatever z is, the
    extremes are reached as z -> +-inf, z + b = 0 gives exactly half the
    floor, larger z forgets more, A_h scales the logit inside the sigmoid,
    the per-channel bias adds to z, and A_h = 1, b = 0 reproduces the plain
    path fed log alpha = -5 sigmoid(z)."""
    z = np.array([1e3, -1e3, 0.0, 2.0, -2.0, 40.0])
    a = _retention(orc, z)
    assert a[0] == math.exp(-5.0) and a[1] == 1.0
    assert a[2] == math.exp(-2.5)
    a2 = _retention(orc, z, g_min=-2.0)
    assert a2[0] == math.exp(-2.0) and a2[1] == 1.0 and a2[2] == math.exp(-1.0)
    r = _rng(41)
    zz = np.sort(r.uniform(-50.0, 50.0, size=16))
    aa = _retention(orc, zz)
    assert np.all(aa >= math.exp(-5.0)) and np.all(aa <= 1.0)
    assert np.all(np.diff(aa) <= 0.0)                   # monotone: more forgetting
    x = r.normal(size=8)
    np.testing.assert_array_equal(_retention(orc, x, A=2.0), _retention(orc, 2.0 * x))
    y = r.normal(size=8)
    np.testing.assert_array_equal(_retention(orc, x, b=y), _retention(orc, x + y))
    # the full recurrence: logits in, the same as the activated log alpha in
    T, H, d = 9, 2, 8
    q, k, v = r.normal(size=(T, H, d)), r.normal(size=(T, H, d)), r.normal(size=(T, H, d))
    zt = r.normal(size=(T, H, d)) * 1.5
    bt = r.uniform(0.1, 1.0, size=(T, H))
    o1, s1 = orc.prefill(q, k, v, zt, bt, decay_from_logit=True)
    o2, s2 = orc.prefill(q, k, v, -5.0 / (1.0 + np.exp(-zt)), bt)
    np.testing.assert_allclose(o1, o2, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(s1, s2, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- short convolution
def _swish(y):
    return y / (1.0 + np.exp(-y))


def pin_short_conv_impulse(orc):
    """A unit impulse through the width-4 causal convolution + Swish returns
    swish(tap x height) at the impulse and the three tokens after it, oldest
    tap last, and exactly zero before it and from four tokens on (a
    constant key overwritten with beta = 1 reads back v's output)."""
    T, d, t0 = 10, 4, 2
    r = _rng(43)
    w = r.normal(size=(3, 1, d, 4))
    w[0, 0] = w[1, 0] = [0.0, 0.0, 0.0, 1.0]         # q, k: identity taps
    e0 = np.zeros((T, 1, d))
    e0[:, 0, 0] = 1.0
    heights = np.array([0.5, -1.25, 2.0, 0.75])
    v = np.zeros((T, 1, d))
    v[t0, 0] = heights
    o, _ = orc.prefill(e0, e0, v, np.zeros((T, 1, d)), np.ones((T, 1)), eps_l2=0.0,
                       conv_weight=w)
    want = np.zeros((T, d))
    for t in range(t0, t0 + 4):
        want[t] = _swish(w[2, 0, :, 3 - (t - t0)] * heights)
    np.testing.assert_allclose(o[:, 0], want, rtol=1e-14, atol=1e-15)
    # the query's convolution, read through S0 = I with beta = 0 (no norm)
    q = np.zeros((T, 1, d))
    q[t0, 0] = heights
    o, _ = orc.prefill(q, np.zeros((T, 1, d)), np.zeros((T, 1, d)), np.zeros((T, 1, d)),
                       np.zeros((T, 1)), np.eye(d)[None, None], l2norm_qk=False,
                       conv_weight=np.repeat(w[2:3], 3, axis=0))
    np.testing.assert_allclose(o[:, 0], want, rtol=1e-14, atol=1e-15)


def _conv_ref(x, w, window):
    """Causal conv of x [T, H, d] with taps w [H, d, 4] (oldest first) after the
    window [3, H, d], by numpy.convolve per channel, then Swish."""
    T, H, d = x.shape
    full = np.concatenate([window, x], axis=0)
    y = np.empty_like(x)
    for h in range(H):
        for c in range(d):
            y[:, h, c] = np.convolve(full[:, h, c], w[h, c, ::-1])[3:3 + T]
    return _swish(y)


def _held_q(orc, q, w, win):
    """The stored convolution + Swish output of q, read back exactly: with
    S0 = I, beta = 0, no decay and no norm, o_t = the stored q_t."""
    T, H, d = q.shape
    z = q * 0                                  # k, v: zeros of q's storage type
    S0 = np.broadcast_to(np.eye(d), (1, H, d, d)).copy()
    o, _ = orc.prefill(q, z, z, np.zeros((T, H, d)), np.zeros((T, H)), S0, l2norm_qk=False,
                       conv_weight=w, conv_state=win)
    return o


def pin_short_conv_storage(orc):
    """With bf16 (fp32) data the convolution's output is held in bf16 (fp32)
    before the rest of the layer, rounded to nearest even.  Against the fp64
    convolution + Swish by numpy.convolve: every stored bf16 value is that
    value rounded to nearest bf16 by the library's conversion, except where it
    lies within the fp32 evaluation error of a rounding boundary (then either
    neighbour); every stored fp32 value is within that evaluation error of it
    (relative 1e-6, plus 2e-6 absolute where the convolution's sum cancels)."""
    import torch
    r = _rng(53)
    T, H, d = 40, 2, 16
    g = torch.Generator().manual_seed(53)
    q = (torch.randn((T, H, d), generator=g) * 2.0).to(torch.bfloat16)
    w = r.normal(size=(3, H, d, 4)) * 0.7
    win = (torch.randn((1, 3, 3, H, d), generator=g) * 2.0).to(torch.bfloat16)
    true = _conv_ref(q.double().numpy(), w[0], win[0, 0].double().numpy())
    held = _held_q(orc, q, w, win)
    want = torch.from_numpy(true).float().bfloat16().double().numpy()
    ok = held == want
    # mismatches only next to a rounding boundary, and only by one bf16 unit
    _, e = np.frexp(np.abs(true))
    ulp = np.ldexp(1.0, e - 8)                 # bf16 spacing at |true| (8 significant bits)
    # the fp32 evaluation error: relative, plus absolute where the sum cancels
    near = np.abs(np.abs(true - want) - ulp / 2) <= 1e-5 * np.abs(true) + 2e-6
    assert np.all(ok | near), f"{int((~(ok | near)).sum())} stored values off"
    assert np.all(np.abs(held - want) <= ulp + 1e-300)
    assert (~ok).sum() <= max(2, ok.size // 1000)
    assert np.mean(held != true) > 0.9              # the rounding happened
    # fp32 data: held in fp32
    q32 = q.float().numpy()
    held32 = _held_q(orc, q32, w, win.float().numpy())
    true32 = _conv_ref(q32.astype(np.float64), w[0], win[0, 0].double().numpy())
    np.testing.assert_allclose(held32, true32, rtol=1e-6, atol=2e-6)
    assert np.all(held32 == held32.astype(np.float32))


def pin_short_conv(orc):
    """Convolution + Swish on q, k and v equals the plain recurrence on inputs
    convolved by numpy.convolve (after the caller's window of earlier rows);
    packed sequences each restart from their own window; a prefill split in
    two (the second part given the first part's last three raw rows) and a
    run of decode steps carrying the window give the same result."""
    r = _rng(47)
    T, H, d = 12, 2, 6
    q, k, v = r.normal(size=(T, H, d)), r.normal(size=(T, H, d)), r.normal(size=(T, H, d))
    la = r.uniform(-5, 0, size=(T, H, d))
    b = r.uniform(0.1, 1, size=(T, H))
    w = r.normal(size=(3, H, d, 4)) * 0.7
    win = r.normal(size=(1, 3, 3, H, d))
    S0 = r.normal(size=(1, H, d, d))
    o, S_T = orc.prefill(q, k, v, la, b, S0, conv_weight=w, conv_state=win, eps_l2=0.0)
    qc, kc, vc = (_conv_ref(x, w[i], win[0, i]) for i, x in enumerate((q, k, v)))
    o2, S2 = orc.prefill(qc, kc, vc, la, b, S0, eps_l2=0.0)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S_T, S2, rtol=1e-12, atol=1e-12)
    # packed: each sequence from its own window
    T1 = 5
    cu = np.array([0, T1, T], dtype=np.int32)
    win2 = r.normal(size=(2, 3, 3, H, d))
    S02 = r.normal(size=(2, H, d, d))
    op, Sp = orc.prefill(q, k, v, la, b, S02, cu, conv_weight=w, conv_state=win2, eps_l2=0.0)
    oa, Sa = orc.prefill(q[:T1], k[:T1], v[:T1], la[:T1], b[:T1], S02[:1], conv_weight=w,
                         conv_state=win2[:1], eps_l2=0.0)
    ob, Sb = orc.prefill(q[T1:], k[T1:], v[T1:], la[T1:], b[T1:], S02[1:], conv_weight=w,
                         conv_state=win2[1:], eps_l2=0.0)
    np.testing.assert_array_equal(op, np.concatenate([oa, ob]))
    np.testing.assert_array_equal(Sp, np.concatenate([Sa, Sb]))
    # split: the second part's window is the first part's last three raw rows
    oa, Sa = orc.prefill(q[:T1], k[:T1], v[:T1], la[:T1], b[:T1], S0, conv_weight=w,
                         conv_state=win, eps_l2=0.0)
    tail = np.stack([x[T1 - 3:T1] for x in (q, k, v)])[None]
    ob, Sb = orc.prefill(q[T1:], k[T1:], v[T1:], la[T1:], b[T1:], Sa, conv_weight=w,
                         conv_state=tail, eps_l2=0.0)
    np.testing.assert_allclose(np.concatenate([oa, ob]), o, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(Sb, S_T, rtol=1e-13, atol=1e-13)
    # decode steps carry the window
    S, cs = S0.copy(), win.copy()
    for t in range(T):
        ot, S, cs = orc.decode_step(q[t:t + 1], k[t:t + 1], v[t:t + 1], la[t:t + 1], b[t:t + 1],
                                    S, conv_weight=w, conv_state=cs, eps_l2=0.0)
        np.testing.assert_allclose(ot[0], o[t], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(S, S_T, rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(cs[0], np.stack([x[T - 3:] for x in (q, k, v)]))


ALL_PINS = [
    pin_brute_force,
    pin_overwrite,
    pin_meeting,
    pin_linear_attention,
    pin_half_life,
    pin_floor,
    pin_scalar_decay,
    pin_l2norm,
    pin_beta_logit,
    pin_split_and_decode,
    pin_gated_rmsnorm,
    pin_input_widening,
    pin_decay_logit,
    pin_short_conv_impulse,
    pin_short_conv_storage,
    pin_short_conv,
]
