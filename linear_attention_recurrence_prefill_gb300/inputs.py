"""Seeded synthetic inputs for the KDA layer core.

This module only draws random numbers in the shapes and distributions of the
five workloads the library is measured on; it holds none of the method's
arithmetic and is shared by the tests, the benchmark and the smoke check.
The CUDA path and the CPU oracle both receive exactly the tensors made here.

Workloads (all d_k = d_v = d):

* ``tiny``     H=2, T=128, d=32, fp32.  q, k ~ N(0,1) then unit-normalised per
               head; v ~ N(0,1); log alpha = -5*sigmoid(N(0,1)) per token and
               key channel; beta = sigmoid(N(0,1)) per token and head; S0 = 0;
               seed 0.
* ``k3``       H=96, T=4096, d=128.  q, k, v bf16 (q, k unit-normalised);
               log alpha fp32 = -5*sigmoid(N(0,1.5)); beta bf16 =
               sigmoid(N(0,1)); S0 ~ N(0, 0.02) fp32; gate logits N(0,1) bf16
               (RMSNorm weight 1); seed 1.
* ``varlen``   8 packed sequences, lengths uniform in [1024, 16384] (seed 2),
               H=96, d=128, bf16, distributions as ``k3``, S0 = 0 per sequence.
* ``decode``   64 sequences, one token per step, H=96, d=128, bf16 q/k/v/beta,
               fp32 log alpha, fp32 state ~ N(0, 0.05); 256 steps pre-drawn;
               seed 3.
* ``extreme``  H=96, T=262144, d=128, bf16; in every head half of the key
               channels (a seeded random half) have log alpha at the floor -5
               and the other half at -1e-4; beta = 1 on every 7th token
               (t mod 7 == 0) and sigmoid(N(0,1)) otherwise; unit keys that
               repeat every 64 tokens; q ~ N(0,1) unit-normalised, v ~ N(0,1),
               S0 = 0, gate as ``k3``; seed 4.

The prologue from raw projections (``prologue_params``, ``conv_window``) draws
synthetic parameters for the optional steps before the recurrence: short-
convolution taps [3 (q, k, v), H, d, 4] ~ N(0, 0.5), decay logits ~ N(0, 1.5),
per-head decay scales and per-channel decay biases either "wide" (A_h ~
U[0.5, 2], b ~ N(0, 0.5)) or "workload" (A_h = 1, b = 0: the bounded sigmoid
then gives the workloads' own log-alpha distribution -5 sigmoid(N(0, 1.5))),
and windows of raw rows before each sequence ~ N(0, 1).

"N(0, s)" is read as mean 0 and standard deviation s.  Draw order inside one
workload: (lengths,) q, k, v, log-alpha noise, beta noise, gate noise, S0.
Large tensors are drawn in token slabs so that the peak transient memory stays
bounded; the slab size is part of the recipe (it fixes the random stream).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

SLAB = 16384  # tokens per draw


@dataclass
class PrefillInputs:
    q: torch.Tensor            # [T, H, d]
    k: torch.Tensor            # [T, H, d]
    v: torch.Tensor            # [T, H, d]
    log_alpha: torch.Tensor    # [T, H, d] fp32
    beta: torch.Tensor         # [T, H]
    S0: torch.Tensor | None    # [N, H, d, d] fp32 or None (= zeros)
    gate: torch.Tensor | None  # [T, H, d] or None
    cu_seqlens: torch.Tensor | None  # [N+1] int32 or None (N = 1)
    N: int
    chunk: int
    name: str
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return self.q.shape[0]

    @property
    def H(self) -> int:
        return self.q.shape[1]

    @property
    def d(self) -> int:
        return self.q.shape[2]


@dataclass
class DecodeInputs:
    q: torch.Tensor          # [steps, N, H, d]
    k: torch.Tensor
    v: torch.Tensor
    log_alpha: torch.Tensor  # [steps, N, H, d] fp32
    beta: torch.Tensor       # [steps, N, H]
    S: torch.Tensor          # [N, H, d, d] fp32 (initial state)
    name: str = "decode"


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, g, device, std: float = 1.0) -> torch.Tensor:
    """N(0, std) in fp32, drawn in slabs along dim 0."""
    out = torch.empty(shape, dtype=torch.float32, device=device)
    for s in range(0, shape[0], SLAB):
        e = min(shape[0], s + SLAB)
        out[s:e] = torch.randn((e - s, *shape[1:]), generator=g, device=device,
                               dtype=torch.float32)
    if std != 1.0:
        out.mul_(std)
    return out


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    """Scale each last-dim vector to unit Euclidean length (input recipe)."""
    return x / torch.linalg.vector_norm(x, dim=-1, keepdim=True).clamp_min(1e-30)


def _k3_like(T: int, H: int, d: int, dtype, g, device, *, with_s0: bool,
             s0_std: float, N: int, la_std: float = 1.5):
    q = _unit_rows(_randn((T, H, d), g, device)).to(dtype)
    k = _unit_rows(_randn((T, H, d), g, device)).to(dtype)
    v = _randn((T, H, d), g, device).to(dtype)
    la = _randn((T, H, d), g, device, std=la_std)
    la = (-5.0 * torch.sigmoid(la)).to(torch.float32)
    beta = torch.sigmoid(_randn((T, H), g, device)).to(dtype)
    gate = _randn((T, H, d), g, device).to(dtype)
    S0 = _randn((N * H, d, d), g, device, std=s0_std).reshape(N, H, d, d) if with_s0 else None
    return q, k, v, la, beta, gate, S0


def tiny(device="cpu", *, seed: int = 0, H: int = 2, T: int = 128, d: int = 32) -> PrefillInputs:
    g = _gen(seed, device)
    q = _unit_rows(_randn((T, H, d), g, device))
    k = _unit_rows(_randn((T, H, d), g, device))
    v = _randn((T, H, d), g, device)
    la = -5.0 * torch.sigmoid(_randn((T, H, d), g, device))
    beta = torch.sigmoid(_randn((T, H), g, device))
    return PrefillInputs(q, k, v, la, beta, None, None, None, 1, 16, "tiny",
                         {"dtype": "f32"})


def k3(device="cpu", *, seed: int = 1, H: int = 96, T: int = 4096, d: int = 128,
       dtype=torch.bfloat16) -> PrefillInputs:
    g = _gen(seed, device)
    q, k, v, la, beta, gate, S0 = _k3_like(T, H, d, dtype, g, device, with_s0=True,
                                           s0_std=0.02, N=1)
    return PrefillInputs(q, k, v, la, beta, S0, gate, None, 1, 64, "k3",
                         {"dtype": "bf16" if dtype == torch.bfloat16 else "f32"})


def varlen_lengths(seed: int = 2, n: int = 8, lo: int = 1024, hi: int = 16384) -> list[int]:
    g = _gen(seed, "cpu")
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def varlen(device="cpu", *, seed: int = 2, H: int = 96, d: int = 128,
           lengths: list[int] | None = None, dtype=torch.bfloat16) -> PrefillInputs:
    lens = lengths if lengths is not None else varlen_lengths(seed)
    T = sum(lens)
    g = _gen(seed + 1000, device)
    q, k, v, la, beta, gate, _ = _k3_like(T, H, d, dtype, g, device, with_s0=False,
                                          s0_std=0.0, N=len(lens))
    cu = torch.zeros(len(lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    return PrefillInputs(q, k, v, la, beta, None, gate, cu.to(device), len(lens), 64,
                         "varlen", {"lengths": lens, "dtype": "bf16"})


def decode(device="cpu", *, seed: int = 3, N: int = 64, H: int = 96, d: int = 128,
           steps: int = 256, dtype=torch.bfloat16) -> DecodeInputs:
    g = _gen(seed, device)
    shp = (steps, N, H, d)
    q = _unit_rows(_randn(shp, g, device)).to(dtype)
    k = _unit_rows(_randn(shp, g, device)).to(dtype)
    v = _randn(shp, g, device).to(dtype)
    la = (-5.0 * torch.sigmoid(_randn(shp, g, device, std=1.5))).to(torch.float32)
    beta = torch.sigmoid(_randn((steps, N, H), g, device)).to(dtype)
    S = _randn((N * H, d, d), g, device, std=0.05).reshape(N, H, d, d)
    return DecodeInputs(q, k, v, la, beta, S)


def extreme(device="cpu", *, seed: int = 4, H: int = 96, T: int = 262144, d: int = 128,
            period: int = 64, dtype=torch.bfloat16) -> PrefillInputs:
    g = _gen(seed, device)
    q = _unit_rows(_randn((T, H, d), g, device)).to(dtype)
    kb = _unit_rows(_randn((period, H, d), g, device))
    reps = (T + period - 1) // period
    k = kb.repeat(reps, 1, 1)[:T].to(dtype).contiguous()
    v = _randn((T, H, d), g, device).to(dtype)
    # which half of each head's channels sits at the floor
    perm = torch.argsort(torch.rand((H, d), generator=g, device=device), dim=1)
    floor_mask = torch.zeros((H, d), dtype=torch.bool, device=device)
    floor_mask.scatter_(1, perm[:, : d // 2], True)
    row = torch.where(floor_mask, torch.tensor(-5.0, device=device),
                      torch.tensor(-1e-4, device=device)).to(torch.float32)
    la = row.unsqueeze(0).expand(T, H, d).contiguous()
    beta = torch.sigmoid(_randn((T, H), g, device))
    t = torch.arange(T, device=device)
    beta[t % 7 == 0] = 1.0
    beta = beta.to(dtype)
    gate = _randn((T, H, d), g, device).to(dtype)
    return PrefillInputs(q, k, v, la, beta, None, gate, None, 1, 64, "extreme",
                         {"dtype": "bf16", "period": period})


@dataclass
class PrologueParams:
    conv_weight: torch.Tensor   # [3, H, d, 4] fp32 (q, k, v taps, oldest row first)
    decay_scale: torch.Tensor   # [H] fp32
    decay_bias: torch.Tensor    # [H, d] fp32


def prologue_params(device="cpu", *, H: int, d: int = 128, seed: int = 5,
                    decay: str = "wide") -> PrologueParams:
    """decay "wide": A_h ~ U[0.5, 2], b ~ N(0, 0.5) (exercises the scale and the
    bias); "workload": A_h = 1, b = 0, which with logits ~ N(0, 1.5) gives the
    workloads' own log-alpha distribution -5 sigmoid(N(0, 1.5))."""
    g = _gen(seed, "cpu")
    w = torch.randn((3, H, d, 4), generator=g) * 0.5
    A = 0.5 + 1.5 * torch.rand((H,), generator=g)
    b = torch.randn((H, d), generator=g) * 0.5
    if decay == "workload":
        A, b = torch.ones_like(A), torch.zeros_like(b)
    elif decay != "wide":
        raise ValueError(f"decay: 'wide' or 'workload', not {decay!r}")
    return PrologueParams(w.to(device), A.to(device), b.to(device))


def decay_logits(shape, device="cpu", *, seed: int = 6) -> torch.Tensor:
    """Decay logits z ~ N(0, 1.5), fp32."""
    return _randn(tuple(shape), _gen(seed, device), device, std=1.5)


def conv_window(N: int, H: int, d: int = 128, device="cpu", *, seed: int = 7,
                dtype=torch.bfloat16) -> torch.Tensor:
    """Raw q, k, v rows of the 3 tokens before each sequence, [N, 3, 3, H, d]."""
    return torch.randn((N, 3, 3, H, d), generator=_gen(seed, "cpu")).to(dtype).to(device)


WORKLOADS = {
    "tiny": tiny,
    "k3": k3,
    "varlen": varlen,
    "extreme": extreme,
}
