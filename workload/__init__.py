"""Seeded synthetic inputs for the DSpark draft + verify step.

This module is shared by the CUDA path's tests and bench and by the oracle's
tests.  It holds only random tensors and the workload tables (SPS capacity
curves, STS temperatures); none of the method's arithmetic.

Five workloads stand in for the trained draft model and the benchmark suites
the pages measure on (GSM8K, MATH500, HumanEval, ...), which are not
available: their logits, hidden states and weights are drawn from the
distributions below with Qwen3-8B shapes.

  tiny   B=4,   V=1024,   r=32,  d=64,   fp32 weights, SPS 1000/(10+0.5n), n<=32
  b1     B=1,   V=151936, r=256, d=4096, bf16 weights, scheduler off (K=7)
  b64    B=64,  V=151936, r=256, d=4096, bf16 weights, stepped SPS, n<=1024
  b256   B=256, V=129280, r=128, d=4096, bf16 weights, bf16 target, sawtooth SPS
  b512   B=512, V=151936, r=256, d=4096, bf16 weights, bf16 target, async, 16 steps
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

GAMMA = 7


def sps_tiny(n: int) -> float:
    return 1000.0 / (10.0 + 0.5 * n)


def sps_stepped(n: int) -> float:
    return 1000.0 / (8.0 + 0.02 * 64 * math.ceil(n / 64))


def sps_sawtooth(n: int) -> float:
    base = 1000.0 / (6.0 + 0.004 * n)
    if n > 128:
        m, rem = divmod(n - 1, 128)
        if m >= 1 and rem < 32:
            return base * (1.0 - 0.15 * (1.0 - rem / 32.0))
    return base


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    V: int
    r: int
    d: int
    seed: int
    w_dtype: torch.dtype
    target_dtype: torch.dtype
    w_std: float
    target_sigma: float
    boost: tuple             # mode boost per draft position k = 1..gamma
    mode: int                # 0 off, 1 sync, 2 async
    sps_len: int
    sps_fn: object = field(compare=False, default=None)
    steps: int = 1
    gamma: int = GAMMA
    u_std: float = 2.0
    conf_std: float = 0.05
    conf_bias: float = 0.5
    tau: float = 1.0

    def sps_table(self) -> torch.Tensor:
        return torch.tensor([self.sps_fn(n) for n in range(1, self.sps_len + 1)], dtype=torch.float32)

    def temperatures(self) -> torch.Tensor:
        return torch.tensor([1.0 + 0.1 * k for k in range(1, self.gamma + 1)], dtype=torch.float32)


_DECAY = tuple(float(11 - k) for k in range(1, GAMMA + 1))   # +10 at k=1 ... +4 at k=7

WORKLOADS = {
    "tiny": Workload("tiny", B=4, V=1024, r=32, d=64, seed=0, w_dtype=torch.float32,
                     target_dtype=torch.float32, w_std=0.3, target_sigma=0.5,
                     boost=(8.0,) * GAMMA, mode=1, sps_len=32, sps_fn=sps_tiny),
    "b1": Workload("b1", B=1, V=151936, r=256, d=4096, seed=1, w_dtype=torch.bfloat16,
                   target_dtype=torch.float32, w_std=0.02, target_sigma=0.5,
                   boost=(8.0,) * GAMMA, mode=0, sps_len=8, sps_fn=sps_stepped),
    "b64": Workload("b64", B=64, V=151936, r=256, d=4096, seed=2, w_dtype=torch.bfloat16,
                    target_dtype=torch.float32, w_std=0.02, target_sigma=0.5,
                    boost=_DECAY, mode=1, sps_len=1024, sps_fn=sps_stepped),
    "b256": Workload("b256", B=256, V=129280, r=128, d=4096, seed=3, w_dtype=torch.bfloat16,
                     target_dtype=torch.bfloat16, w_std=0.02, target_sigma=0.7,
                     boost=_DECAY, mode=1, sps_len=2048, sps_fn=sps_sawtooth),
    "b512": Workload("b512", B=512, V=151936, r=256, d=4096, seed=4, w_dtype=torch.bfloat16,
                     target_dtype=torch.bfloat16, w_std=0.02, target_sigma=0.5,
                     boost=_DECAY, mode=2, sps_len=4096, sps_fn=sps_stepped, steps=16),
}


def custom(base: str = "tiny", **kw) -> Workload:
    """A workload like `base` with some fields replaced (small parity cases)."""
    w = WORKLOADS[base]
    d = {f: getattr(w, f) for f in w.__dataclass_fields__}
    d.update(kw)
    if "gamma" in kw and "boost" not in kw:
        d["boost"] = (w.boost + (w.boost[-1],) * kw["gamma"])[: kw["gamma"]]
    if "sps_len" not in kw:       # the capacity table must cover R + B*gamma tokens
        d["sps_len"] = max(w.sps_len, d["B"] * (d["gamma"] + 1))
    return Workload(**d)


def _gen(device, *seed_parts) -> torch.Generator:
    g = torch.Generator(device=device)
    s = 0
    for p in seed_parts:
        s = (s * 1_000_003 + int(p)) % (2 ** 62)
    g.manual_seed(s)
    return g


def _boosted_logits(B, rows, V, std, boosts, g, device):
    """N(0, std^2) logits with +boosts[k] at one uniform 'mode' token per (b, k)."""
    x = torch.randn((B, rows, V), generator=g, device=device, dtype=torch.float32) * std
    mode = torch.randint(0, V, (B, rows), generator=g, device=device)
    add = torch.tensor(boosts, dtype=torch.float32, device=device).expand(B, rows)
    x.scatter_add_(2, mode.unsqueeze(-1), add.unsqueeze(-1).contiguous())
    return x


def draft_weights(w: Workload, device="cpu") -> dict:
    """W1 [V,r] and W2 [r,V] alone, the same values weights() draws."""
    g = _gen(device, w.seed, 1)
    W1 = (torch.randn((w.V, w.r), generator=g, device=device) * w.w_std).to(w.w_dtype)
    W2 = (torch.randn((w.r, w.V), generator=g, device=device) * w.w_std).to(w.w_dtype)
    return dict(W1=W1.contiguous(), W2=W2.contiguous())


def weights(w: Workload, device="cpu") -> dict:
    """Draft-head parameters: W1 [V,r], W2 [r,V], emb [V,d], w_c [2d], b_c."""
    g = _gen(device, w.seed, 1)
    W1 = (torch.randn((w.V, w.r), generator=g, device=device) * w.w_std).to(w.w_dtype)
    W2 = (torch.randn((w.r, w.V), generator=g, device=device) * w.w_std).to(w.w_dtype)
    emb = torch.randn((w.V, w.d), generator=g, device=device, dtype=torch.float32)
    w_c = torch.randn((2 * w.d,), generator=g, device=device, dtype=torch.float32) * w.conf_std
    return dict(W1=W1.contiguous(), W2=W2.contiguous(), emb=emb, w_c=w_c, b_c=w.conf_bias,
                T=w.temperatures().to(device), sps=w.sps_table().to(device))


def step_inputs(w: Workload, step: int = 0, device="cpu", anchor=None) -> dict:
    """Per-step activations: U [B,gamma,V] fp32, target [B,gamma+1,V], h [B,gamma,d], anchor [B].

    Target rows 0..gamma-1 are U plus N(0, sigma^2); row gamma (the bonus
    distribution) is an independent boosted draw plus the same perturbation."""
    g = _gen(device, w.seed, 2, step)
    U = _boosted_logits(w.B, w.gamma, w.V, w.u_std, w.boost, g, device)
    extra = _boosted_logits(w.B, 1, w.V, w.u_std, (w.boost[-1],), g, device)
    target = torch.cat([U, extra], dim=1)
    target.add_(torch.randn(target.shape, generator=g, device=device) * w.target_sigma)
    target = target.to(w.target_dtype)
    h = torch.randn((w.B, w.gamma, w.d), generator=g, device=device, dtype=torch.float32)
    if anchor is None:
        anchor = torch.randint(0, w.V, (w.B,), generator=g, device=device)
    return dict(U=U, target=target.contiguous(), h=h, anchor=anchor.to(torch.int32))


def inputs(w: Workload, step: int = 0, device="cpu") -> dict:
    d = weights(w, device)
    d.update(step_inputs(w, step, device))
    return d


def sts_validation(N: int, gamma: int = GAMMA, seed: int = 0, T_true=None, device="cpu"):
    """A synthetic validation set for the STS fit: raw confidence scores
    [N, gamma] fp32 (the logits of c_k) and accepted lengths [N] int32.

    Scores s_k ~ N(3 - 0.3k, 2.5^2), confidence falling along the block.  The
    target accepts draft k with probability 1 / (1 + exp(-s_k / T*_k)), left
    to right until its first rejection, so the probability that prefix k is
    accepted is the STS survival at T = T*, and the raw confidences are
    over-confident wherever T*_k > 1.  T* defaults to the workloads' inference
    temperatures 1 + 0.1k."""
    if T_true is None:
        T_true = [1.0 + 0.1 * k for k in range(1, gamma + 1)]
    T_true = torch.tensor(T_true, dtype=torch.float64, device=device)
    assert T_true.numel() == gamma
    g = _gen(device, seed, 7, N, gamma)
    mean = torch.tensor([3.0 - 0.3 * k for k in range(1, gamma + 1)], dtype=torch.float64, device=device)
    score = (torch.randn((N, gamma), generator=g, device=device, dtype=torch.float64) * 2.5 + mean).float()
    p_acc = torch.sigmoid(score.double() / T_true)
    ok = torch.rand((N, gamma), generator=g, device=device, dtype=torch.float64) < p_acc
    first_rej = torch.where(ok.all(dim=1), torch.full((N,), gamma, device=device),
                            torch.argmin(ok.to(torch.int8), dim=1))
    return score.contiguous(), first_rej.to(torch.int32).contiguous()


# The STS fit measured by the benchmark: a validation set of 2^20 drafted
# blocks, 256 candidate temperatures evenly spaced on [0.25, 4], 15 bins.
STS_FIT = dict(N=1 << 20, gamma=GAMMA, G=256, M=15, lo=0.25, hi=4.0, seed=0)


def sts_grid(G: int, lo: float = 0.25, hi: float = 4.0) -> torch.Tensor:
    return torch.linspace(lo, hi, G, dtype=torch.float32)


def rnn_head(w: Workload, device="cpu") -> dict:
    """Parameters of the RNN draft head for workload w (rank r): input
    embedding E [V,r] ~ N(0,1), W_ih and W_hh [3r,r] and the biases [3r]
    ~ U(-1/sqrt(r), 1/sqrt(r)) (the usual GRU initialisation), s0 [r] ~
    N(0, 0.5^2).  Matrices in bf16 (the head's weight dtype), vectors fp32."""
    g = _gen(device, w.seed, 5)
    r = w.r
    a = 1.0 / math.sqrt(r)

    def unif(shape):
        return (torch.rand(shape, generator=g, device=device) * 2 - 1) * a

    return dict(E=torch.randn((w.V, r), generator=g, device=device).to(torch.bfloat16).contiguous(),
                W_ih=unif((3 * r, r)).to(torch.bfloat16).contiguous(),
                W_hh=unif((3 * r, r)).to(torch.bfloat16).contiguous(),
                b_ih=unif((3 * r,)).float().contiguous(), b_hh=unif((3 * r,)).float().contiguous(),
                s0=(torch.randn((r,), generator=g, device=device) * 0.5).float().contiguous())
