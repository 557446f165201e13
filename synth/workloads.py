"""Workload definitions and seeded generators.

Recipe (the pages run no verify-step benchmark of their own, so these
distributions stand in for real model logits):

* target logits ~ N(0, sigma_t^2) + a Zipf rank bias, bias_v = -s * ln(1 + pi(v))
  for one seeded permutation pi of the vocabulary per case (shared by all rows);
* draft logits = a * target + N(0, tau^2), tau either fixed or drawn per sequence;
* draft tokens: sample-mode sequences draw x_i from softmax(draft_i / T) (the
  drafter's own sampling, which the sampling rule presupposes); greedy-mode
  sequences take the draft argmax, as a greedy drafter does;
* logits are rounded to the storage dtype (bf16: round to nearest even) before
  the draft tokens are drawn, so the tokens follow the distribution the
  verifier actually sees;
* LM-head case: hidden ~ N(0, 1), W ~ N(0, 0.02^2), both bf16; the draft logits
  of positions 0..K-1 are hidden . W + N(0, 1), rounded to bf16.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

# Workloads: c1..c5 are the five configurations of the verify step.
WORKLOADS = {
    "c1": dict(B=1, K=4, V=1000, dtype="f32", sigma_t=3.0, zipf_s=1.1, draft_scale=1.0,
               tau=1.0, T=1.0, modes="both"),
    "c2": dict(B=8, K=5, V=32000, dtype="f32", sigma_t=3.0, zipf_s=1.1, draft_scale=1.0,
               tau=(0.3, 1.0, 3.0), T=1.0, modes="sample"),
    "c3": dict(B=64, K=4, V=128256, dtype="bf16", sigma_t=4.0, zipf_s=1.05, draft_scale=0.8,
               tau=1.5, T=0.8, modes="half"),
    "c4": dict(B=256, K=8, V=151936, dtype="bf16", sigma_t=4.0, zipf_s=1.1, draft_scale=1.0,
               tau=("uniform", 0.2, 3.0), T=1.0, modes="sample"),
    "c5": dict(B=32, K=5, V=128256, d=4096, dtype="bf16", w_sigma=0.02, tau=1.0, T=1.0,
               modes="sample"),
}

GREEDY, SAMPLE = 0, 1


@dataclass
class LogitsCase:
    target: torch.Tensor        # [B, K+1, V], float32 or bfloat16
    draft: torch.Tensor         # [B, K, V], same dtype
    tokens: torch.Tensor        # [B, K] int32
    modes: torch.Tensor         # [B] int32, 0 greedy / 1 sample
    temperature: float

    @property
    def shape(self):
        B, K1, V = self.target.shape
        return B, K1 - 1, V


@dataclass
class LMHeadCase:
    hidden: torch.Tensor        # [B, K+1, d] bf16
    W: torch.Tensor             # [d, V] bf16
    draft: torch.Tensor         # [B, K, V] bf16
    tokens: torch.Tensor        # [B, K] int32
    modes: torch.Tensor         # [B] int32
    temperature: float


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def zipf_rank_bias(V: int, s: float, seed: int, device="cpu") -> torch.Tensor:
    """bias_v = -s * ln(1 + pi(v)) with pi a seeded permutation of range(V)."""
    perm = torch.randperm(V, generator=_gen(seed, "cpu"))
    return (-s * torch.log1p(perm.to(torch.float64))).to(torch.float32).to(device)


def _storage(x: torch.Tensor, dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if dtype == "bf16" else x.to(torch.float32)


def _draw_tokens(draft: torch.Tensor, modes: torch.Tensor, T: float, g) -> torch.Tensor:
    B, K, V = draft.shape
    probs = torch.softmax(draft.float().reshape(B * K, V) / T, dim=-1)
    sampled = torch.multinomial(probs, 1, generator=g).reshape(B, K)
    greedy = draft.float().argmax(dim=-1)
    m = modes.to(draft.device).reshape(B, 1).bool()
    return torch.where(m, sampled, greedy).to(torch.int32)


def make_modes(B: int, modes) -> torch.Tensor:
    if isinstance(modes, torch.Tensor):
        return modes.to(torch.int32)
    if modes in ("sample", SAMPLE):
        return torch.ones(B, dtype=torch.int32)
    if modes in ("greedy", GREEDY):
        return torch.zeros(B, dtype=torch.int32)
    if modes == "half":  # first half greedy, second half sample
        m = torch.ones(B, dtype=torch.int32)
        m[: B // 2] = 0
        return m
    raise ValueError(f"unknown modes {modes!r}")


def make_logits_case(B: int, K: int, V: int, dtype: str = "f32", sigma_t: float = 3.0,
                     zipf_s: float = 1.1, draft_scale: float = 1.0, tau=1.0, T: float = 1.0,
                     modes="sample", seed: int = 0, device="cpu") -> LogitsCase:
    """Seeded logits case with the recipe in the module docstring."""
    g = _gen(seed, device)
    bias = zipf_rank_bias(V, zipf_s, seed + 7919, device)
    target = torch.randn(B, K + 1, V, generator=g, device=device) * sigma_t + bias
    if isinstance(tau, tuple) and tau and tau[0] == "uniform":
        lo, hi = tau[1], tau[2]
        taus = lo + (hi - lo) * torch.rand(B, 1, 1, generator=g, device=device)
    else:
        taus = torch.full((B, 1, 1), float(tau), device=device)
    draft = draft_scale * target[:, :K] + torch.randn(B, K, V, generator=g, device=device) * taus
    target = _storage(target, dtype)
    draft = _storage(draft, dtype)
    m = make_modes(B, modes).to(device)
    tokens = _draw_tokens(draft, m, T, g)
    return LogitsCase(target.contiguous(), draft.contiguous(), tokens.contiguous(), m, float(T))


def make_workload(name: str, seed: int = 0, device="cpu", tau=None, modes=None, B=None):
    """The named workload (c1..c4) as a LogitsCase; c5 as an LMHeadCase.

    c2 sweeps tau over (0.3, 1.0, 3.0): pass tau= to pick one (default 1.0).
    c1 runs in both modes: pass modes= (default sample)."""
    w = dict(WORKLOADS[name])
    if name == "c5":
        return make_lmhead_case(B=B or w["B"], K=w["K"], V=w["V"], d=w["d"], w_sigma=w["w_sigma"],
                                tau=w["tau"], T=w["T"], seed=seed, device=device)
    if name == "c2":
        w["tau"] = 1.0 if tau is None else tau
    elif tau is not None:
        w["tau"] = tau
    if w["modes"] == "both":
        w["modes"] = "sample"
    if modes is not None:
        w["modes"] = modes
    if B is not None:
        w["B"] = B
    return make_logits_case(B=w["B"], K=w["K"], V=w["V"], dtype=w["dtype"], sigma_t=w["sigma_t"],
                            zipf_s=w["zipf_s"], draft_scale=w["draft_scale"], tau=w["tau"], T=w["T"],
                            modes=w["modes"], seed=seed, device=device)


def make_lmhead_case(B: int, K: int, V: int, d: int, w_sigma: float = 0.02, tau: float = 1.0,
                     T: float = 1.0, modes="sample", seed: int = 0, device="cpu") -> LMHeadCase:
    g = _gen(seed, device)
    hidden = torch.randn(B, K + 1, d, generator=g, device=device).to(torch.bfloat16)
    W = (torch.randn(d, V, generator=g, device=device) * w_sigma).to(torch.bfloat16)
    # The drafter: the target's own head on the first K positions, plus noise.
    base = (hidden[:, :K].float().reshape(B * K, d) @ W.float()).reshape(B, K, V)
    draft = (base + torch.randn(B, K, V, generator=g, device=device) * tau).to(torch.bfloat16)
    m = make_modes(B, modes).to(device)
    tokens = _draw_tokens(draft, m, T, g)
    return LMHeadCase(hidden.contiguous(), W.contiguous(), draft.contiguous(), tokens.contiguous(),
                      m, float(T))


def to_numpy_logits(x: torch.Tensor):
    """CPU numpy view for the oracle: float32 stays float32, bf16 becomes raw uint16 bits."""
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view("uint16")
    return x.numpy()
