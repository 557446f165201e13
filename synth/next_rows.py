"""Seeded inputs for the decode-loop pieces around the verify step: ragged
draft counts, candidate trees and token contexts. Generation only; no verify,
lookup or commit arithmetic lives here."""
from __future__ import annotations

import numpy as np
import torch

from .workloads import _storage, zipf_rank_bias

# Sizes the benchmark reports these pieces on.
NEXT_ROWS = {
    # per-sequence draft counts on the B=256, K=8, V=151936 bf16 workload
    "ragged": dict(base="c4", lens=("uniform", 0, 8)),
    # greedy tree verify: 64 trees of 32 nodes over V=128256 bf16 rows
    "tree": dict(B=64, N=32, V=128256, dtype="bf16", sigma_t=4.0, zipf_s=1.05, p_follow=0.6),
    # prompt lookup over 256 contexts of up to 16384 tokens (vocab 32000)
    "lookup": dict(B=256, L_max=16384, vocab=32000, max_ngram=3, n_drafts=8, copy_prob=0.3),
    # commit of K+1 = 9 tokens per sequence into 256 contexts of 16384 slots
    "commit": dict(B=256, L_max=16384, K=8),
}


def make_draft_lens(B: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    """Per-sequence draft counts, uniform over 0..K, seeded; the first four
    sequences take 0, K, 1 and K - 1 so both ends occur."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, K + 1, B).astype(np.int32)
    lens[:4] = [0, K, min(1, K), max(K - 1, 0)][:min(4, B)]
    return torch.from_numpy(lens).to(device)


def make_tree_case(B: int, N: int, V: int, dtype: str = "bf16", sigma_t: float = 4.0,
                   zipf_s: float = 1.05, p_follow: float = 0.6, seed: int = 0, device="cpu"):
    """B candidate trees of N nodes: target rows N(0, sigma_t^2) + Zipf rank
    bias (one row per node), node 0 the root; node i hangs under a uniformly
    drawn earlier node and carries its parent's top token with probability
    p_follow (a drafter that often agrees), else a uniform token.
    Returns (target [B, N, V], tokens [B, N] int32, parents [B, N] int32)."""
    g = torch.Generator(device=device).manual_seed(seed)
    bias = zipf_rank_bias(V, zipf_s, seed + 7919, device)
    target = _storage(torch.randn(B, N, V, generator=g, device=device) * sigma_t + bias, dtype)
    top = target.float().argmax(dim=2).cpu().numpy()  # first maximum of the stored values
    rng = np.random.default_rng(seed)
    parents = np.full((B, N), -1, np.int32)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for i in range(1, N):
            parents[b, i] = rng.integers(0, i)
            tokens[b, i] = top[b, parents[b, i]] if rng.random() < p_follow else rng.integers(0, V)
    return (target.contiguous(), torch.from_numpy(tokens).to(device),
            torch.from_numpy(parents).to(device))


def make_contexts(B: int, L_max: int, vocab: int, seed: int, copy_prob: float = 0.3):
    """Token contexts that partly copy earlier spans of themselves (as an
    answer quotes its prompt), lengths uniform over 0..L_max with 0, 1, 2 and
    L_max among the first four. Returns (tokens [B, L_max], lengths [B]) as
    int32 numpy arrays."""
    rng = np.random.default_rng(seed)
    tok = rng.integers(0, vocab, (B, L_max)).astype(np.int32)
    for b in range(B):
        i = 8
        while i < L_max:
            if rng.random() < copy_prob:
                src = int(rng.integers(0, i - 4))
                n = int(rng.integers(2, 24))
                span = tok[b, src:src + n]
                tok[b, i:i + len(span)] = span[:max(0, min(len(span), L_max - i))]
                i += n
            else:
                i += int(rng.integers(1, 16))
    lens = rng.integers(0, L_max + 1, B).astype(np.int32)
    lens[:min(4, B)] = [0, 1, 2, L_max][:min(4, B)]
    return tok, lens
