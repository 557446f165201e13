"""Comparison of the CUDA path's outputs with the oracle's (test infrastructure).

The GPU computes in float32 and the oracle in float64, so a decision that
lies within rounding of its threshold may legitimately differ. Such
sequences are near-ties; they are counted, reported and excluded, and every
other sequence must match exactly (tokens and accepted counts).

Near-tie bands:
  accept test   |u * P_d(x) - P_t(x)| < ACCEPT_TIE_REL * P_d(x) at any tested
                position (the band the verify step's specification gives);
  final draw    the draw's target t lies within DRAW_TIE_ABS of an edge of the
                chosen token's cumulative interval, in probability units (the
                pages' distributions sum to one). The band is set from a
                measurement, not a model: the kernel reports its own distances
                from t to both edges of the token it chose, and over every
                sample sequence of the GPU parity suite (about 10^4 sequences:
                c1-c4, all cluster sizes, temperatures 0.05-10, misaligned and
                ragged rows) they differ from the oracle's by at most
                2.85e-7; the band is 1.75 times that. It is absolute, not relative
                to the draw's total mass S_r: the error comes from the rows'
                probabilities (each with its own float32 normaliser), so it
                does not shrink with the residual's mass.
"""
from __future__ import annotations

import numpy as np

ACCEPT_TIE_REL = 1e-6
DRAW_TIE_ABS = 5e-7
PROB_RTOL = 1e-5


def near_ties(ref: dict, accept_rel: float = ACCEPT_TIE_REL, draw_abs: float = DRAW_TIE_ABS,
              draw_scale=None) -> np.ndarray:
    """Boolean [B]: the oracle's decisions for this sequence sit within the
    float32 rounding band of a threshold. draw_scale optionally widens the
    draw band per sequence (e.g. for logits computed by a GEMM)."""
    tie = ref["accept_margin"] < accept_rel
    band = draw_abs if draw_scale is None else draw_abs * np.asarray(draw_scale)
    tie |= ref["draw_margin"] < band
    return tie


def compare(gpu_tokens: np.ndarray, gpu_n: np.ndarray, ref: dict, ties=None) -> dict:
    """Exact comparison outside the near-ties. Returns counts and the first
    mismatching sequences."""
    gpu_tokens = np.asarray(gpu_tokens)
    gpu_n = np.asarray(gpu_n)
    if ties is None:
        ties = near_ties(ref)
    B = gpu_n.shape[0]
    same_n = gpu_n == ref["n_accepted"]
    same_t = (gpu_tokens == ref["tokens"]).all(axis=1)
    ok = same_n & same_t
    bad = np.flatnonzero(~ok & ~ties)
    return {
        "sequences": int(B),
        "near_ties": int(ties.sum()),
        "near_tie_mismatches": int((~ok & ties).sum()),
        "mismatches": int(bad.size),
        "first_mismatches": [
            {"b": int(b), "gpu_n": int(gpu_n[b]), "ref_n": int(ref["n_accepted"][b]),
             "gpu_tokens": gpu_tokens[b].tolist(), "ref_tokens": ref["tokens"][b].tolist(),
             "accept_margin": float(ref["accept_margin"][b]),
             "draw_margin": float(ref["draw_margin"][b])}
            for b in bad[:5]],
    }


def compare_probabilities(gpu_p: np.ndarray, ref_p: np.ndarray, n_accepted: np.ndarray,
                          rtol: float = PROB_RTOL) -> float:
    """Largest relative error of the exposed P(x_i) over the tested positions
    i <= min(n_accepted, K-1) of valid sample sequences."""
    K = ref_p.shape[1]
    worst = 0.0
    for b in range(ref_p.shape[0]):
        n = int(n_accepted[b])
        if n < 0:
            continue
        for i in range(min(n, K - 1) + 1):
            r = ref_p[b, i]
            if not np.isfinite(r) or r == 0.0:
                continue
            worst = max(worst, abs(float(gpu_p[b, i]) - r) / r)
    return worst
