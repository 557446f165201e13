"""The residual-fallback path of the final draw, on the GPU, in both kernels.

After a rejection the draw is from norm(max(0, P_t - P_d)) ("Speculative
decoding" (leoniemonigatti.com blog), section "Rejection sampling"). In
exact arithmetic that residual has positive mass whenever a draft token is
rejected; in float32 it can sum to zero, and the kernel then draws from P_t
of the same row instead and sets SV_FLAG_RESIDUAL_FALLBACK. This test builds
sequences that take that path on purpose:

  - K = 1, fp32 rows of V = 2048 (two CTAs per sequence hold one 4 KB chunk
    of each row); target row 0 equals draft row 0 except at the draft token
    x = 0, whose target logit is lower by delta = 4e-5, so that
    P_t(x) / P_d(x) = exp(-delta) ~ 1 - 4e-5;
  - Philox sequence ids (found with the oracle's own generator) whose
    accept uniform u_0 is at least 1 - 2^-15 > exp(-delta): the draft token
    is rejected, by a margin far outside any rounding;
  - element 256 holds the row's maximum and element 0 (the draft token) is
    e^-12 below it: both land in the same lane's running sum of pass 1, where
    the two rows' difference at x (about 2.5e-10) is far below half an ulp of
    that sum. The rows' normalisers then come out bit-identical, every other
    element's P_t and P_d are the same float, and the residual is exactly 0.

Odd sequences are ordinary ones (independent target and draft rows), so in
the grouped plan (clusters of 2 CTAs, 2 sequences each, the batch dealt out
snake-wise) every cluster holds one sequence that falls back and one that
does not. The falling-back sequences must reject (n_accepted = 0) and draw
their token by the inverse CDF of P_t row 0 at u2 (checked against float64
unless the draw lies within 1e-6 of an interval edge); the ordinary ones
must agree with the oracle exactly outside the near-tie bands.
"""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from speculative_decoding_verification_24_gb300 import binding, spec_verify_ex
from speculative_decoding_verification_24_gb300.build import build
from test_gpu_parity import check, run_pair

import synth

pytestmark = pytest.mark.gpu

SEED = 7
V = 2048
DELTA = 4e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def near_one_ids(n):
    """n Philox sequence ids whose position-0 accept uniform is >= 1 - 2^-15."""
    ids = np.arange(0, 8_000_000, dtype=np.uint64)
    u, _ = orc.philox_uniforms(SEED, ids, 1)
    hits = ids[np.asarray(u).reshape(-1) >= 1.0 - 2.0 ** -15]
    assert hits.size >= n
    return hits[:n]


def build_case(B):
    g = torch.Generator().manual_seed(11)
    target = torch.empty(B, 2, V, dtype=torch.float32)
    draft = torch.empty(B, 1, V, dtype=torch.float32)
    tokens = torch.zeros(B, 1, dtype=torch.int32)
    ids = np.empty(B, dtype=np.uint64)
    special = near_one_ids((B + 1) // 2)
    for b in range(B):
        if b % 2 == 0:
            row = -20.0 - 4.0 * torch.rand(V, generator=g)
            row[256] = 0.0    # the row's maximum: e = 1
            row[0] = -12.0    # the draft token: same lane and accumulator as element 256
            draft[b, 0] = row
            target[b, 0] = row
            target[b, 0, 0] = -12.0 - DELTA
            target[b, 1] = 3.0 * torch.randn(V, generator=g)
            ids[b] = special[b // 2]
        else:
            target[b] = 3.0 * torch.randn(2, V, generator=g)
            draft[b, 0] = target[b, 0] + torch.randn(V, generator=g)
            tokens[b, 0] = int(torch.multinomial(torch.softmax(draft[b, 0], 0), 1, generator=g))
            ids[b] = 1_000_000_000 + b
    modes = torch.ones(B, dtype=torch.int32)
    case = synth.LogitsCase(target.cuda(), draft.cuda(), tokens.cuda(), modes.cuda(), 1.0)
    return case, torch.from_numpy(ids.astype(np.int64)).cuda()


def pt_draw(row, u2):
    """Inverse CDF of softmax(row) at u2 in float64, and the draw's distance
    to the nearest interval edge."""
    x = row.astype(np.float64)
    p = np.exp(x - x.max())
    p /= p.sum()
    cum = np.cumsum(p)
    k = int(np.searchsorted(cum, u2, side="right"))
    lo = cum[k - 1] if k > 0 else 0.0
    return k, min(u2 - lo, cum[k] - u2)


@pytest.mark.parametrize("plan", [{"seqs_per_cluster": 1, "cluster_size": 2},
                                  {"seqs_per_cluster": 2, "cluster_size": 2}])
def test_a_residual_that_sums_to_zero_falls_back_to_the_target_row(plan):
    B = 64
    case, ids = build_case(B)
    g, ref = run_pair(case, seed=SEED, seq_ids=ids, **plan)
    flags = int(g["status_word"][0])
    assert flags & binding.SV_FLAG_RESIDUAL_FALLBACK, (plan, flags)
    assert not flags & ~binding.SV_FLAG_RESIDUAL_FALLBACK, (plan, flags)
    _, u2 = orc.philox_uniforms(SEED, ids.cpu().numpy().astype(np.uint64), 1)
    u2 = np.asarray(u2).reshape(B, -1)[:, 0]
    target = case.target.cpu().numpy()
    checked = 0
    for b in range(0, B, 2):
        assert g["n_accepted"][b] == 0, (plan, b)
        tok, margin = pt_draw(target[b, 0], float(u2[b]))
        if margin > 1e-6:
            assert g["tokens"][b, 0] == tok, (plan, b, g["tokens"][b], tok)
            checked += 1
        # P_t of row 0 summed to one: the fallback's draw mass
        assert abs(float(g["residual_mass"][b]) - 1.0) < 1e-5, (plan, b, g["residual_mass"][b])
    assert checked >= B // 2 - 2
    # the ordinary sequences agree with the oracle (the falling-back ones
    # are near-ties there: the oracle's float64 residual has mass ~1e-10)
    keep = np.arange(1, B, 2)
    sub = {k: (v[keep] if isinstance(v, np.ndarray) and v.shape[:1] == (B,) else v) for k, v in g.items()}
    subref = {k: (v[keep] if isinstance(v, np.ndarray) and v.shape[:1] == (B,) else v) for k, v in ref.items()}
    check(sub, subref, f"fallback batch, ordinary sequences {plan}", max_tie_fraction=1.0)
