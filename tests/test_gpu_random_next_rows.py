"""Greedy tree verification and prompt lookup over seeded random shapes (GPU).

Both are integer work (argmax decisions on logits both sides read in their
stored type; window matching on token ids), so every case must agree with
the oracle exactly. The shapes, dtypes, vocabularies, n-gram and draft counts
and buffer alignments are drawn from fixed seeds, so the same cases run every
time; they reach both prompt-lookup kernels (the whole-context one for
L_max <= 24576, a multiple of 4, on a 16-byte aligned buffer; the cluster
one otherwise).
"""
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from speculative_decoding_verification_24_gb300 import spec_prompt_lookup, spec_verify_tree
from speculative_decoding_verification_24_gb300.build import build
from synth.workloads import to_numpy_logits
from test_gpu_prompt_lookup import contexts
from test_gpu_tree import random_trees

pytestmark = pytest.mark.gpu

# SV_SOAK_CASES raises the count (a longer soak of the same seeded cases)
N_CASES = int(os.environ.get("SV_SOAK_CASES", "12"))


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def draw_tree_case(i):
    rng = np.random.default_rng(5000 + i)
    B = int(rng.integers(1, 49))
    N = int(rng.integers(1, 33))
    V = int(rng.choice([int(rng.integers(2, 64)), int(rng.integers(64, 5000)), int(rng.integers(5000, 70000))]))
    dtype = torch.float32 if rng.random() < 0.5 else torch.bfloat16
    p_follow = float(rng.uniform(0.3, 0.95))
    return B, N, V, dtype, p_follow, int(rng.integers(0, 1 << 20))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_tree_matches_oracle(i):
    B, N, V, dtype, p_follow, seed = draw_tree_case(i)
    target, tokens, parents = random_trees(B, N, V, seed=seed, dtype=dtype, p_follow=p_follow)
    t, n, last = spec_verify_tree(target.cuda(), tokens.cuda(), parents.cuda())
    torch.cuda.synchronize()
    ref = orc.verify_tree(to_numpy_logits(target), tokens.numpy(), parents.numpy())
    label = (i, B, N, V, dtype, p_follow)
    assert (n.cpu().numpy() == ref["n_accepted"]).all(), label
    assert (last.cpu().numpy() == ref["last_node"]).all(), label
    assert (t.cpu().numpy() == ref["tokens"]).all(), label


def draw_lookup_case(i):
    rng = np.random.default_rng(6000 + i)
    L_max = int(rng.choice([int(rng.integers(1, 600)), int(rng.integers(600, 24577)), int(rng.integers(24577, 40000))]))
    if rng.random() < 0.5:
        L_max = max(4, L_max - L_max % 4)  # whole-context kernel when it fits
    B = int(rng.integers(4, max(5, min(300, 4_000_000 // L_max)) + 1))  # the context generator pins lengths 0, 1, 2, L_max
    vocab = int(rng.choice([int(rng.integers(2, 8)), int(rng.integers(8, 100)), int(rng.integers(100, 40000))]))
    m = int(rng.integers(1, 17))
    k = int(rng.integers(1, 65))
    copy_prob = float(rng.uniform(0.1, 0.6))
    unaligned = bool(rng.random() < 0.25)
    return B, L_max, vocab, m, k, copy_prob, unaligned, int(rng.integers(0, 1 << 20))


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_prompt_lookup_matches_oracle(i):
    B, L_max, vocab, m, k, copy_prob, unaligned, seed = draw_lookup_case(i)
    tok, lens = contexts(B, L_max, vocab, seed=seed, copy_prob=copy_prob)
    if unaligned:  # a buffer 4 bytes past a 16-byte boundary
        big = torch.zeros(tok.size + 1, dtype=torch.int32, device="cuda")
        ctx = big[1:].view(B, L_max)
        ctx.copy_(torch.from_numpy(tok))
    else:
        ctx = torch.from_numpy(tok).cuda()
    d, n = spec_prompt_lookup(ctx, torch.from_numpy(lens).cuda(), m, k)
    torch.cuda.synchronize()
    ref = orc.prompt_lookup(tok, lens, m, k)
    label = (i, B, L_max, vocab, m, k, copy_prob, unaligned)
    assert (n.cpu().numpy() == ref["n_drafts"]).all(), label
    assert (d.cpu().numpy() == ref["drafts"]).all(), label
