"""Prompt lookup drafting on the GPU against the oracle (exact: integer work)."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from speculative_decoding_verification_24_gb300 import spec_prompt_lookup
from speculative_decoding_verification_24_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def contexts(B, L_max, vocab, seed, copy_prob=0.3):
    """Token sequences that partly copy earlier spans of themselves (as when
    an answer quotes its prompt), with lengths from 0 to L_max."""
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
    lens[:4] = [0, 1, 2, L_max]
    return tok, lens


@pytest.mark.parametrize("B,L_max,vocab,m,k", [
    (64, 512, 8, 3, 5), (64, 4096, 50, 4, 8), (32, 8192, 32000, 3, 10), (16, 300, 3, 16, 64),
    (8, 1, 5, 1, 1),
    # one CTA per 4096-token tile, up to 8 per sequence (uneven parts, several
    # tiles per CTA, windows that straddle a part or tile boundary)
    (6, 20000, 7, 3, 8), (4, 40000, 100, 5, 16), (5, 12289, 3, 16, 64),
    # the whole-context kernel (L_max a multiple of 4, at most 24576 tokens in
    # shared memory): its largest size, the full benchmark shape, and the
    # first size past it (the cluster kernel again)
    (7, 24576, 11, 3, 8), (256, 16384, 32000, 3, 8), (5, 24580, 9, 4, 12),
])
def test_prompt_lookup_matches_oracle(B, L_max, vocab, m, k):
    tok, lens = contexts(B, L_max, vocab, seed=B + L_max + vocab)
    d, n = spec_prompt_lookup(torch.from_numpy(tok).cuda(), torch.from_numpy(lens).cuda(), m, k)
    torch.cuda.synchronize()
    ref = orc.prompt_lookup(tok, lens, m, k)
    assert (n.cpu().numpy() == ref["n_drafts"]).all()
    assert (d.cpu().numpy() == ref["drafts"]).all()
    if L_max > 16:
        assert (ref["n_drafts"] > 0).sum() >= B // 4


def test_prompt_lookup_invalid_lengths():
    tok, lens = contexts(6, 64, 10, seed=1)
    lens[2], lens[4] = -3, 65
    d, n = spec_prompt_lookup(torch.from_numpy(tok).cuda(), torch.from_numpy(lens).cuda(), 3, 4)
    torch.cuda.synchronize()
    ref = orc.prompt_lookup(tok, lens, 3, 4)
    assert (n.cpu().numpy() == ref["n_drafts"]).all() and (d.cpu().numpy() == ref["drafts"]).all()
    assert n[2] == -1 and n[4] == -1


def test_prompt_lookup_unaligned_contexts_take_the_cluster_kernel():
    # a context buffer that starts 4 bytes past a 16-byte boundary cannot be
    # bulk-copied; the result must not change
    tok, lens = contexts(9, 2048, 20, seed=5)
    big = torch.zeros(tok.size + 1, dtype=torch.int32, device="cuda")
    view = big[1:].view(9, 2048)
    view.copy_(torch.from_numpy(tok))
    d, n = spec_prompt_lookup(view, torch.from_numpy(lens).cuda(), 3, 6)
    torch.cuda.synchronize()
    ref = orc.prompt_lookup(tok, lens, 3, 6)
    assert (n.cpu().numpy() == ref["n_drafts"]).all() and (d.cpu().numpy() == ref["drafts"]).all()
