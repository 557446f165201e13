"""A greedy speculative decode loop kept on the GPU: prompt lookup drafts from
each sequence's context, the verify step checks them (each sequence with its
own draft count), and the commit step appends what was kept. With the greedy
rule the result must equal plain greedy decoding of the target, token for
token ("Inference-4", section "Draft-model speculative decoding"; section
"Prompt lookup decoding" for the drafter). The target is a deterministic toy
function of the last token, so greedy decoding falls into short cycles that
the drafter learns to copy; its logits are built on the host each round."""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_24_gb300 import spec_commit, spec_prompt_lookup, spec_verify_ex
from speculative_decoding_verification_24_gb300.build import build

pytestmark = pytest.mark.gpu

V = 97


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def toy_logits(context):
    a = context[-1] if context else 0
    return np.random.default_rng(a * 1009 + 13).normal(0.0, 3.0, V).astype(np.float32)


def plain_greedy(prompt, n):
    seq = list(prompt)
    for _ in range(n):
        seq.append(int(np.argmax(toy_logits(seq))))
    return seq


def test_lookup_verify_commit_loop_equals_plain_greedy_decoding():
    B, K, L_max, rounds = 12, 6, 256, 30
    rng = np.random.default_rng(0)
    prompts = [rng.integers(0, V, int(rng.integers(2, 9))).tolist() for _ in range(B)]
    ctx = torch.zeros(B, L_max, dtype=torch.int32)
    for b, p in enumerate(prompts):
        ctx[b, :len(p)] = torch.tensor(p, dtype=torch.int32)
    ctx = ctx.cuda()
    lens = torch.tensor([len(p) for p in prompts], dtype=torch.int32).cuda()
    accepted_total = 0
    for _ in range(rounds):
        drafts, nd = spec_prompt_lookup(ctx, lens, max_ngram=3, n_drafts=K)
        torch.cuda.synchronize()
        c_host, l_host, d_host, n_host = (ctx.cpu().numpy(), lens.cpu().numpy(), drafts.cpu().numpy(),
                                          nd.cpu().numpy())
        target = np.zeros((B, K + 1, V), np.float32)
        for b in range(B):
            seq = c_host[b, :l_host[b]].tolist()
            for i in range(n_host[b] + 1):
                target[b, i] = toy_logits(seq + d_host[b, :i].tolist())
        out = spec_verify_ex(torch.from_numpy(target).cuda(), None, drafts, 1.0, modes="greedy",
                             draft_lens=nd)
        committed = spec_commit(ctx, lens, out["tokens"], out["n_accepted"])
        torch.cuda.synchronize()
        assert (committed.cpu().numpy() >= 1).all()
        accepted_total += int(out["n_accepted"].sum())
    c_host, l_host = ctx.cpu().numpy(), lens.cpu().numpy()
    for b in range(B):
        got = c_host[b, :l_host[b]].tolist()
        assert got == plain_greedy(prompts[b], len(got) - len(prompts[b]))
    assert accepted_total > B * rounds  # the drafter copies cycles: more than one token per round
