"""Greedy tree verification on the GPU against the oracle (exact: greedy
decisions compare logits, which both sides read in their stored type)."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from speculative_decoding_verification_24_gb300 import spec_verify, spec_verify_tree
from speculative_decoding_verification_24_gb300.build import build
from synth.workloads import to_numpy_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def random_trees(B, N, V, seed, dtype, p_follow=0.6):
    """Target rows ~ N(0, 3^2); every node hangs under a random earlier node
    and takes its parent's argmax with probability p_follow (so accepted paths
    of several lengths occur), else a random token."""
    g = torch.Generator().manual_seed(seed)
    target = (torch.randn(B, N, V, generator=g) * 3.0).to(dtype)
    am = target.float().argmax(dim=2)  # first maximum, as both sides take it
    rng = np.random.default_rng(seed)
    parents = np.full((B, N), -1, np.int32)
    tokens = np.zeros((B, N), np.int32)
    for b in range(B):
        for i in range(1, N):
            parents[b, i] = rng.integers(0, i)
            if rng.random() < p_follow:
                tokens[b, i] = int(am[b, parents[b, i]])
            else:
                tokens[b, i] = rng.integers(0, V)
    return target, torch.from_numpy(tokens), torch.from_numpy(parents)


def run(target, tokens, parents):
    t, n, last = spec_verify_tree(target.cuda(), tokens.cuda(), parents.cuda())
    torch.cuda.synchronize()
    ref = orc.verify_tree(to_numpy_logits(target), tokens.numpy(), parents.numpy())
    return t.cpu().numpy(), n.cpu().numpy(), last.cpu().numpy(), ref


@pytest.mark.parametrize("B,N,V,dtype", [
    (16, 1, 1000, torch.float32), (16, 8, 1000, torch.float32), (32, 32, 32000, torch.float32),
    (16, 24, 128256, torch.bfloat16), (7, 32, 4099, torch.bfloat16),
])
def test_tree_matches_oracle(B, N, V, dtype):
    target, tokens, parents = random_trees(B, N, V, seed=B * 100 + N, dtype=dtype)
    t, n, last, ref = run(target, tokens, parents)
    assert (n == ref["n_accepted"]).all(), (n, ref["n_accepted"])
    assert (last == ref["last_node"]).all()
    assert (t == ref["tokens"]).all()
    if N > 1:
        assert n.max() >= 2  # the case exercises multi-node paths


def test_chain_tree_equals_linear_greedy():
    B, K, V = 8, 6, 32000
    g = torch.Generator().manual_seed(4)
    target = torch.randn(B, K + 1, V, generator=g) * 3.0
    am = target.argmax(dim=2)
    drafts = torch.where(torch.rand(B, K, generator=g) < 0.7, am[:, :K],
                         torch.randint(0, V, (B, K), generator=g)).to(torch.int32)
    lin_t, lin_n = spec_verify(target.cuda(), None, drafts.cuda(), mode="greedy")
    tokens = torch.cat([torch.zeros(B, 1, dtype=torch.int32), drafts], dim=1)
    parents = torch.arange(-1, K, dtype=torch.int32).expand(B, K + 1).contiguous()
    t, n, last = spec_verify_tree(target.cuda(), tokens.cuda(), parents.cuda())
    torch.cuda.synchronize()
    assert torch.equal(t.cpu(), lin_t.cpu()) and torch.equal(n.cpu(), lin_n.cpu())
    assert torch.equal(last.cpu(), lin_n.cpu())


def test_invalid_trees_are_flagged():
    B, N, V = 4, 6, 500
    target, tokens, parents = random_trees(B, N, V, seed=9, dtype=torch.float32, p_follow=1.0)
    parents[1, 3] = 5          # a parent that is not an earlier node
    tokens[2, 1] = V + 3       # an out-of-range token on a tested node (child of the root)
    target[3, 2, 7] = float("nan")
    t, n, last, ref = run(target, tokens, parents)
    assert (n == ref["n_accepted"]).all() and (t == ref["tokens"]).all() and (last == ref["last_node"]).all()
    assert n[1] == -1 and n[2] == -1 and n[3] == -1 and n[0] >= 0
