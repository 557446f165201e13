"""The fused LM-head verify over seeded random shapes (GPU).

Each case draws B, K, d, V, the temperature and the mode from a fixed seed,
within the entry point's limits (B*(K+1) <= 256 rows, d a multiple of 64, V a
multiple of 8), with hidden states and W in {-1, 0, 1}: every partial sum of
the GEMM is a small integer, so its fp32 logits are exact. The tile partials
in the workspace are then checked against their definition on the oracle's
logits, and the decisions against the oracle: token for token in greedy
mode (integer logits tie often; the lowest index must win on both sides),
exactly outside the ordinary near-tie bands in sample mode. A second group
repeats calls and requires the same bits each time.
"""
import os

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from oracle.parity import compare, near_ties
from speculative_decoding_verification_24_gb300 import spec_verify_lmhead, spec_verify_lmhead_workspace_bytes
from test_gpu_lmhead import bits, check, check_parts

pytestmark = pytest.mark.gpu

# SV_SOAK_CASES raises the count (a longer soak of the same seeded cases)
N_CASES = int(os.environ.get("SV_SOAK_CASES", "16"))


def draw_case(i):
    rng = np.random.default_rng(3000 + i)
    K = int(rng.integers(1, 13))
    B = int(rng.integers(1, min(40, 256 // (K + 1)) + 1))
    d = int(rng.choice([64, 128, 192, 320, 512]))
    V = 8 * int(rng.integers(1, 2500))
    T = float(rng.choice([0.5, 1.0, 2.0]))
    mode = str(rng.choice(["sample", "greedy"]))
    return dict(B=B, K=K, d=d, V=V, T=T, mode=mode, seed=int(rng.integers(0, 1 << 20)))


def make_inputs(c):
    g = torch.Generator().manual_seed(c["seed"])
    B, K, d, V, T = c["B"], c["K"], c["d"], c["V"], c["T"]
    hidden = torch.randint(-1, 2, (B, K + 1, d), generator=g).to(torch.bfloat16)
    W = torch.randint(-1, 2, (d, V), generator=g).to(torch.bfloat16)
    ref_logits = orc.lmhead_logits(bits(hidden.reshape(B * (K + 1), d)), bits(W))
    draft = (torch.from_numpy(ref_logits.reshape(B, K + 1, V)[:, :K]).float()
             + torch.randn(B, K, V, generator=g) * 1.5).to(torch.bfloat16)
    p = torch.softmax(draft.float() / T, dim=-1).reshape(B * K, V)
    tokens = torch.multinomial(p, 1, generator=g).reshape(B, K).to(torch.int32)
    if c["mode"] == "greedy":  # drafts that often match the target argmax
        top = torch.from_numpy(ref_logits.reshape(B, K + 1, V)[:, :K].argmax(axis=2)).to(torch.int32)
        tokens = torch.where(torch.rand(B, K, generator=g) < 0.7, top, tokens)
    return hidden, W, draft, tokens, ref_logits


def run(c, hidden, W, draft, tokens, ws):
    return spec_verify_lmhead(hidden.cuda(), W.cuda(), draft.cuda() if c["mode"] == "sample" else None,
                              tokens.cuda(), c["T"], mode=c["mode"], seed=7, workspace=ws)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_exact_logits(i):
    c = draw_case(i)
    label = f"lmhead random {i}: {c}"
    hidden, W, draft, tokens, ref_logits = make_inputs(c)
    B, K, d, V = c["B"], c["K"], c["d"], c["V"]
    ws = torch.empty(spec_verify_lmhead_workspace_bytes(B, K, d, V), dtype=torch.uint8, device="cuda")
    out_t, out_n = run(c, hidden, W, draft, tokens, ws)
    torch.cuda.synchronize()
    check_parts(ws, ref_logits, V, c["mode"], c["T"])
    ref = orc.verify(ref_logits.reshape(B, K + 1, V), bits(draft) if c["mode"] == "sample" else None,
                     tokens.numpy(), c["T"], 1 if c["mode"] == "sample" else 0, seed=7)
    got_t, got_n = out_t.cpu().numpy(), out_n.cpu().numpy()
    if c["mode"] == "greedy":
        assert np.array_equal(got_t, ref["tokens"]) and np.array_equal(got_n, ref["n_accepted"]), label
    else:
        check(compare(got_t, got_n, ref, ties=near_ties(ref)), 0.0)
    assert (got_n >= 0).all(), label


@pytest.mark.parametrize("i", range(100, 106))
def test_repeated_calls_agree_bit_for_bit(i):
    c = draw_case(i)
    hidden, W, draft, tokens, _ = make_inputs(c)
    B, K, d, V = c["B"], c["K"], c["d"], c["V"]
    ws = torch.empty(spec_verify_lmhead_workspace_bytes(B, K, d, V), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        t, n = run(c, hidden, W, draft, tokens, ws)
        torch.cuda.synchronize()
        outs.append((t.clone(), n.clone(), ws.clone()))
    for t, n, w in outs[1:]:
        assert torch.equal(t, outs[0][0]) and torch.equal(n, outs[0][1]), (i, c)
        # the GEMM's logits and partials are the same bits every time
        assert torch.equal(w, outs[0][2]), (i, c)
