"""The LM head on the tensor cores, and the verify step fed by it (GPU).

The product logits[M, V] = hidden[M, d] . W[d, V] takes bf16 inputs whose
products are exact in fp32; the tensor cores add them in fp32, one K = 16
slice per instruction. The oracle computes the same sum exactly (fp64). With
d/16 additions into an fp32 accumulator, each rounding costs at most 2^-23 of
the running magnitude, so every element must satisfy
    |gpu - exact| <= (d/16 + 1) * 2^-23 * sum_k |hidden[m,k] * W[k,v]|.
Small-integer inputs make every partial sum exactly representable, and there
the result must be bit-exact: any wrong operand layout or index fails it.

The verify step then runs on the fp32 logits the GEMM wrote. The oracle runs
on its exact fp64 logits, so a decision may legitimately differ where the
logit error delta (measured over every element of the case) could move it:
the accept test |u*P_d - P_t| and the draw's distance to an interval edge
move by at most 2*delta/T relative (every logit moves by <= delta, the
log-normaliser by <= delta), and a greedy argmax by a top-2 gap < 2*delta.
That worst-case band is wide next to the probability intervals of a flat
V = 128256 distribution (logit spread ~1.3), so most draws fall inside it;
what keeps the check sharp is that decisions inside the band must still
agree on all but max(1, 1%) of the sequences, as on the logits path.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import oracle as orc
from oracle.parity import ACCEPT_TIE_REL, DRAW_TIE_ABS, compare, near_ties
from speculative_decoding_verification_24_gb300 import (spec_lmhead_logits, spec_verify_lmhead,
                                                        spec_verify_lmhead_workspace_bytes)
from speculative_decoding_verification_24_gb300.build import build
from synth.workloads import to_numpy_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def bits(x):
    return to_numpy_logits(x)


def exact_and_bound(hidden, W):
    """Oracle logits (fp64) and the fp32-accumulation bound per element."""
    hb, wb = bits(hidden), bits(W)
    ref = orc.lmhead_logits(hb, wb)
    d = hb.shape[1]
    mag = np.abs(orc.bf16_to_f64(hb)) @ np.abs(orc.bf16_to_f64(wb))
    return ref, (d // 16 + 1) * 2.0 ** -23 * mag + 1e-30


def randn_bf16(shape, scale, g):
    return (torch.randn(*shape, generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("M,d,V", [
    (1, 64, 128), (16, 64, 256), (6, 128, 1000), (100, 320, 640), (192, 256, 1000),
    (256, 512, 8200), (33, 1024, 136), (192, 4096, 2048),
])
def test_gemm_within_fp32_accumulation_bound(M, d, V):
    g = torch.Generator().manual_seed(M * 7919 + d * 31 + V)
    hidden = randn_bf16((M, d), 1.0, g)
    W = randn_bf16((d, V), 0.02, g)
    out = spec_lmhead_logits(hidden.cuda(), W.cuda())
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    ref, bound = exact_and_bound(hidden, W)
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert (err <= bound).all(), (worst, got[worst], ref[worst], bound[worst])


@pytest.mark.parametrize("M,d,V", [(192, 4096, 1024), (7, 192, 392), (256, 128, 8200)])
def test_gemm_bit_exact_on_small_integers(M, d, V):
    # values in {-2, ..., 2}: every partial sum is an integer below 2^24
    g = torch.Generator().manual_seed(d + V)
    hidden = torch.randint(-2, 3, (M, d), generator=g).to(torch.bfloat16)
    W = torch.randint(-2, 3, (d, V), generator=g).to(torch.bfloat16)
    out = spec_lmhead_logits(hidden.cuda(), W.cuda()).cpu().numpy().astype(np.float64)
    ref = orc.lmhead_logits(bits(hidden), bits(W))
    assert np.array_equal(out, ref)


def test_gemm_c_loop_agrees_with_matrix_product():
    # the oracle's two forms of the product on a small case
    g = torch.Generator().manual_seed(5)
    hidden, W = randn_bf16((3, 64), 1.0, g), randn_bf16((64, 40), 0.5, g)
    a = orc.lmhead_logits(bits(hidden), bits(W))
    b = orc.lmhead_logits(bits(hidden), bits(W), use_c=True)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


def check(res, delta):
    assert res["mismatches"] == 0, (res, delta)
    assert res["near_tie_mismatches"] <= max(1, 0.01 * res["sequences"]), (res, delta)


def greedy_ties(ref_logits, B, K1, delta):
    top2 = np.sort(ref_logits.reshape(B, K1, -1), axis=-1)[..., -2:]
    return ((top2[..., 1] - top2[..., 0]) < 2 * delta + 1e-12).any(axis=1)


def run_lmhead_case(case, seed, mode):
    B, K1, d = case.hidden.shape
    K, V = K1 - 1, case.W.shape[1]
    hidden, W = case.hidden.cuda(), case.W.cuda()
    draft, tokens = case.draft.cuda(), case.tokens.cuda()
    ws = torch.empty(spec_verify_lmhead_workspace_bytes(B, K, d, V), dtype=torch.uint8, device="cuda")
    out_t, out_n = spec_verify_lmhead(hidden, W, draft if mode == "sample" else None, tokens,
                                      case.temperature, mode=mode, seed=seed, workspace=ws)
    logits = spec_lmhead_logits(hidden, W)
    torch.cuda.synchronize()
    # the fused call's logits are the standalone GEMM's, bit for bit
    ws_logits = ws[:B * K1 * V * 4].view(torch.float32).reshape(B * K1, V)
    assert torch.equal(ws_logits, logits)
    ref_logits = orc.lmhead_logits(bits(case.hidden.reshape(B * K1, d)), bits(case.W))
    delta = float(np.abs(logits.cpu().numpy().astype(np.float64) - ref_logits).max())
    ref = orc.verify(ref_logits.reshape(B, K1, V), bits(case.draft) if mode == "sample" else None,
                     case.tokens.numpy(), case.temperature, 1 if mode == "sample" else 0, seed=seed,
                     threads=16)
    return out_t.cpu().numpy(), out_n.cpu().numpy(), ref, ref_logits, delta


@pytest.mark.parametrize("seed", [0, 1, 2, 4])
def test_verify_lmhead_full_workload_sample(seed):
    case = synth.make_workload("c5", seed=seed)
    B, K1, _ = case.hidden.shape
    got_t, got_n, ref, _, delta = run_lmhead_case(case, seed, "sample")
    T = case.temperature
    assert delta < 1e-3, delta
    ties = near_ties(ref, accept_rel=ACCEPT_TIE_REL + 2.2 * delta / T,
                     draw_abs=DRAW_TIE_ABS + 4.4 * delta / T)
    check(compare(got_t, got_n, ref, ties=ties), delta)
    assert (ref["n_accepted"] >= 0).all()


def test_verify_lmhead_greedy():
    case = synth.make_workload("c5", seed=3)
    B, K1, _ = case.hidden.shape
    got_t, got_n, ref, ref_logits, delta = run_lmhead_case(case, 3, "greedy")
    check(compare(got_t, got_n, ref, ties=greedy_ties(ref_logits, B, K1, delta)), delta)


def test_verify_lmhead_small_ragged_vocab():
    case = synth.make_lmhead_case(B=3, K=4, V=1000, d=192, seed=11)
    got_t, got_n, ref, _, delta = run_lmhead_case(case, 11, "sample")
    ties = near_ties(ref, accept_rel=ACCEPT_TIE_REL + 2.2 * delta, draw_abs=DRAW_TIE_ABS + 4.4 * delta)
    check(compare(got_t, got_n, ref, ties=ties), delta)
