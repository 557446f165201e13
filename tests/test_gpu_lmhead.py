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
V = 128256 distribution (logit spread ~1.3), so most draws fall inside it.
This comparison checks the GEMM's accuracy. The decisions themselves are
pinned by a second one: the oracle runs on the very fp32 logits the GEMM
wrote (and the same draft rows), and the fused verify must then agree with
it exactly outside the ordinary near-tie bands, as on the logits path.
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


def log_ties(label, res, ref):
    import json
    import os
    path = os.environ.get("SV_PARITY_LOG")
    if not path:
        return
    acc = int((ref["accept_margin"] < ACCEPT_TIE_REL).sum())
    dm = ref["draw_margin"][np.isfinite(ref["draw_margin"])]
    with open(path, "a") as f:
        f.write(json.dumps({"case": label, "sequences": res["sequences"], "near_ties": res["near_ties"],
                            "accept_near_ties": acc, "draw_near_ties": res["near_ties"] - acc,
                            "near_tie_mismatches": res["near_tie_mismatches"],
                            "mismatches": res["mismatches"],
                            "draw_margins": sorted(float(x) for x in dm)}) + "\n")


def check(res, delta):
    assert res["mismatches"] == 0, (res, delta)
    assert res["near_tie_mismatches"] <= max(1, 0.01 * res["sequences"]), (res, delta)


def greedy_ties(ref_logits, B, K1, delta):
    top2 = np.sort(ref_logits.reshape(B, K1, -1), axis=-1)[..., -2:]
    return ((top2[..., 1] - top2[..., 0]) < 2 * delta + 1e-12).any(axis=1)


def gemm_ctas(V):
    """The LM-head GEMM runs one CTA per SM over the 128-column tiles (at most
    one CTA per tile); CTA b computes tiles b, b + G, b + 2G, ..."""
    tiles = (V + 127) // 128
    return min(tiles, torch.cuda.get_device_properties(0).multi_processor_count)


def workspace_parts(ws, M, V):
    """The target rows' partials the fused call leaves after its fp32 logits,
    one per GEMM CTA and row: [G, M, 2] float32 (sample: R, s; greedy: the
    maximum and, as int32 bits, its index)."""
    off = (M * V * 4 + 255) // 256 * 256
    G = gemm_ctas(V)
    return ws[off:off + G * M * 8].view(torch.float32).reshape(G, M, 2).cpu().numpy()


def expected_parts(logits, V, mode, T):
    """Each GEMM CTA's partial of every row over the columns of its tiles,
    from the definition: sample R = ceil(max(l) * c) with c = log2(e)/T (both
    products rounded to float32, as the scale is a float32) and
    s = sum 2^(l*c - R) in float64; greedy the largest logit and its lowest
    index."""
    M = logits.shape[0]
    tiles = (V + 127) // 128
    G = gemm_ctas(V)
    pad = np.full((M, tiles * 128), -np.inf)
    pad[:, :V] = logits
    blk = pad.reshape(M, tiles, 128)
    c32 = np.float32(1.4426950408889634 / T)
    first = np.zeros((G, M))
    second = np.zeros((G, M)) if mode == "sample" else np.zeros((G, M), dtype=np.int64)
    for b in range(G):
        cols = blk[:, b::G, :].reshape(M, -1)  # its tiles in order: increasing column index
        if mode == "sample":
            R = np.ceil(cols.max(axis=1).astype(np.float32) * c32).astype(np.float64)
            first[b] = R
            second[b] = np.exp2(cols * np.float64(c32) - R[:, None]).sum(axis=1)
        else:
            loc = cols.argmax(axis=1)  # first occurrence
            first[b] = cols.max(axis=1)
            second[b] = (b + G * (loc // 128)) * 128 + loc % 128
    return first, second


def check_parts(ws, logits, V, mode, T):
    got = workspace_parts(ws, logits.shape[0], V)
    if mode == "sample":
        R, s = expected_parts(logits, V, mode, T)
        assert np.array_equal(got[..., 0].astype(np.float64), R)
        np.testing.assert_allclose(got[..., 1], s, rtol=1e-5)
    else:
        v, i = expected_parts(logits, V, mode, T)
        assert np.array_equal(got[..., 0].astype(np.float64), v)
        assert np.array_equal(got[..., 1].copy().view(np.int32), i)


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
    if mode == "sample":
        # the fused call's logits are the standalone GEMM's, bit for bit
        ws_logits = ws[:B * K1 * V * 4].view(torch.float32).reshape(B * K1, V)
        assert torch.equal(ws_logits, logits)
    else:
        # a greedy call stores no logits (it decides from the partials): the
        # standalone GEMM's are the same bits (the sample cases check that)
        ws_logits = logits
    # the epilogue's per-tile partials are the reductions of those logits
    check_parts(ws, logits.cpu().numpy().astype(np.float64), V, mode, case.temperature)
    ref_logits = orc.lmhead_logits(bits(case.hidden.reshape(B * K1, d)), bits(case.W))
    delta = float(np.abs(logits.cpu().numpy().astype(np.float64) - ref_logits).max())
    ref = orc.verify(ref_logits.reshape(B, K1, V), bits(case.draft) if mode == "sample" else None,
                     case.tokens.numpy(), case.temperature, 1 if mode == "sample" else 0, seed=seed,
                     threads=16)
    # the oracle on the GPU's own fp32 logits: the fused verify must decide
    # exactly as the oracle does on those values (ordinary near-tie bands)
    ref_gpu = orc.verify(ws_logits.cpu().numpy().reshape(B, K1, V),
                         bits(case.draft) if mode == "sample" else None, case.tokens.numpy(),
                         case.temperature, 1 if mode == "sample" else 0, seed=seed, threads=16)
    return out_t.cpu().numpy(), out_n.cpu().numpy(), ref, ref_logits, delta, ref_gpu


@pytest.mark.parametrize("seed", [0, 1, 2, 4])
def test_verify_lmhead_full_workload_sample(seed):
    case = synth.make_workload("c5", seed=seed)
    B, K1, _ = case.hidden.shape
    got_t, got_n, ref, _, delta, ref_gpu = run_lmhead_case(case, seed, "sample")
    T = case.temperature
    assert delta < 1e-3, delta
    # GEMM accuracy: against the oracle on exact logits, bands widened by
    # the measured logit error
    ties = near_ties(ref, accept_rel=ACCEPT_TIE_REL + 2.2 * delta / T,
                     draw_abs=DRAW_TIE_ABS + 4.4 * delta / T)
    check(compare(got_t, got_n, ref, ties=ties), delta)
    assert (ref["n_accepted"] >= 0).all()
    # every decision at full size: against the oracle on the GPU's logits,
    # the ordinary bands, the same cap on near-ties as the logits path
    res = compare(got_t, got_n, ref_gpu)
    check(res, 0.0)
    log_ties(f"c5 seed={seed}", res, ref_gpu)
    # c5's rows are nearly flat (logit spread ~1.3 over V = 128256), so the
    # chosen token's residual interval is only a few 1e-6 wide and the draw
    # band (measured on the logits path) covers a large share of draws: up to
    # 8 of 32 in the measured seeds. Those are counted, and must still agree
    # but for max(1, 1%) of the sequences.
    assert res["near_ties"] <= 0.35 * res["sequences"], res
    assert (ref_gpu["n_accepted"] >= 0).all()


def test_verify_lmhead_greedy():
    case = synth.make_workload("c5", seed=3)
    B, K1, _ = case.hidden.shape
    got_t, got_n, ref, ref_logits, delta, ref_gpu = run_lmhead_case(case, 3, "greedy")
    check(compare(got_t, got_n, ref, ties=greedy_ties(ref_logits, B, K1, delta)), delta)
    # on the GPU's own logits greedy has no near-ties: equal maxima resolve
    # to the lowest index on both sides
    assert np.array_equal(got_t, ref_gpu["tokens"]) and np.array_equal(got_n, ref_gpu["n_accepted"])


def test_verify_lmhead_small_ragged_vocab():
    case = synth.make_lmhead_case(B=3, K=4, V=1000, d=192, seed=11)
    got_t, got_n, ref, _, delta, ref_gpu = run_lmhead_case(case, 11, "sample")
    ties = near_ties(ref, accept_rel=ACCEPT_TIE_REL + 2.2 * delta, draw_abs=DRAW_TIE_ABS + 4.4 * delta)
    check(compare(got_t, got_n, ref, ties=ties), delta)
    check(compare(got_t, got_n, ref_gpu), 0.0)


@pytest.mark.parametrize("mode,B,K,d,V,T", [
    ("greedy", 8, 4, 128, 1000, 1.0), ("greedy", 32, 5, 64, 8200, 1.0), ("sample", 6, 3, 64, 1000, 4.0),
    ("sample", 20, 7, 128, 3000, 6.0),
    # M = 256 rows (the largest N; two rows per epilogue thread in the tile
    # merge) and 63 rows per sequence in the verify launch's merge
    ("greedy", 8, 31, 64, 1000, 1.0), ("sample", 8, 31, 64, 1000, 4.0),
    # the smallest call, and a last tile of 8 columns (one W box, two lanes
    # of the draft warps)
    ("sample", 1, 1, 64, 8, 1.0), ("greedy", 2, 3, 64, 136, 1.0), ("sample", 2, 3, 64, 136, 2.0),
])
def test_verify_lmhead_exact_logits(mode, B, K, d, V, T):
    # small-integer operands: the GEMM's logits are exact, so the tile
    # partials are checked against the oracle's own logits, and greedy
    # argmax ties (frequent with integer logits) must resolve to the lowest
    # index exactly as the oracle's do
    g = torch.Generator().manual_seed(B * 131 + V)
    hidden = torch.randint(-1, 2, (B, K + 1, d), generator=g).to(torch.bfloat16)
    W = torch.randint(-1, 2, (d, V), generator=g).to(torch.bfloat16)
    ref_logits = orc.lmhead_logits(bits(hidden.reshape(B * (K + 1), d)), bits(W))
    draft = (torch.from_numpy(ref_logits.reshape(B, K + 1, V)[:, :K]).float()
             + torch.randn(B, K, V, generator=g) * 1.5).to(torch.bfloat16)
    p = torch.softmax(draft.float() / T, dim=-1).reshape(B * K, V)
    tokens = torch.multinomial(p, 1, generator=g).reshape(B, K).to(torch.int32)
    if mode == "greedy":  # drafts that often match the target argmax
        top = torch.from_numpy(ref_logits.reshape(B, K + 1, V)[:, :K].argmax(axis=2)).to(torch.int32)
        tokens = torch.where(torch.rand(B, K, generator=g) < 0.7, top, tokens)
    ws = torch.empty(spec_verify_lmhead_workspace_bytes(B, K, d, V), dtype=torch.uint8, device="cuda")
    out_t, out_n = spec_verify_lmhead(hidden.cuda(), W.cuda(), draft.cuda() if mode == "sample" else None,
                                      tokens.cuda(), T, mode=mode, seed=7, workspace=ws)
    torch.cuda.synchronize()
    check_parts(ws, ref_logits, V, mode, T)
    ref = orc.verify(ref_logits.reshape(B, K + 1, V), bits(draft) if mode == "sample" else None,
                     tokens.numpy(), T, 1 if mode == "sample" else 0, seed=7)
    ties = near_ties(ref) if mode == "sample" else None
    res = compare(out_t.cpu().numpy(), out_n.cpu().numpy(), ref, ties=ties)
    if mode == "greedy":
        assert np.array_equal(out_t.cpu().numpy(), ref["tokens"]) and np.array_equal(out_n.cpu().numpy(), ref["n_accepted"])
    else:
        check(res, 0.0)


@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_verify_lmhead_full_size_exact_logits(mode):
    # c5's full shape (B=32, K=5, d=4096, V=128256) with hidden and W in
    # {-1, 0, 1}: every partial sum is an integer of magnitude <= 4096, so the
    # GEMM is exact and the fused verify must decide exactly as the oracle
    # does on its own logits (ordinary near-tie bands; greedy ties resolve to
    # the lowest index on both sides)
    B, K, d, V, T = 32, 5, 4096, 128256, 8.0
    g = torch.Generator().manual_seed(55)
    hidden = torch.randint(-1, 2, (B, K + 1, d), generator=g).to(torch.bfloat16)
    W = torch.randint(-1, 2, (d, V), generator=g).to(torch.bfloat16)
    ref_logits = orc.lmhead_logits(bits(hidden.reshape(B * (K + 1), d)), bits(W)).reshape(B, K + 1, V)
    draft = (torch.from_numpy(ref_logits[:, :K]).float() + torch.randn(B, K, V, generator=g) * 8.0).to(torch.bfloat16)
    p = torch.softmax(draft.float() / T, dim=-1).reshape(B * K, V)
    tokens = torch.multinomial(p, 1, generator=g).reshape(B, K).to(torch.int32)
    if mode == "greedy":
        top = torch.from_numpy(ref_logits[:, :K].argmax(axis=2)).to(torch.int32)
        tokens = torch.where(torch.rand(B, K, generator=g) < 0.7, top, tokens)
    ws = torch.empty(spec_verify_lmhead_workspace_bytes(B, K, d, V), dtype=torch.uint8, device="cuda")
    out_t, out_n = spec_verify_lmhead(hidden.cuda(), W.cuda(), draft.cuda() if mode == "sample" else None,
                                      tokens.cuda(), T, mode=mode, seed=21, workspace=ws)
    torch.cuda.synchronize()
    if mode == "sample":
        gpu_logits = ws[:B * (K + 1) * V * 4].view(torch.float32).reshape(B, K + 1, V).cpu().numpy()
    else:  # a greedy call stores no logits; the GEMM alone computes the same
        gpu_logits = spec_lmhead_logits(hidden.reshape(B * (K + 1), d).cuda(), W.cuda()).cpu().numpy().reshape(B, K + 1, V)
    assert np.array_equal(gpu_logits.astype(np.float64), ref_logits)
    ref = orc.verify(ref_logits, bits(draft) if mode == "sample" else None, tokens.numpy(), T,
                     1 if mode == "sample" else 0, seed=21, threads=16)
    got_t, got_n = out_t.cpu().numpy(), out_n.cpu().numpy()
    if mode == "greedy":
        assert np.array_equal(got_t, ref["tokens"]) and np.array_equal(got_n, ref["n_accepted"])
    else:
        res = compare(got_t, got_n, ref)
        check(res, 0.0)
        assert res["near_ties"] <= 0.35 * res["sequences"], res
    assert (ref["n_accepted"] >= 0).all()


def misaligned_copy(x, elems):
    """x on the GPU, starting `elems` elements past a 256-byte aligned base
    (the rows keep that misalignment: V is a multiple of 8)."""
    n = x.numel()
    buf = torch.empty(n + 64, dtype=x.dtype, device="cuda")
    view = buf[elems:elems + n].view(x.shape)
    view.copy_(x.cuda())
    assert view.data_ptr() % 16 == (elems * x.element_size()) % 16
    return view


@pytest.mark.parametrize("draft_dtype,offset", [
    (torch.float32, 0),   # fp32 draft rows: 16-byte loads in the GEMM's draft warps
    (torch.float32, 1),   # fp32 draft 4 bytes off 16: element loads; draft row with its own slot geometry
    (torch.bfloat16, 1),  # bf16 draft 2 bytes off: element loads, and a draft span read 2 bytes in
    (torch.bfloat16, 2),  # bf16 draft 4 bytes off
    (torch.bfloat16, 4),  # bf16 draft 8 bytes off: 8-byte loads still aligned, span 8 bytes in
])
def test_verify_lmhead_draft_layouts(draft_dtype, offset):
    case = synth.make_lmhead_case(B=5, K=4, V=3000, d=128, seed=40 + offset, w_sigma=0.1)
    B, K1, d = case.hidden.shape
    K, V = K1 - 1, case.W.shape[1]
    draft = case.draft.to(draft_dtype)
    draft_dev = misaligned_copy(draft, offset)
    hidden, W, tokens = case.hidden.cuda(), case.W.cuda(), case.tokens.cuda()
    ws = torch.empty(spec_verify_lmhead_workspace_bytes(B, K, d, V), dtype=torch.uint8, device="cuda")
    out_t, out_n = spec_verify_lmhead(hidden, W, draft_dev, tokens, case.temperature, seed=9, workspace=ws)
    logits = spec_lmhead_logits(hidden, W)
    torch.cuda.synchronize()
    # the draft rows' partials (after the target rows') are their reductions
    M, Md, tiles, G = B * K1, B * K, (V + 127) // 128, gemm_ctas(V)
    off = (M * V * 4 + 255) // 256 * 256 + (tiles * M * 8 + 255) // 256 * 256
    got = ws[off:off + G * Md * 8].view(torch.float32).reshape(G, Md, 2).cpu().numpy()
    R, s = expected_parts(draft.float().reshape(Md, V).numpy().astype(np.float64), V, "sample", case.temperature)
    assert np.array_equal(got[..., 0].astype(np.float64), R)
    np.testing.assert_allclose(got[..., 1], s, rtol=1e-5)
    ref_logits = orc.lmhead_logits(bits(case.hidden.reshape(B * K1, d)), bits(case.W))
    delta = float(np.abs(logits.cpu().numpy().astype(np.float64) - ref_logits).max())
    ref = orc.verify(ref_logits.reshape(B, K1, V), bits(draft), case.tokens.numpy(), case.temperature, 1,
                     seed=9)
    ties = near_ties(ref, accept_rel=ACCEPT_TIE_REL + 2.2 * delta, draw_abs=DRAW_TIE_ABS + 4.4 * delta)
    check(compare(out_t.cpu().numpy(), out_n.cpu().numpy(), ref, ties=ties), delta)
