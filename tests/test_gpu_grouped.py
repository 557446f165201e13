"""Parity of the grouped verify kernel with the oracle (GPU).

A plain call over a large batch runs clusters that each verify several
sequences, every CTA of a cluster streaming its slice of V of all of them
(seqs_per_cluster; the library picks such a plan by default for c3).
These cases force the plan over shapes that reach its corners: clusters with
unequal sequence counts, mixed modes and per-sequence draft counts (so the
in-kernel ordering by rows read matters), odd and unaligned rows (partial
edge slots), 31 rows per sequence, B = 256, many clusters, every cluster
size, invalid inputs, the timeout path and the slow paths of the reductions.
"""
import numpy as np
import pytest
import torch

import synth
from speculative_decoding_verification_24_gb300 import SpecVerifyError, binding, spec_verify_ex
from speculative_decoding_verification_24_gb300.build import build
from test_gpu_parity import Tally, check, run_pair

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def mixed_modes(B, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 2, (B,), generator=g, dtype=torch.int32)


def ragged_lens(B, K, seed):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(0, K + 1, (B,), generator=g, dtype=torch.int32)
    lens[0], lens[-1] = 0, K
    return lens


# B, K, V, dtype, modes, cluster size, sequences per cluster
CASES = [
    (37, 3, 5000, "f32", "sample", 8, 4),     # 10 clusters, the last with 1 sequence
    (37, 3, 5000, "f32", "greedy", 8, 8),
    (64, 4, 20000, "bf16", "mixed", 16, 4),
    (64, 4, 20000, "bf16", "mixed", 8, 2),
    (100, 2, 1001, "f32", "sample", 4, 3),    # odd V: partial slots at slice ends
    (100, 2, 1003, "bf16", "mixed", 2, 2),
    (19, 15, 3000, "bf16", "sample", 8, 3),   # 31 rows a sequence, 93 a cluster
    (256, 1, 257, "f32", "mixed", 16, 8),     # B at the limit, 32 clusters of 16
    (25, 5, 32000, "f32", "sample", 8, 5),
    (48, 7, 50257, "bf16", "sample", 16, 7),  # 105 rows a cluster
]


@pytest.mark.parametrize("B,K,V,dtype,modes,cs,spc", CASES)
def test_grouped_parity(B, K, V, dtype, modes, cs, spc):
    m = mixed_modes(B, B + V) if modes == "mixed" else modes
    case = synth.make_logits_case(B=B, K=K, V=V, dtype=dtype, modes=m, seed=B * 13 + K + V, device="cuda")
    label = f"grouped {B},{K},{V},{dtype},{modes},cs={cs},spc={spc}"
    tally = Tally(label)
    for s in range(3):
        g, ref = run_pair(case, seed=s, cluster_size=cs, seqs_per_cluster=spc)
        tally.add(check(g, ref, f"{label} seed={s}", max_tie_fraction=1.0))
        assert int(g["status_word"][0]) == 0
    tally.check()


@pytest.mark.parametrize("B,K,V,dtype,cs,spc", [(64, 4, 20000, "bf16", 8, 2), (90, 6, 3001, "f32", 16, 6),
                                                (40, 8, 7000, "bf16", 8, 7)])
def test_grouped_ragged_draft_counts_and_mixed_modes(B, K, V, dtype, cs, spc):
    """Rows read differ per sequence (mode and draft count), so the clusters'
    shares come from the in-kernel ordering by rows read."""
    case = synth.make_logits_case(B=B, K=K, V=V, dtype=dtype, modes=mixed_modes(B, V), seed=V + K,
                                  device="cuda")
    lens = ragged_lens(B, K, B + K)
    target, draft = case.target.clone(), case.draft.clone()
    for b in range(B):  # rows past a sequence's count must not be read
        target[b, int(lens[b]) + 1:] = float("nan")
        draft[b, int(lens[b]):] = float("nan")
    case = synth.LogitsCase(target, draft, case.tokens, case.modes, case.temperature)
    tally = Tally(f"grouped ragged {B},{K},{V}")
    for s in range(3):
        g, ref = run_pair(case, seed=s, cluster_size=cs, seqs_per_cluster=spc, draft_lens=lens)
        tally.add(check(g, ref, f"grouped ragged {B},{K},{V} seed={s}", max_tie_fraction=1.0))
        assert int(g["status_word"][0]) == 0
        assert (g["n_accepted"] <= lens.numpy()).all()
    tally.check()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_grouped_unaligned_row_starts(dtype):
    B, K, V, off = 30, 3, 1997, 3
    base = synth.make_logits_case(B=B, K=K, V=V, dtype=dtype, modes=mixed_modes(B, 1), seed=off, device="cuda")
    big_t = torch.empty(B * (K + 1) * V + off, dtype=base.target.dtype, device="cuda")
    big_d = torch.empty(B * K * V + 2 * off + 1, dtype=base.draft.dtype, device="cuda")
    tgt = big_t[off:].view(B, K + 1, V)
    drf = big_d[2 * off + 1:].view(B, K, V)
    tgt.copy_(base.target)
    drf.copy_(base.draft)
    case = synth.LogitsCase(tgt, drf, base.tokens, base.modes, base.temperature)
    for s in range(3):
        g, ref = run_pair(case, seed=s, cluster_size=8, seqs_per_cluster=3)
        check(g, ref, f"grouped unaligned {dtype}", max_tie_fraction=1.0)


def test_grouped_masked_tokens_and_huge_spread():
    """The exact (slow) paths of the pass-1 reduction: -inf runs and logits
    far above the warp's running maximum."""
    for dtype in ("f32", "bf16"):
        case = synth.make_logits_case(B=40, K=4, V=6000, dtype=dtype, sigma_t=40.0, seed=19, device="cuda")
        case.target[:, :, ::5] = float("-inf")
        case.draft[:, :, 1::7] = float("-inf")
        for s in range(3):
            g, ref = run_pair(case, seed=s, cluster_size=8, seqs_per_cluster=4)
            check(g, ref, f"grouped masked {dtype}", max_tie_fraction=1.0)
            emitted = g["tokens"][np.arange(40), g["n_accepted"]]
            assert (emitted % 5 != 0).all()


def test_grouped_invalid_inputs_are_flagged_without_faulting():
    case = synth.make_logits_case(B=24, K=4, V=700, dtype="f32", seed=3, device="cuda")
    case.tokens[1, 2] = 700
    case.tokens[2, 0] = -5
    case.target[3, 4, 10] = float("nan")
    case.draft[4, 1, 20] = float("inf")
    case.target[5, 0, :] = float("-inf")
    modes = case.modes.clone()
    modes[6] = 7  # not a mode
    lens = torch.full((24,), 4, dtype=torch.int32)
    lens[7] = 5  # past K
    g, ref = run_pair(case, seed=0, modes=modes, cluster_size=8, seqs_per_cluster=4, draft_lens=lens)
    bad = [1, 2, 3, 4, 5, 6, 7]
    assert g["n_accepted"][bad].tolist() == [-1] * len(bad)
    assert (g["tokens"][bad] == -1).all()
    flags = int(g["status_word"][0])
    assert flags & binding.SV_FLAG_BAD_TOKEN and flags & binding.SV_FLAG_BAD_ROW
    assert flags & binding.SV_FLAG_BAD_MODE and flags & binding.SV_FLAG_BAD_LENGTH
    ok = [b for b in range(24) if b not in bad]
    np.testing.assert_array_equal(g["n_accepted"][ok], ref["n_accepted"][ok])
    np.testing.assert_array_equal(g["tokens"][ok], ref["tokens"][ok])


def test_grouped_timeout_is_reported_and_the_context_stays_usable():
    case = synth.make_workload("c3", seed=77, device="cuda")
    out = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=case.modes, seed=1,
                         debug=True, flags=binding.SV_ARG_TEST_WAIT_TIMEOUT, cluster_size=8, seqs_per_cluster=2)
    torch.cuda.synchronize()
    assert int(out["status_word"].cpu()[0]) & binding.SV_FLAG_TIMEOUT
    assert (out["n_accepted"].cpu() == -1).all()
    assert (out["tokens"].cpu() == -1).all()
    again = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=case.modes, seed=1,
                           debug=True, cluster_size=8, seqs_per_cluster=2)
    torch.cuda.synchronize()
    assert int(again["status_word"].cpu()[0]) == 0
    assert (again["n_accepted"].cpu() >= 0).all()


def test_grouped_plans_the_kernel_cannot_hold_are_refused():
    case = synth.make_logits_case(B=40, K=31, V=3000, dtype="bf16", seed=5, device="cuda")
    for kw in ({"seqs_per_cluster": 9}, {"seqs_per_cluster": -1},
               {"seqs_per_cluster": 2},                      # 2 x 63 rows > 120
               {"seqs_per_cluster": 2, "overlap_previous": True}):
        with pytest.raises(SpecVerifyError):
            spec_verify_ex(case.target, case.draft, case.tokens, 1.0, modes="sample", seed=0, **kw)
    small = synth.make_logits_case(B=40, K=3, V=3000, dtype="bf16", seed=5, device="cuda")
    with pytest.raises(SpecVerifyError):  # more sequences per cluster than its CTAs
        spec_verify_ex(small.target, small.draft, small.tokens, 1.0, modes="sample", seed=0,
                       cluster_size=2, seqs_per_cluster=4)
    torch.cuda.synchronize()


@pytest.mark.parametrize("name,explicit", [("c3", {"cluster_size": 8, "seqs_per_cluster": 2}),
                                           ("c4", {"seqs_per_cluster": 1})])
def test_the_automatic_plan(name, explicit):
    """The plan a plain call gets by default: c3 (B=64, half greedy) runs 32
    clusters of 8 CTAs with two sequences each; c4 (B=256), for which no
    grouped plan fits the GPU in one wave, one cluster per sequence. The
    default call equals, bit for bit, the call that asks for that plan."""
    case = synth.make_workload(name, seed=31, device="cuda")
    a = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=case.modes, seed=2,
                       debug=True)
    b = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=case.modes, seed=2,
                       debug=True, **explicit)
    torch.cuda.synchronize()
    for k in ("tokens", "n_accepted", "p_target", "p_draft", "residual_mass", "draw_edges", "status_word"):
        torch.testing.assert_close(a[k], b[k], rtol=0, atol=0, equal_nan=True, msg=k)


@pytest.mark.parametrize("name,overlap,want", [
    ("c3", False, {"grouped": True, "clusters": 32, "cluster_size": 8, "max_seqs_per_cluster": 2}),
    ("c4", False, {"grouped": False, "clusters": 256, "cluster_size": 1, "max_seqs_per_cluster": 1}),
    ("c2", False, {"grouped": False, "clusters": 8, "cluster_size": 16, "max_seqs_per_cluster": 1}),
    ("c3", True, {"grouped": False, "clusters": 64, "cluster_size": 1, "max_seqs_per_cluster": 1}),
])
def test_spec_verify_plan_reports_the_launch(name, overlap, want):
    """spec_verify_plan reports the launch a call makes (nothing enqueued):
    the grouped plan for c3 alone, one cluster per sequence otherwise."""
    from speculative_decoding_verification_24_gb300 import spec_verify_plan
    case = synth.make_workload(name, seed=32, device="cuda", **({"tau": 1.0} if name == "c2" else {}))
    got = spec_verify_plan(case.target, case.draft, case.tokens, case.temperature, modes=case.modes, seed=0,
                           overlap_previous=overlap)
    assert got == want, (name, overlap, got)
    with pytest.raises(SpecVerifyError):  # refused exactly as the call would be
        spec_verify_plan(case.target, case.draft, case.tokens, case.temperature, modes=case.modes, seed=0,
                         seqs_per_cluster=9)
