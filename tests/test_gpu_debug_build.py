"""The debug build on the GPU (libspecverify_debug.so, built from the same
sources with SPECVERIFY_DEBUG): its verify kernel checks every global load
and store against the buffers of the call, skips an access outside them and
reports it with SV_FLAG_DEBUG_BOUNDS; it never traps. On valid calls it must
compute exactly what the release build computes and report nothing. The
checks are shown to fire with a test-only flag that makes them take the
target logits to end halfway through the buffer: the skipped accesses all lie
inside the real buffer, so nothing can fault."""
import numpy as np
import pytest
import torch

import synth
from speculative_decoding_verification_24_gb300 import (binding, spec_verify_ex, spec_verify_lmhead,
                                                        spec_verify_tree)
from speculative_decoding_verification_24_gb300.build import build

pytestmark = pytest.mark.gpu

KEYS = ("tokens", "n_accepted", "p_target", "p_draft", "residual_mass", "draw_edges")


@pytest.fixture(scope="module")
def dbg():
    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return binding.load_library(binding.DEBUG_LIB_PATH)


def both(case, dbg, seed=3, **kw):
    rel = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=case.modes,
                         seed=seed, debug=True, **kw)
    deb = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=case.modes,
                         seed=seed, debug=True, lib=dbg, **kw)
    torch.cuda.synchronize()
    return rel, deb


def assert_same(rel, deb):
    for k in KEYS:
        torch.testing.assert_close(deb[k], rel[k], rtol=0, atol=0, equal_nan=True, msg=k)
    assert int(rel["status_word"][0]) == 0 and int(deb["status_word"][0]) == 0


@pytest.mark.parametrize("dtype,V,modes", [("f32", 1000, "sample"), ("bf16", 4099, "half"),
                                           ("f32", 32000, "sample"), ("bf16", 7, "greedy")])
def test_debug_build_computes_what_the_release_build_computes(dbg, dtype, V, modes):
    case = synth.make_logits_case(B=12, K=5, V=V, dtype=dtype, modes=modes, seed=V, device="cuda")
    assert_same(*both(case, dbg))
    # calls launched to overlap the previous one (one CTA per sequence) too
    assert_same(*both(case, dbg, seed=4, overlap_previous=True))


def test_debug_build_on_unaligned_rows_and_ragged_lengths(dbg):
    base = synth.make_logits_case(B=6, K=4, V=997, dtype="bf16", seed=2, device="cuda")
    B, K1, V = base.target.shape
    big_t = torch.empty(B * K1 * V + 3, dtype=base.target.dtype, device="cuda")
    big_d = torch.empty(B * (K1 - 1) * V + 5, dtype=base.draft.dtype, device="cuda")
    tgt = big_t[3:].view(B, K1, V)
    drf = big_d[5:].view(B, K1 - 1, V)
    tgt.copy_(base.target)
    drf.copy_(base.draft)
    case = synth.LogitsCase(tgt, drf, base.tokens, base.modes, base.temperature)
    lens = torch.tensor([0, 4, 1, 3, 2, 4], dtype=torch.int32, device="cuda")
    assert_same(*both(case, dbg, draft_lens=lens))


@pytest.mark.parametrize("B,K,V,dtype,modes,cs,spc", [(40, 4, 3001, "bf16", "half", 8, 4),
                                                        (37, 3, 2000, "f32", "sample", 4, 3),
                                                        (64, 4, 20000, "bf16", "half", 8, 2)])
def test_debug_build_grouped_kernel(dbg, B, K, V, dtype, modes, cs, spc):
    # several sequences per cluster (the plan a lone call over a large batch
    # gets), with per-sequence draft counts: every access checked, none outside
    case = synth.make_logits_case(B=B, K=K, V=V, dtype=dtype, modes=modes, seed=B + V, device="cuda")
    lens = torch.tensor([(3 * b) % (K + 1) for b in range(B)], dtype=torch.int32, device="cuda")
    assert_same(*both(case, dbg, cluster_size=cs, seqs_per_cluster=spc))
    assert_same(*both(case, dbg, seed=4, cluster_size=cs, seqs_per_cluster=spc, draft_lens=lens))


def test_debug_build_tree_verification(dbg):
    t, x, par = synth.make_tree_case(4, 8, 3000, "bf16", seed=9, device="cuda")
    rel = spec_verify_tree(t, x, par)
    lib_rel = binding.library()
    torch.cuda.synchronize()
    # the tree entry point through the debug library's C ABI
    out = torch.empty(4, 8, dtype=torch.int32, device="cuda")
    n = torch.empty(4, dtype=torch.int32, device="cuda")
    last = torch.empty(4, dtype=torch.int32, device="cuda")
    st = dbg.spec_verify_tree(t.data_ptr(), binding.SV_BF16, x.data_ptr(), par.data_ptr(), 4, 8, 3000,
                              out.data_ptr(), n.data_ptr(), last.data_ptr(),
                              torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0 and lib_rel is not dbg
    assert torch.equal(out, rel[0]) and torch.equal(n, rel[1]) and torch.equal(last, rel[2])


def test_debug_checks_fire_and_skip_without_faulting(dbg):
    case = synth.make_logits_case(B=16, K=4, V=5000, dtype="bf16", seed=7, device="cuda")
    out = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=case.modes,
                         seed=1, debug=True, lib=dbg, flags=binding.SV_ARG_TEST_DEBUG_SHRINK)
    torch.cuda.synchronize()
    assert int(out["status_word"][0]) & binding.SV_FLAG_DEBUG_BOUNDS
    # the sequences whose rows all lie in the lower half read nothing that
    # was skipped: they decide exactly as in a normal call
    rel = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=case.modes,
                         seed=1, debug=True)
    torch.cuda.synchronize()
    assert torch.equal(out["tokens"][:7], rel["tokens"][:7])
    # the context stays usable: the next normal call is exact
    assert_same(*both(case, dbg, seed=2))


def test_release_build_ignores_the_debug_flag(dbg):
    case = synth.make_logits_case(B=8, K=3, V=2000, dtype="f32", seed=8, device="cuda")
    a = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=case.modes,
                       seed=5, debug=True, flags=binding.SV_ARG_TEST_DEBUG_SHRINK)
    b = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=case.modes,
                       seed=5, debug=True)
    torch.cuda.synchronize()
    assert_same(a, b)


@pytest.mark.parametrize("mode", ["sample", "greedy"])
def test_debug_build_fused_lmhead(dbg, mode):
    # the verify launch that merges the GEMM's tile partials, through both builds
    case = synth.make_lmhead_case(B=4, K=3, V=1000, d=128, seed=13, device="cuda")
    outs = []
    for lib in (None, dbg):
        t, n = spec_verify_lmhead(case.hidden, case.W, case.draft if mode == "sample" else None, case.tokens,
                                  case.temperature, mode=mode, seed=6, lib=lib)
        torch.cuda.synchronize()
        outs.append((t.cpu().numpy(), n.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
