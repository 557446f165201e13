"""GB300-native batched verify step of speculative decoding.

The compute path is libspecverify.so (hand-written sm_103a CUDA kernels behind
the C ABI in include/specverify.h); this package is its Python binding.
"""
from .binding import (SV_BF16, SV_F32, SV_GREEDY, SV_SAMPLE, SpecVerifyError, library, spec_verify,
                      spec_verify_ex, spec_lmhead_logits, spec_verify_lmhead, spec_verify_lmhead_noalloc,
                      spec_verify_lmhead_workspace_bytes, spec_verify_plan, spec_verify_tree, spec_prompt_lookup, spec_commit,
                      sv_status_string, sv_version)

__all__ = ["spec_verify", "spec_verify_ex", "spec_verify_lmhead", "spec_lmhead_logits",
           "spec_verify_lmhead_noalloc", "spec_verify_tree", "spec_prompt_lookup", "spec_commit",
           "spec_verify_lmhead_workspace_bytes", "spec_verify_plan", "sv_status_string", "sv_version",
           "SpecVerifyError", "library", "SV_F32", "SV_BF16", "SV_GREEDY", "SV_SAMPLE"]
