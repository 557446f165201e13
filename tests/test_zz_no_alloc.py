"""spec_verify_lmhead_noalloc: the LM-head verify with its workspace (logits
and per-tile partials) in the library's static device scratch, against
spec_verify_lmhead with a workspace of the caller's.

The file name sorts last so that, in a full run, the static scratch is first
touched after every other test has used the library; the GPU test also
passes alone. The first test needs no GPU: an oversized request is refused on
the host before any device work.
"""
import pytest
import torch

import synth
from speculative_decoding_verification_24_gb300 import binding
from speculative_decoding_verification_24_gb300 import spec_verify_lmhead, spec_verify_lmhead_noalloc
from speculative_decoding_verification_24_gb300.build import build

FAKE = 0x10000  # never dereferenced: the call fails validation first


def test_oversized_request_is_refused_on_the_host():
    build()
    lib = binding.library()
    # B = 13, K = 4 at V = 128256: fp32 logits plus 8-byte partials per row
    # and 128-column tile need 34.3 MB > 32 MiB
    rc = lib.spec_verify_lmhead_noalloc(FAKE, FAKE, FAKE, FAKE, 13, 4, 4096, 128256, 1, 1.0, 1, 0,
                                        FAKE, FAKE, None)
    assert rc == binding.SV_ERR_SCRATCH_LIMIT
    assert b"SV_LMHEAD_SCRATCH_BYTES" in lib.sv_status_string(rc)
    # B = 12 fits: that call gets as far as its host checks (a bad alignment)
    rc = lib.spec_verify_lmhead_noalloc(FAKE + 2, FAKE, FAKE, FAKE, 12, 4, 4096, 128256, 1, 1.0, 1,
                                        0, FAKE, FAKE, None)
    assert rc == 9
    need = binding.spec_verify_lmhead_workspace_bytes
    assert need(12, 4, 4096, 128256) <= binding.SV_LMHEAD_SCRATCH_BYTES < need(13, 4, 4096, 128256)


@pytest.mark.gpu
def test_two_calls_in_a_row_match_the_workspace_entry_point():
    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    # B=8, K=5 of the LM-head workload: 48 rows x 128256 fp32 = 24.6 MB of logits
    # (25.3 MB of workspace with the partials)
    cases = [synth.make_lmhead_case(B=8, K=5, V=128256, d=4096, seed=s, device="cuda")
             for s in (21, 22)]
    for mode in ("sample", "greedy"):
        want = []
        for i, case in enumerate(cases):
            draft = case.draft if mode == "sample" else None
            want.append(spec_verify_lmhead(case.hidden, case.W, draft, case.tokens,
                                           case.temperature, mode=mode, seed=100 + i))
        # two no-alloc calls back to back on one stream: the second reuses the
        # scratch the first wrote
        got = []
        for i, case in enumerate(cases):
            draft = case.draft if mode == "sample" else None
            got.append(spec_verify_lmhead_noalloc(case.hidden, case.W, draft, case.tokens,
                                                  case.temperature, mode=mode, seed=100 + i))
        torch.cuda.synchronize()
        for i in range(len(cases)):
            assert torch.equal(got[i][0], want[i][0]), (i, mode)
            assert torch.equal(got[i][1], want[i][1]), (i, mode)
            assert (got[i][1] >= 0).all()
