"""The failure path of the verify kernel, without a GPU fault: a test flag
makes one bounded mbarrier wait per CTA run out (on a barrier nothing
completes). The call must report SV_FLAG_TIMEOUT, mark every sequence
invalid, and leave the context usable for the next call."""
import pytest
import torch

import synth
from speculative_decoding_verification_24_gb300 import binding, spec_verify_ex
from speculative_decoding_verification_24_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("name,modes", [("c2", "sample"), ("c1", "greedy")])
def test_a_wait_that_gives_up_is_reported_and_the_context_stays_usable(name, modes):
    case = synth.make_workload(name, seed=77, device="cuda", **({"tau": 1.0} if name == "c2" else {}))
    out = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=modes, seed=1,
                         debug=True, flags=binding.SV_ARG_TEST_WAIT_TIMEOUT)
    torch.cuda.synchronize()
    assert int(out["status_word"].cpu()[0]) & binding.SV_FLAG_TIMEOUT
    assert (out["n_accepted"].cpu() == -1).all()
    assert (out["tokens"].cpu() == -1).all()
    # the next call on the same context runs normally
    again = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=modes, seed=1,
                           debug=True)
    torch.cuda.synchronize()
    assert int(again["status_word"].cpu()[0]) == 0
    assert (again["n_accepted"].cpu() >= 0).all()
