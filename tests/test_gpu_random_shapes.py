"""Parity of the verify step with the oracle over seeded random shapes (GPU).

Each case draws B, K, V, the element type, the modes (all sample, all greedy
or mixed), per-sequence draft counts or none, the temperature and the launch
(the default plan, an explicit cluster size, the grouped kernel, or a call
launched to overlap the previous one) from a fixed seed, so the same cases run
every time. Every case is compared with the oracle as the other parity tests
do (exact outside the near-tie bands); the near-ties of all cases together are
capped.
"""
import os

import numpy as np
import pytest
import torch

import synth
from speculative_decoding_verification_24_gb300 import spec_verify_ex
from test_gpu_parity import Tally, check, run_pair

pytestmark = pytest.mark.gpu

# SV_SOAK_CASES raises the count (a longer soak of the same seeded cases)
N_CASES = int(os.environ.get("SV_SOAK_CASES", "32"))


def draw_case(i):
    rng = np.random.default_rng(1000 + i)
    B = int(rng.integers(1, 97))
    K = int(rng.integers(1, 13))
    V = int(rng.choice([int(rng.integers(2, 64)), int(rng.integers(64, 5000)), int(rng.integers(5000, 70000))]))
    dtype = str(rng.choice(["f32", "bf16"]))
    kind = str(rng.choice(["sample", "greedy", "mixed"]))
    modes = (torch.from_numpy(rng.integers(0, 2, B).astype(np.int32)) if kind == "mixed" else kind)
    lens = torch.from_numpy(rng.integers(0, K + 1, B).astype(np.int32)) if rng.random() < 0.4 else None
    T = float(rng.choice([0.5, 1.0, 2.0]))
    launch = str(rng.choice(["default", "cluster", "grouped", "overlap"]))
    kw = {}
    if launch == "cluster":
        kw["cluster_size"] = int(rng.choice([1, 2, 4, 8, 16]))
    elif launch == "grouped":
        cs = int(rng.choice([2, 4, 8, 16]))
        spc_max = min(8, cs, 120 // (2 * K + 1))
        if spc_max >= 2:
            kw["cluster_size"] = cs
            kw["seqs_per_cluster"] = int(rng.integers(2, spc_max + 1))
    elif launch == "overlap":
        kw["overlap_previous"] = True
    return dict(B=B, K=K, V=V, dtype=dtype, kind=kind, modes=modes, lens=lens, T=T, kw=kw, seed=int(rng.integers(0, 1 << 30)))


@pytest.fixture(scope="module")
def tally():
    t = Tally("random shapes")
    yield t
    t.check()


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape(i, tally):
    c = draw_case(i)
    case = synth.make_logits_case(B=c["B"], K=c["K"], V=c["V"], dtype=c["dtype"], modes=c["modes"], T=c["T"],
                                  seed=c["seed"], device="cuda")
    target, draft = case.target, case.draft
    if c["lens"] is not None:
        # rows past a sequence's draft count must not be read
        target, draft = target.clone(), draft.clone()
        for b in range(c["B"]):
            target[b, int(c["lens"][b]) + 1:] = float("nan")
            draft[b, int(c["lens"][b]):] = float("nan")
        case = synth.LogitsCase(target, draft, case.tokens, case.modes, case.temperature)
    label = (f"random {i}: B={c['B']} K={c['K']} V={c['V']} {c['dtype']} {c['kind']}"
             f"{' ragged' if c['lens'] is not None else ''} T={c['T']} {c['kw']}")
    g, ref = run_pair(case, seed=c["seed"] % 1000, draft_lens=c["lens"], **c["kw"])
    tally.add(check(g, ref, label, max_tie_fraction=1.0))
    assert int(g["status_word"][0]) == 0, label


@pytest.mark.parametrize("i", range(2000, 2024))
def test_repeated_calls_agree_bit_for_bit(i):
    """The same call three times gives the same bits in every output (the
    kernels' merge orders are fixed; a race would show here), and reports
    nothing."""
    c = draw_case(i)
    case = synth.make_logits_case(B=c["B"], K=c["K"], V=c["V"], dtype=c["dtype"], modes=c["modes"], T=c["T"],
                                  seed=c["seed"], device="cuda")
    lens = None if c["lens"] is None else c["lens"].cuda()
    outs = []
    for _ in range(3):
        o = spec_verify_ex(case.target, case.draft, case.tokens, case.temperature, modes=case.modes.cuda(),
                           seed=c["seed"] % 1000, debug=True, draft_lens=lens, **c["kw"])
        outs.append({k: v.clone() for k, v in o.items() if isinstance(v, torch.Tensor)})
    torch.cuda.synchronize()
    assert int(outs[0]["status_word"][0]) == 0
    for o in outs[1:]:
        for k, v in o.items():
            torch.testing.assert_close(v, outs[0][k], rtol=0, atol=0, equal_nan=True, msg=f"case {i} {k}")
