"""Host-side arithmetic of the benchmark (CPU only): the acceptance statistics
it reports and the algorithmic bytes a verify call is charged with."""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def test_acceptance_counts_by_hand():
    # 4 steps of B = 3 sequences, K = 2; step i uses input set i % 6, and the
    # c2 sets cycle over three noise levels (set k -> level k % 3)
    n = np.array([[0, 1, 2],
                  [2, 2, -1],   # an invalid sequence is left out
                  [1, 0, 0],
                  [2, 1, 0]])
    got = bench.acceptance("c2", n, first=1, count=3, n_sets=6, K=2)
    rows = np.array([2, 2, 1, 0, 0, 2, 1, 0])  # steps 1..3, valid only
    assert got["all"]["sequences"] == 8
    assert np.isclose(got["all"]["mean_tokens_per_verify"], (rows + 1).mean())
    assert np.allclose(got["all"]["accepted_at_position"], [(rows > 0).mean(), (rows > 1).mean()])
    # step 1 -> set 1 -> tau 1.0; step 2 -> set 2 -> tau 3.0; step 3 -> set 3 -> tau 0.3
    assert got["tau=1.0"]["sequences"] == 2 and np.isclose(got["tau=1.0"]["mean_tokens_per_verify"], 3.0)
    assert np.isclose(got["tau=3.0"]["mean_tokens_per_verify"], (2 + 1 + 1) / 3)
    assert np.allclose(got["tau=0.3"]["accepted_at_position"], [2 / 3, 1 / 3])


def test_acceptance_other_workloads_have_no_levels():
    n = np.array([[4, 4], [0, 3]])
    got = bench.acceptance("c4", n, first=0, count=2, n_sets=2, K=4)
    assert set(got) == {"all"}
    assert np.isclose(got["all"]["mean_tokens_per_verify"], (5 + 5 + 1 + 4) / 4)


def test_algorithmic_bytes_by_hand():
    import torch

    class Case:  # B = 3 sequences, K = 4, V = 10 fp32; sequences 0, 2 sample, 1 greedy
        target = torch.zeros(3, 5, 10, dtype=torch.float32)
        modes = torch.tensor([1, 0, 1], dtype=torch.int32)

    row = 10 * 4
    # every target row, the draft rows of the two sample sequences
    base = 3 * 5 * row + 2 * 4 * row
    assert bench.min_bytes(Case) == base
    # sequence 0 rejects at 2 (target and draft row 2 again), sequence 2
    # accepts all 4 (target row 4 again for the bonus); greedy reads nothing more
    assert bench.alg_bytes(Case, np.array([2, 1, 4])) == base + 2 * row + row
    # an invalid sample sequence takes no second pass
    assert bench.alg_bytes(Case, np.array([-1, 0, 4])) == base + row


def test_both_arms_describe_the_workload_identically():
    # the reference arm and the GPU arm build their config from one function
    a = bench.bench_config("c4", 256, 8, 151936, 2, 1_476_000_000, 126 * 2**20, 1)
    b = bench.bench_config("c4", 256, 8, 151936, 2, 1_476_000_000, 126 * 2**20, 1)
    assert a == b and a["workload"].startswith("c4:") and a["rows_per_step"] == 256 * 9


def test_input_sets_exceed_twice_l2():
    l2 = 126 * 2**20
    for name in ("c2", "c3", "c4"):
        n, one = bench.n_input_sets(name, l2)
        assert n >= 2 and n * one > 2 * l2
    n2, _ = bench.n_input_sets("c2", l2)
    assert n2 % 3 == 0  # the c2 sets cycle over three draft-noise levels


def test_sub_results_have_fixed_step_counts():
    for name in ("c2", "c3", "c5", "ragged", "tree", "lookup", "commit"):
        assert bench.SUB_STEPS[name] >= 50
