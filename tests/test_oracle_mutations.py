"""The pins catch plausible mistakes in the oracle (CPU only).

Each case plants one mistake in a private copy of ``oracle/oracle.c`` (a
transposed operand, a wrong sign, row or uniform, a dropped term), compiles
it, and checks that at least one quick pin fails against the mutant, while
all of them pass against the real oracle. Mistakes that change nothing
observable (swapping two independent uniforms, ``>`` for ``>=`` on a set of
measure zero) are not planted.
"""
import contextlib
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

from oracle import oracle as orc

from test_oracle_pins import (chi2_stat, chi2_threshold, exact_joint_law, expected_tokens,
                              plain_greedy, run_fixed_pair, softmax64, speculative_greedy,
                              toy_target_logits)
import json

SRC = os.path.join(os.path.dirname(orc.__file__), "oracle.c")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

MUTATIONS = [
    ("accept test operands transposed", "if (!(u[i] * pd < pt))", "if (!(u[i] * pt < pd))"),
    ("residual sign flipped", "double d = Pt[v] - Pd[v];", "double d = Pd[v] - Pt[v];"),
    ("residual not clipped at zero", "r[v] = d > 0.0 ? d : 0.0;", "r[v] = d;"),
    ("bonus drawn from the last draft row",
     "row_softmax(tgt, dtype_t, tgt_off + (size_t)K * V, V, T, Pt);",
     "row_softmax(tgt, dtype_t, tgt_off + (size_t)(K - 1) * V, V, T, Pt);"),
    ("residual draw reuses the accept uniform", "token = inverse_cdf(r, V, u2[j]",
     "token = inverse_cdf(r, V, u[j]"),
    ("temperature dropped",
     "exp((logit_at(base, dtype, row_off + (size_t)v) - m) / T)",
     "exp((logit_at(base, dtype, row_off + (size_t)v) - m))"),
    ("argmax ties go to the last index", "if (l > best) {", "if (l >= best) {"),
    ("philox key not bumped", "k0 += PHILOX_W0;", "k0 += 0u;"),
    ("philox multipliers swapped", "(uint64_t)PHILOX_M0 * (uint64_t)c0",
     "(uint64_t)PHILOX_M1 * (uint64_t)c0"),
    ("greedy emits the draft at the mismatch", "tokens[j] = a;", "tokens[j] = j < K ? x[j] : a;"),
    ("accept test reads the next target row",
     "row_softmax(tgt, dtype_t, tgt_off + (size_t)i * V, V, T, Pt);",
     "row_softmax(tgt, dtype_t, tgt_off + (size_t)(i + 1) * V, V, T, Pt);"),
    ("accept uniform on half the range", "*u = (double)(w[0] >> 8) * (1.0 / 16777216.0);",
     "*u = (double)(w[0] >> 9) * (1.0 / 16777216.0);"),
    ("verification does not stop at the first rejection", "            j = i;\n            break;",
     "            j = i;"),
    ("softmax denominator skips the last token", "for (int v = 0; v < V; ++v) {\n        double e",
     "for (int v = 0; v < V - 1; ++v) {\n        double e"),
]


# ----------------------------------------------------------------- quick pins


def pin_fixed_uniform_cases():
    g = json.load(open(os.path.join(GOLDEN, "fixed_uniform_cases.json")))
    for case in g["cases"]:
        r = orc.verify(np.log(np.array(case["p_target"]))[None],
                       np.log(np.array(case["p_draft"]))[None],
                       np.array(case["tokens"], dtype=np.int32)[None], 1.0, orc.SAMPLE,
                       uniforms=(np.array(case["u"])[None], np.array(case["u2"])[None]))
        assert r["tokens"][0].tolist() == case["expected_tokens"]


def pin_softmax():
    rng = np.random.default_rng(7)
    B, K, V, T = 4, 3, 300, 0.8
    tgt = rng.normal(0, 4, (B, K + 1, V)).astype(np.float32)
    drf = (tgt[:, :K] + rng.normal(0, 1, (B, K, V))).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    r = orc.verify(tgt, drf, x, T, orc.SAMPLE,
                   uniforms=(np.zeros((B, K + 1)), np.full((B, K + 1), 0.5)))
    Pt, Pd = softmax64(tgt, T), softmax64(drf, T)
    for b in range(B):
        for i in range(K):
            np.testing.assert_allclose(r["p_target"][b, i], Pt[b, i, x[b, i]], rtol=1e-12)
            np.testing.assert_allclose(r["p_draft"][b, i], Pd[b, i, x[b, i]], rtol=1e-12)


def pin_greedy():
    V, n = 50, 30
    rng = np.random.default_rng(3)
    prompt = [int(t) for t in rng.integers(0, V, 5)]

    def drafter(seq, k, rng):
        out, s = [], list(seq)
        for _ in range(k):
            t = int(np.argmax(toy_target_logits(s, V)))
            if rng.random() < 0.3:
                t = int(rng.integers(0, V))
            out.append(t)
            s.append(t)
        return out

    out, _ = speculative_greedy(prompt, n, V, 4, drafter, rng)
    assert out == plain_greedy(prompt, n, V)


def pin_ties():
    rows = np.zeros((1, 2, 16), dtype=np.float32)
    rows[0, 0, [3, 8]] = 1.0
    r = orc.verify(rows, None, np.array([[5]], dtype=np.int32), 1.0, orc.GREEDY)
    assert r["tokens"][0].tolist() == [3, -1]


def pin_joint_law():
    V, K = 3, 2
    rng = np.random.default_rng(32)
    p_t = rng.dirichlet(np.ones(V), size=K + 1)
    p_d = rng.dirichlet(np.ones(V), size=K)
    law = exact_joint_law(p_t, p_d)
    toks, nacc = run_fixed_pair(p_t, p_d, 150_000, seed=4)
    keys = sorted(law)
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    for t, n in zip(toks, nacc):
        key = (int(n), tuple(int(v) for v in t[:n + 1]))
        assert key in index, key
        counts[index[key]] += 1
    stat, dof = chi2_stat(counts, np.array([law[k] for k in keys]))
    assert stat < chi2_threshold(dof)


def pin_expected_length():
    K, V, N = 4, 8, 100_000
    rng = np.random.default_rng(1)
    p_t1 = rng.dirichlet(np.ones(V))
    p_d1 = 0.5 * p_t1 + 0.5 * rng.dirichlet(np.ones(V))
    alpha = float(np.minimum(p_t1, p_d1).sum())
    _, nacc = run_fixed_pair(np.tile(p_t1, (K + 1, 1)), np.tile(p_d1, (K, 1)), N, seed=3)
    emitted = nacc + 1.0
    assert abs(emitted.mean() - expected_tokens(alpha, K)) < 3.29 * emitted.std() / np.sqrt(N)


def pin_philox_against_aten(shim):
    rng = np.random.default_rng(1)
    for _ in range(100):
        seed = int(rng.integers(0, 2**64, dtype=np.uint64))
        seq = int(rng.integers(0, 2**32, dtype=np.uint64))
        pos = int(rng.integers(0, 2**32, dtype=np.uint64))
        ours = orc.philox4x32_10([pos, seq, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
        out = np.zeros(4, dtype=np.uint32)
        shim.aten_philox_words(seed, 0, pos | (seq << 32), out.ctypes.data)
        assert ours.tolist() == out.tolist()


def pin_uniform_range():
    u, u2 = orc.philox_uniforms(5, np.arange(4000, dtype=np.uint64), 4)
    for x in (u.ravel(), u2.ravel()):
        counts = np.bincount(np.minimum((x * 20).astype(int), 19), minlength=20)
        stat, dof = chi2_stat(counts, np.full(20, 0.05))
        assert stat < chi2_threshold(dof)


# ----------------------------------------------------------------- harness


@pytest.fixture(scope="module")
def shim(tmp_path_factory):
    include = os.path.join(os.path.dirname(torch.__file__), "include")
    so = str(tmp_path_factory.mktemp("shim") / "aten_philox.so")
    src = os.path.join(os.path.dirname(__file__), "aten_philox_shim.cpp")
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-I", include, "-o", so, src],
                   check=True)
    lib = ctypes.CDLL(so)
    lib.aten_philox_words.argtypes = [ctypes.c_uint64] * 3 + [ctypes.c_void_p]
    return lib


def all_pins(shim):
    return [pin_fixed_uniform_cases, pin_softmax, pin_greedy, pin_ties, pin_joint_law,
            pin_expected_length, lambda: pin_philox_against_aten(shim), pin_uniform_range]


@contextlib.contextmanager
def oracle_library(path):
    saved = orc._load()
    orc._lib = orc._bind(path)
    try:
        yield
    finally:
        orc._lib = saved


def failing_pins(shim):
    failed = []
    for i, pin in enumerate(all_pins(shim)):
        try:
            pin()
        except (AssertionError, IndexError, ValueError):
            failed.append(i)
    return failed


def test_real_oracle_passes_every_quick_pin(shim):
    assert failing_pins(shim) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, shim, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    so = str(tmp_path / "liboracle_mutant.so")
    subprocess.run(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", so, str(mutant), "-lm"],
                   check=True)
    with oracle_library(so):
        failed = failing_pins(shim)
    assert failed, f"no pin caught the planted mistake: {name}"
