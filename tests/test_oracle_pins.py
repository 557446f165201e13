"""Pins of the oracle to facts outside itself (CPU only).

Each test checks the oracle against something it does not compute the same
way: a library Philox run as a black box, a float64 softmax written with
numpy, plain greedy decoding of a toy target, the target distribution itself
(chi-square), the expected-length closed form and the worked example printed
on the pages, an exact enumeration of the joint law on tiny vocabularies, and
cases derived by hand from the rule with the uniforms fixed.
"""
import ctypes
import json
import os
import subprocess

import numpy as np
import pytest
import torch

from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
CHI2_P = 1e-3


def chi2_threshold(dof: int) -> float:
    from scipy.stats import chi2
    return float(chi2.ppf(1.0 - CHI2_P, dof))


def chi2_stat(counts, probs):
    counts = np.asarray(counts, dtype=np.float64)
    n = counts.sum()
    exp = np.asarray(probs, dtype=np.float64) * n
    keep = exp > 0
    assert counts[~keep].sum() == 0, "observed an outcome of probability zero"
    return float(((counts[keep] - exp[keep]) ** 2 / exp[keep]).sum()), int(keep.sum()) - 1


def softmax64(logits, T=1.0):
    z = np.asarray(logits, dtype=np.float64) / T
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


# --------------------------------------------------------------------------- Philox


@pytest.fixture(scope="module")
def aten_philox(tmp_path_factory):
    """ATen's header-only Philox4_32 engine, compiled into a tiny shim."""
    include = os.path.join(os.path.dirname(torch.__file__), "include")
    if not os.path.exists(os.path.join(include, "ATen", "core", "PhiloxRNGEngine.h")):
        pytest.skip("ATen Philox header not available")
    so = str(tmp_path_factory.mktemp("shim") / "aten_philox.so")
    src = os.path.join(os.path.dirname(__file__), "aten_philox_shim.cpp")
    subprocess.run(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-I", include, "-o", so, src],
                   check=True)
    lib = ctypes.CDLL(so)
    lib.aten_philox_words.argtypes = [ctypes.c_uint64] * 3 + [ctypes.c_void_p]
    lib.aten_philox_words.restype = None

    def words(seed, subsequence, offset):
        out = np.zeros(4, dtype=np.uint32)
        lib.aten_philox_words(seed, subsequence, offset, out.ctypes.data)
        return out

    return words


def test_philox_matches_aten_black_box(aten_philox):
    # Counter (pos, seq_lo, seq_hi, 0) and key (seed_lo, seed_hi) map onto
    # ATen's (offset = pos | seq_lo << 32, subsequence = seq_hi, seed).
    rng = np.random.default_rng(1)
    for _ in range(2000):
        seed = int(rng.integers(0, 2**64, dtype=np.uint64))
        seq = int(rng.integers(0, 2**64, dtype=np.uint64))
        pos = int(rng.integers(0, 2**32, dtype=np.uint64))
        ours = orc.philox4x32_10([pos, seq & 0xFFFFFFFF, seq >> 32, 0],
                                 [seed & 0xFFFFFFFF, seed >> 32])
        ref = aten_philox(seed, seq >> 32, pos | ((seq & 0xFFFFFFFF) << 32))
        assert ours.tolist() == ref.tolist()


def test_philox_uniforms_are_uniform_and_exact_in_float():
    ids = np.arange(20000, dtype=np.uint64)
    u, u2 = orc.philox_uniforms(12345, ids, 50)
    for x in (u, u2):
        x = x.ravel()
        assert x.min() >= 0.0 and x.max() <= 1.0 - 2.0**-24
        # exactly representable in float32 (24-bit grid)
        assert np.array_equal(x.astype(np.float32).astype(np.float64), x)
        counts = np.bincount(np.minimum((x * 1000).astype(int), 999), minlength=1000)
        stat, dof = chi2_stat(counts, np.full(1000, 1e-3))
        assert stat < chi2_threshold(dof)
    # u and u2 are not the same stream
    assert abs(np.corrcoef(u.ravel(), u2.ravel())[0, 1]) < 0.01


# --------------------------------------------------------------------------- softmax


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f64"])
@pytest.mark.parametrize("T", [1.0, 0.8, 2.5])
def test_probabilities_match_float64_softmax(dtype, T):
    rng = np.random.default_rng(7)
    B, K, V = 6, 3, 777
    tgt = rng.normal(0, 4, (B, K + 1, V))
    drf = tgt[:, :K] + rng.normal(0, 1, (B, K, V))
    if dtype == "f32":
        tgt, drf = tgt.astype(np.float32), drf.astype(np.float32)
        wide_t, wide_d = tgt.astype(np.float64), drf.astype(np.float64)
    elif dtype == "bf16":
        tgt = torch.from_numpy(tgt).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        drf = torch.from_numpy(drf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        wide_t, wide_d = orc.bf16_to_f64(tgt), orc.bf16_to_f64(drf)
    else:
        wide_t, wide_d = tgt, drf
    tokens = rng.integers(0, V, (B, K)).astype(np.int32)
    # u = 0 accepts every draft with P_t > 0, so every position is tested.
    uni = (np.zeros((B, K + 1)), np.full((B, K + 1), 0.5))
    r = orc.verify(tgt, drf, tokens, T, orc.SAMPLE, uniforms=uni)
    Pt, Pd = softmax64(wide_t, T), softmax64(wide_d, T)
    for b in range(B):
        for i in range(K):
            np.testing.assert_allclose(r["p_target"][b, i], Pt[b, i, tokens[b, i]], rtol=1e-12)
            np.testing.assert_allclose(r["p_draft"][b, i], Pd[b, i, tokens[b, i]], rtol=1e-12)


# --------------------------------------------------------------------------- greedy


def toy_target_logits(context, V, salt=0):
    """A deterministic toy target: logits are a seeded function of the last
    three tokens and the length of the context."""
    key = (salt, len(context)) + tuple(int(t) for t in context[-3:])
    seed = abs(hash(key)) % (2**63)
    return np.random.default_rng(seed).normal(0.0, 3.0, V).astype(np.float32)


def plain_greedy(prompt, n, V):
    seq = list(prompt)
    for _ in range(n):
        seq.append(int(np.argmax(toy_target_logits(seq, V))))
    return seq


def prompt_lookup_drafts(seq, k, max_ngram=3):
    """Draft by copying what followed the latest earlier occurrence of the
    trailing n-gram (longest n first), as in the prompt lookup drafter of
    'Inference-4' (brunomaga.github.io), section 'Prompt lookup decoding'."""
    for n in range(max_ngram, 0, -1):
        if len(seq) <= n:
            continue
        tail = seq[-n:]
        for start in range(len(seq) - n - 1, -1, -1):
            if seq[start:start + n] == tail:
                follow = seq[start + n:start + n + k]
                if follow:
                    return follow
    return []


def speculative_greedy(prompt, n, V, K, drafter, rng):
    seq = list(prompt)
    verifies = 0
    while len(seq) < len(prompt) + n:
        drafts = drafter(seq, K, rng)
        if len(drafts) < K:  # pad short proposals with random tokens
            drafts = list(drafts) + list(rng.integers(0, V, K - len(drafts)))
        rows = np.stack([toy_target_logits(seq + list(drafts[:i]), V) for i in range(K + 1)])
        r = orc.verify(rows[None], None, np.asarray(drafts, dtype=np.int32)[None], 1.0, orc.GREEDY)
        j = int(r["n_accepted"][0])
        assert 0 <= j <= K
        seq.extend(int(t) for t in r["tokens"][0, :j + 1])
        verifies += 1
    return seq[:len(prompt) + n], verifies


@pytest.mark.parametrize("V", [50, 5000])
def test_greedy_equals_plain_target_decoding(V):
    """'Inference-4' (brunomaga.github.io), section 'Draft-model speculative
    decoding': with greedy decoding the output is identical to greedy decoding
    with the target alone, whatever the drafts."""
    rng = np.random.default_rng(3)
    prompt = [int(t) for t in rng.integers(0, V, 6)]
    n = 60
    ref = plain_greedy(prompt, n, V)

    def random_drafter(seq, k, rng):
        return list(rng.integers(0, V, k))

    def noisy_lookahead_drafter(seq, k, rng):
        out, s = [], list(seq)
        for _ in range(k):
            t = int(np.argmax(toy_target_logits(s, V)))
            if rng.random() < 0.25:
                t = int(rng.integers(0, V))
            out.append(t)
            s.append(t)
        return out

    def lookup_drafter(seq, k, rng):
        return prompt_lookup_drafts(seq, k)

    for K in (1, 4, 7):
        for drafter in (random_drafter, noisy_lookahead_drafter, lookup_drafter):
            out, verifies = speculative_greedy(prompt, n, V, K, drafter, rng)
            assert out == ref
            if drafter is noisy_lookahead_drafter and K > 1:
                assert verifies < n  # several tokens per verify were accepted


def test_greedy_ties_take_lowest_index_like_torch_argmax():
    V = 64
    rows = np.zeros((1, 3, V), dtype=np.float32)
    rows[0, 1, [5, 9, 40]] = 2.0   # three-way tie at the maximum
    rows[0, 2, [63, 1]] = 1.0
    for row in rows[0]:
        assert int(torch.argmax(torch.from_numpy(row))) == int(np.argmax(row))
    r = orc.verify(rows, None, np.array([[0, 7]], dtype=np.int32), 1.0, orc.GREEDY)
    # position 0: argmax of an all-zero row is 0 -> draft 0 accepted;
    # position 1: argmax is 5, draft 7 rejected -> correction 5.
    assert r["n_accepted"][0] == 1
    assert r["tokens"][0].tolist() == [0, 5, -1]
    r = orc.verify(rows, None, np.array([[0, 5]], dtype=np.int32), 1.0, orc.GREEDY)
    assert r["tokens"][0].tolist() == [0, 5, 1]  # bonus: argmax of row 2 is 1


# --------------------------------------------------------------------------- sampling law


def run_fixed_pair(p_t_rows, p_d_rows, n_trials, seed, batch=50000):
    """Sequences whose positions all carry the given distributions; drafts
    drawn from P_d with numpy (the drafter), verify by the oracle."""
    K = p_d_rows.shape[0]
    V = p_t_rows.shape[1]
    lt = np.log(np.maximum(p_t_rows, 0.0), where=p_t_rows > 0, out=np.full_like(p_t_rows, -np.inf))
    ld = np.log(np.maximum(p_d_rows, 0.0), where=p_d_rows > 0, out=np.full_like(p_d_rows, -np.inf))
    rng = np.random.default_rng(seed)
    toks, nacc = [], []
    done = 0
    while done < n_trials:
        B = min(batch, n_trials - done)
        x = np.stack([rng.choice(V, size=B, p=p_d_rows[i]) for i in range(K)], axis=1).astype(np.int32)
        tgt = np.ascontiguousarray(np.broadcast_to(lt, (B, K + 1, V)))
        drf = np.ascontiguousarray(np.broadcast_to(ld, (B, K, V)))
        ids = np.arange(done, done + B, dtype=np.uint64)
        r = orc.verify(tgt, drf, x, 1.0, orc.SAMPLE, seed=seed, seq_ids=ids, threads=4)
        toks.append(r["tokens"])
        nacc.append(r["n_accepted"])
        done += B
    return np.concatenate(toks), np.concatenate(nacc)


@pytest.mark.slow
def test_lossless_chi_square_v16():
    """'Speculative decoding' (leoniemonigatti.com blog), section 'Rejection
    sampling', and 'Inference-4', section 'Draft-model speculative decoding':
    accepted plus resampled tokens are distributed exactly as the target."""
    rng = np.random.default_rng(11)
    V, K, N = 16, 3, 1_000_000
    p_t = rng.dirichlet(np.full(V, 0.7), size=K + 1)
    p_d = rng.dirichlet(np.full(V, 0.7), size=K)
    toks, nacc = run_fixed_pair(p_t, p_d, N, seed=2024)
    assert (nacc >= 0).all()
    for i in range(K + 1):
        reached = nacc >= i
        counts = np.bincount(toks[reached, i], minlength=V)
        stat, dof = chi2_stat(counts, p_t[i])
        assert dof == 15
        assert stat < chi2_threshold(dof), (i, stat)
    # bonus position alone
    counts = np.bincount(toks[nacc == K, K], minlength=V)
    stat, dof = chi2_stat(counts, p_t[K])
    assert stat < chi2_threshold(dof)


def expected_tokens(alpha, K):
    return float(K + 1) if alpha == 1.0 else (1 - alpha ** (K + 1)) / (1 - alpha)


@pytest.mark.slow
@pytest.mark.parametrize("K", [4, 8])
def test_mean_tokens_per_verify_matches_closed_form(K):
    """'Inference-4', section 'The idea', and 'Speculative decoding'
    (leoniemonigatti.com blog), section 'Why speculative decoding is fast':
    with i.i.d. acceptance alpha, tokens per verify = (1-alpha^(K+1))/(1-alpha).
    For a fixed pair alpha = sum_v min(P_t, P_d) = 1 - TV(P_t, P_d)."""
    rng = np.random.default_rng(K)
    V, N = 12, 400_000
    p_t1 = rng.dirichlet(np.ones(V))
    p_d1 = 0.5 * p_t1 + 0.5 * rng.dirichlet(np.ones(V))
    alpha = float(np.minimum(p_t1, p_d1).sum())
    toks, nacc = run_fixed_pair(np.tile(p_t1, (K + 1, 1)), np.tile(p_d1, (K, 1)), N, seed=99 + K)
    emitted = nacc + 1.0
    se = emitted.std(ddof=1) / np.sqrt(N)
    assert abs(emitted.mean() - expected_tokens(alpha, K)) < 3 * se
    assert emitted.min() >= 1 and emitted.max() <= K + 1


def test_worked_example_gamma4_alpha07():
    g = json.load(open(os.path.join(GOLDEN, "expected_tokens.json")))["worked_example"]
    K, alpha = g["gamma"], g["alpha"]
    closed = expected_tokens(alpha, K)
    assert abs(closed - g["printed_tokens_per_step"]) < g["printed_precision"]
    N = 300_000
    # two constructions with alpha = 0.7: one degenerate, one not
    pairs = [(np.array([1.0, 0.0]), np.array([0.7, 0.3])),
             (np.array([0.6, 0.4]), np.array([0.3, 0.7]))]
    for p_t1, p_d1 in pairs:
        assert abs(np.minimum(p_t1, p_d1).sum() - alpha) < 1e-12
        _, nacc = run_fixed_pair(np.tile(p_t1, (K + 1, 1)), np.tile(p_d1, (K, 1)), N, seed=5)
        emitted = nacc + 1.0
        se = emitted.std(ddof=1) / np.sqrt(N)
        assert abs(emitted.mean() - closed) < 3 * se


def test_endpoints_alpha_one_and_zero():
    g = json.load(open(os.path.join(GOLDEN, "expected_tokens.json")))["endpoints"]
    assert g["alpha_zero_tokens"] == 1
    K, V = 6, 10
    rng = np.random.default_rng(2)
    p = rng.dirichlet(np.ones(V))
    # P_d = P_t: every draft accepted, K+1 tokens each verify
    _, nacc = run_fixed_pair(np.tile(p, (K + 1, 1)), np.tile(p, (K, 1)), 20000, seed=1)
    assert (nacc == K).all()
    # disjoint supports: every first draft rejected, exactly 1 token
    p_t = np.zeros(V); p_t[:5] = 0.2
    p_d = np.zeros(V); p_d[5:] = 0.2
    toks, nacc = run_fixed_pair(np.tile(p_t, (K + 1, 1)), np.tile(p_d, (K, 1)), 20000, seed=1)
    assert (nacc == 0).all()
    assert (toks[:, 0] < 5).all() and (toks[:, 1:] == -1).all()


def test_target_at_least_as_confident_always_accepts():
    """'What is speculative decoding?' (atomic.chat guide), section 'How
    speculative decoding works': P_t(x) >= P_d(x) is always accepted."""
    V, K = 8, 5
    rng = np.random.default_rng(4)
    p_t = rng.dirichlet(np.ones(V), size=K + 1)
    p_d = rng.dirichlet(np.ones(V), size=K)
    B = 5000
    x = np.zeros((B, K), dtype=np.int32)
    for i in range(K):
        ok = np.flatnonzero(p_t[i] >= p_d[i])
        x[:, i] = rng.choice(ok, size=B)
    lt, ld = np.log(p_t), np.log(p_d)
    tgt = np.ascontiguousarray(np.broadcast_to(lt, (B, K + 1, V)))
    drf = np.ascontiguousarray(np.broadcast_to(ld, (B, K, V)))
    r = orc.verify(tgt, drf, x, 1.0, orc.SAMPLE, seed=77)
    assert (r["n_accepted"] == K).all()
    assert (r["tokens"][:, :K] == x).all()


def test_one_hot_draft_accepts_with_target_probability():
    """Special case of the rule: P_d one-hot at x accepts with probability
    P_t(x); on rejection the residual is P_t without x, renormalised."""
    V, K, N = 6, 1, 200_000
    p_t = np.array([[0.1, 0.25, 0.05, 0.3, 0.2, 0.1], [1 / 6] * 6])
    p_d = np.zeros((1, V)); p_d[0, 3] = 1.0
    toks, nacc = run_fixed_pair(p_t, p_d, N, seed=8)
    # exact, sequence by sequence: accepted iff u * 1 < P_t(x) = 0.3
    u, _ = orc.philox_uniforms(8, np.arange(N, dtype=np.uint64), K + 1)
    np.testing.assert_array_equal(nacc == 1, u[:, 0] < 0.3)
    acc = (nacc == 1).mean()
    z_crit = 3.2905  # two-sided p = 1e-3, as for the chi-square tests
    assert abs(acc - 0.3) < z_crit * np.sqrt(0.3 * 0.7 / N)
    rej = toks[nacc == 0, 0]
    expect = p_t[0].copy(); expect[3] = 0.0; expect /= expect.sum()
    stat, dof = chi2_stat(np.bincount(rej, minlength=V), expect)
    assert stat < chi2_threshold(dof)


def exact_joint_law(p_t, p_d):
    """Exact law of (n_accepted, emitted tokens) by enumeration of draft
    tuples, acceptance and the final draw (V and K tiny)."""
    K, V = p_d.shape
    law = {}

    def add(key, pr):
        if pr > 0:
            law[key] = law.get(key, 0.0) + pr

    def walk(i, prefix, pr):
        if i == K:
            for y in range(V):
                add((K, tuple(prefix) + (y,)), pr * p_t[K, y])
            return
        for x in range(V):
            px = p_d[i, x]
            if px == 0:
                continue
            a = min(1.0, p_t[i, x] / px)
            walk(i + 1, prefix + [x], pr * px * a)
            if a < 1.0:
                res = np.maximum(p_t[i] - p_d[i], 0.0)
                res = res / res.sum()
                for y in range(V):
                    add((i, tuple(prefix) + (y,)), pr * px * (1 - a) * res[y])

    walk(0, [], 1.0)
    return law


@pytest.mark.slow
@pytest.mark.parametrize("V,K", [(3, 2), (4, 1), (2, 2)])
def test_joint_law_matches_exact_enumeration(V, K):
    rng = np.random.default_rng(V * 10 + K)
    p_t = rng.dirichlet(np.ones(V), size=K + 1)
    p_d = rng.dirichlet(np.ones(V), size=K)
    law = exact_joint_law(p_t, p_d)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    # the enumeration's first-token marginal is P_t of row 0 (losslessness)
    first = np.zeros(V)
    for (n, toks), pr in law.items():
        first[toks[0]] += pr
    np.testing.assert_allclose(first, p_t[0], atol=1e-12)
    N = 400_000
    toks, nacc = run_fixed_pair(p_t, p_d, N, seed=31 + V)
    keys = sorted(law)
    index = {k: i for i, k in enumerate(keys)}
    counts = np.zeros(len(keys))
    for t, n in zip(toks, nacc):
        counts[index[(int(n), tuple(int(v) for v in t[:n + 1]))]] += 1
    stat, dof = chi2_stat(counts, np.array([law[k] for k in keys]))
    assert stat < chi2_threshold(dof)


def test_fixed_uniform_cases_derived_by_hand():
    g = json.load(open(os.path.join(GOLDEN, "fixed_uniform_cases.json")))
    for case in g["cases"]:
        p_t = np.array(case["p_target"])
        p_d = np.array(case["p_draft"])
        r = orc.verify(np.log(p_t)[None], np.log(p_d)[None],
                       np.array(case["tokens"], dtype=np.int32)[None], 1.0, orc.SAMPLE,
                       uniforms=(np.array(case["u"])[None], np.array(case["u2"])[None]))
        assert r["tokens"][0].tolist() == case["expected_tokens"], case["name"]
        assert int(r["n_accepted"][0]) == case["expected_n_accepted"], case["name"]


# --------------------------------------------------------------------------- edge cases


def test_invalid_sequences_are_flagged():
    rng = np.random.default_rng(0)
    B, K, V = 5, 3, 20
    tgt = rng.normal(0, 2, (B, K + 1, V)).astype(np.float32)
    drf = rng.normal(0, 2, (B, K, V)).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    x[1, 2] = V          # out of range
    x[2, 0] = -1         # out of range
    tgt[3, K, :] = -np.inf   # a row with no finite maximum
    drf[4, 1, 7] = np.nan    # NaN in a draft row
    for mode in (orc.GREEDY, orc.SAMPLE):
        r = orc.verify(tgt, drf, x, 1.0, mode, seed=3)
        for b in (1, 2, 3):
            assert r["n_accepted"][b] == -1 and (r["tokens"][b] == -1).all()
        assert r["n_accepted"][0] >= 0
        # the NaN sits in a draft row: only sample mode reads it
        assert (r["n_accepted"][4] == -1) == (mode == orc.SAMPLE)


def test_masked_tokens_are_never_emitted():
    rng = np.random.default_rng(5)
    B, K, V = 4000, 2, 30
    tgt = rng.normal(0, 1, (B, K + 1, V)).astype(np.float32)
    tgt[:, :, ::3] = -np.inf   # every third token masked in the target
    drf = rng.normal(0, 1, (B, K, V)).astype(np.float32)
    x = rng.integers(0, V, (B, K)).astype(np.int32)
    r = orc.verify(tgt, drf, x, 1.0, orc.SAMPLE, seed=9)
    n = r["n_accepted"]
    emitted = r["tokens"][np.arange(B), n]
    assert (emitted % 3 != 0).all()
    # a masked draft token has P_t = 0 and is always rejected
    assert ((x[:, 0] % 3 == 0) <= (n == 0)).all()


def test_lmhead_logits_c_loop_matches_float64_matmul():
    rng = np.random.default_rng(6)
    M, d, V = 3, 64, 300
    h = torch.from_numpy(rng.normal(0, 1, (M, d))).to(torch.bfloat16)
    w = torch.from_numpy(rng.normal(0, 0.02, (d, V))).to(torch.bfloat16)
    hb = h.view(torch.int16).numpy().view(np.uint16)
    wb = w.view(torch.int16).numpy().view(np.uint16)
    a = orc.lmhead_logits(hb, wb, use_c=True)
    b = orc.lmhead_logits(hb, wb)
    c = h.double().numpy() @ w.double().numpy()
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(a, c, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mode", [0, 1])
def test_ragged_draft_lengths_equal_separate_fixed_k_calls(mode):
    """Continuous batching: a sequence that verifies only its first Kb of the
    layout's K drafts gives exactly the result of a call laid out with K = Kb
    (same Philox stream: the same sequence id); positions past Kb emit -1."""
    rng = np.random.default_rng(7)
    B, K, V = 7, 5, 40
    tgt = rng.normal(0, 2, (B, K + 1, V))
    drf = tgt[:, :K] + rng.normal(0, 1, (B, K, V))
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    lens = np.array([0, 1, 2, 3, 4, 5, 2], dtype=np.int32)
    got = orc.verify(tgt, drf, tok, 1.0, mode, seed=11, draft_lens=lens)
    for b in range(B):
        k = int(lens[b])
        one = orc.verify(np.ascontiguousarray(tgt[b:b + 1, :k + 1]),
                         np.ascontiguousarray(drf[b:b + 1, :k]) if mode else None,
                         np.ascontiguousarray(tok[b:b + 1, :k]), 1.0, mode, seed=11, seq_ids=[b])
        assert got["n_accepted"][b] == one["n_accepted"][0]
        assert (got["tokens"][b, :k + 1] == one["tokens"][0]).all()
        assert (got["tokens"][b, k + 1:] == -1).all()
        if mode:
            assert np.isnan(got["p_target"][b, k:]).all()


def test_ragged_full_lengths_equal_the_fixed_layout_and_bad_lengths_are_invalid():
    rng = np.random.default_rng(8)
    B, K, V = 5, 4, 30
    tgt = rng.normal(0, 2, (B, K + 1, V))
    drf = tgt[:, :K] + rng.normal(0, 1, (B, K, V))
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    a = orc.verify(tgt, drf, tok, 1.0, 1, seed=3)
    b = orc.verify(tgt, drf, tok, 1.0, 1, seed=3, draft_lens=np.full(B, K))
    assert (a["tokens"] == b["tokens"]).all() and (a["n_accepted"] == b["n_accepted"]).all()
    c = orc.verify(tgt, drf, tok, 1.0, 1, seed=3, draft_lens=[K, -1, K + 1, 0, K])
    assert list(c["n_accepted"][[1, 2]]) == [-1, -1]
    assert (c["tokens"][[1, 2]] == -1).all()
    assert c["n_accepted"][3] == 0 and c["tokens"][3, 0] >= 0 and (c["tokens"][3, 1:] == -1).all()


# ----------------------------------------------------------------- tree verify


def random_tree(rng, N, greedy_prefix, V, p_follow=0.5):
    """A candidate tree of N nodes (node 0 the root): each new node hangs
    under a random earlier node and carries, with probability p_follow, the
    token plain greedy decoding emits there (if its parent is on the greedy
    path), else a random token."""
    parents = [-1]
    tokens = [0]
    on_path = [0]  # depth along the greedy path, or -1 off it
    for i in range(1, N):
        p = int(rng.integers(0, i))
        parents.append(p)
        d = on_path[p]
        if d >= 0 and d < len(greedy_prefix) and rng.random() < p_follow:
            tokens.append(greedy_prefix[d])
            on_path.append(d + 1)
        else:
            t = int(rng.integers(0, V))
            tokens.append(t)
            on_path.append(d + 1 if d >= 0 and d < len(greedy_prefix) and t == greedy_prefix[d] else -1)
    return np.array(tokens, np.int32), np.array(parents, np.int32)


def node_context(prompt, tokens, parents, i):
    path = []
    while i != 0:
        path.append(int(tokens[i]))
        i = int(parents[i])
    return list(prompt) + path[::-1]


@pytest.mark.parametrize("N,V", [(8, 6), (24, 30), (32, 500)])
def test_tree_verify_equals_plain_greedy_decoding(N, V):
    """'Inference-4', section 'Medusa': every candidate in the tree is
    verified in one pass and the longest accepted path is kept. With the
    greedy rule the kept tokens plus the next one must be exactly what plain
    greedy decoding of the target emits, and the path must be the longest one
    whose tokens all follow plain greedy decoding (by brute force)."""
    rng = np.random.default_rng(N * 1000 + V)
    for trial in range(20):
        prompt = [int(t) for t in rng.integers(0, V, 4)]
        greedy = plain_greedy(prompt, N, V)[len(prompt):]
        tokens, parents = random_tree(rng, N, greedy, V)
        target = np.stack([toy_target_logits(node_context(prompt, tokens, parents, i), V) for i in range(N)])
        out = orc.verify_tree(target[None], tokens[None], parents[None])
        n = int(out["n_accepted"][0])
        assert out["tokens"][0, :n + 1].tolist() == greedy[:n + 1]
        assert (out["tokens"][0, n + 1:] == -1).all()
        # brute force: the deepest node whose whole path follows greedy decoding
        best_depth = 0
        for i in range(1, N):
            path = node_context([], tokens, parents, i)
            if path == greedy[:len(path)]:
                best_depth = max(best_depth, len(path))
        assert n == best_depth
        last = int(out["last_node"][0])
        assert len(node_context([], tokens, parents, last)) == n


def test_chain_tree_equals_linear_greedy_verify():
    rng = np.random.default_rng(12)
    B, K, V = 6, 7, 20
    target = rng.normal(0, 2, (B, K + 1, V))
    am = target.argmax(axis=2)
    drafts = np.where(rng.random((B, K)) < 0.7, am[:, :K], rng.integers(0, V, (B, K))).astype(np.int32)
    lin = orc.verify(target, None, drafts, 1.0, 0)
    tokens = np.concatenate([np.zeros((B, 1), np.int32), drafts], axis=1)
    parents = np.broadcast_to(np.arange(-1, K, dtype=np.int32), (B, K + 1))
    tree = orc.verify_tree(target, tokens, parents)
    assert (tree["n_accepted"] == lin["n_accepted"]).all()
    assert (tree["tokens"] == lin["tokens"]).all()
    assert (tree["last_node"] == lin["n_accepted"]).all()


def test_tree_ties_take_the_lowest_node_and_invalid_trees_are_flagged():
    V = 5
    target = np.zeros((1, 5, V))
    target[0, :, 2] = 1.0  # argmax 2 everywhere
    # nodes 1 and 2 both hold the argmax under the root; node 3 under 2, node 4 under 1
    tokens = np.array([[0, 2, 2, 2, 2]], np.int32)
    out = orc.verify_tree(target, tokens, [[-1, 0, 0, 2, 1]])
    assert out["n_accepted"][0] == 2 and out["last_node"][0] == 3  # nodes 3 and 4 equally deep: lower wins
    out = orc.verify_tree(target, tokens, [[-1, 0, 0, 1, 2]])
    assert out["n_accepted"][0] == 2 and out["last_node"][0] == 3
    bad = orc.verify_tree(target, tokens, [[-1, 0, 3, 1, 2]])  # parent not earlier
    assert bad["n_accepted"][0] == -1 and (bad["tokens"][0] == -1).all()
    # an out-of-range token on an untested node (its parent was rejected) is ignored
    ok = orc.verify_tree(target, np.array([[0, 1, 2, 9, 2]], np.int32), [[-1, 0, 0, 1, 2]])
    assert ok["n_accepted"][0] == 2 and ok["last_node"][0] == 4
    bad_tok = orc.verify_tree(target, np.array([[0, 1, 2, 2, 9]], np.int32), [[-1, 0, 0, 1, 2]])
    assert bad_tok["n_accepted"][0] == -1


# ----------------------------------------------------------------- prompt lookup


def test_prompt_lookup_golden_cases():
    cases = json.load(open(os.path.join(GOLDEN, "prompt_lookup_cases.json")))["cases"]
    for c in cases:
        L = len(c["tokens"])
        row = np.array([c["tokens"] + [0] * (12 - L)], np.int32)
        out = orc.prompt_lookup(row, [L], c["max_ngram"], c["n_drafts"])
        n = int(out["n_drafts"][0])
        assert out["drafts"][0, :n].tolist() == c["drafts"], c["why"]
        assert (out["drafts"][0, n:] == -1).all()


def test_prompt_lookup_properties_by_brute_force():
    """On random short sequences over a small alphabet: the drafts follow an
    occurrence of the last n-gram; no later occurrence of that n-gram and no
    occurrence of any longer one exists; with no drafts, no n-gram recurs."""
    rng = np.random.default_rng(2)
    for trial in range(400):
        L = int(rng.integers(0, 30))
        seq = rng.integers(0, 4, L).tolist()
        m, k = int(rng.integers(1, 5)), int(rng.integers(1, 8))
        row = np.array([seq + [9] * (32 - L)], np.int32)
        out = orc.prompt_lookup(row, [L], m, k)
        got = out["drafts"][0, :int(out["n_drafts"][0])].tolist()

        def occurrences(n):
            return [s for s in range(0, L - n) if seq[s:s + n] == seq[L - n:]] if 0 < n < L else []

        found = [(n, occurrences(n)) for n in range(m, 0, -1) if occurrences(n)]
        if not found:
            assert got == []
            continue
        n, occ = found[0]
        assert got == seq[occ[-1] + n: occ[-1] + n + k]
        assert all(not occurrences(n2) for n2 in range(n + 1, m + 1))


def test_prompt_lookup_invalid_length():
    out = orc.prompt_lookup(np.zeros((2, 8), np.int32), [9, -1], 3, 2)
    assert (out["n_drafts"] == -1).all() and (out["drafts"] == -1).all()
