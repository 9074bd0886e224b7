"""Pins for the oracle's lossless verify (accept / residual / bonus).

Sources: DSpark explainer (papers.franksyz.com mainline topic 31) section 2
(left-to-right verify, correction on the first rejection, bonus token when
every draft is accepted), section 3 (accept with min(1, p/q), residual
max(0, p - q) renormalised, a bad drafter is still lossless), section 16
(check the acceptance/residual implementation exhaustively on a small
vocabulary and compare sampled frequencies); llama.cpp PR 25173
"Losslessness" (greedy output identical to non-speculative greedy).
"""
import json
import os

import numpy as np
import pytest
from scipy import stats

from speculative_decoding_dspark_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "verify_law_worked_examples.json")


def _law(orc, p, q):
    """Exact output law of one verify position, from the oracle's own p, q and
    residual weights: q(v) min(1, p/q) + (1 - sum_y q(y) min(1, p/q)) res(v)."""
    acc = np.where(q > 0, np.minimum(1.0, np.divide(p, q, out=np.ones_like(p), where=q > 0)), 1.0)
    accepted = q * acc
    res, total = orc.residual_weights(p, q)
    res_n = res / total if total > 0 else np.zeros_like(res)
    return accepted + (1.0 - accepted.sum()) * res_n, acc, accepted.sum(), res_n


def test_worked_examples(orc):
    data = json.load(open(GOLDEN))
    for case in data["cases"]:
        p, q = np.array(case["p"]), np.array(case["q"])
        law, acc, beta, res_n = _law(orc, p, q)
        np.testing.assert_allclose(acc, case["accept_prob"], atol=1e-15)
        assert beta == pytest.approx(case["total_accept"], abs=1e-15)
        np.testing.assert_allclose(res_n, case["residual_normalised"], atol=1e-15)
        np.testing.assert_allclose(law, p, atol=1e-15)
        wrong = q * acc + (1.0 - beta) * p
        np.testing.assert_allclose(wrong, case["law_if_resampled_from_p"], atol=1e-15)


def _tiny():
    w = inputs.workload("tiny_exhaustive")
    d = inputs.draft_inputs(w)
    T = inputs.target_full(w, d["U"])
    return w, d, T


def test_exhaustive_law_equals_target(orc):
    """Every position k and every previous token of the V=64 workload: the exact
    law of the committed token equals the target's p (to 1e-12)."""
    w, d, T = _tiny()
    V, gamma = w["V"], w["gamma"]
    invT = float(np.float32(1.0) / np.float32(w["temperature"]))
    for k in range(gamma):
        # one request per previous token, each with base logits U_k at position 0
        U = np.repeat(d["U"][:, k:k + 1, :], V, axis=0)
        out = orc.markov_draft(U, d["W1"], d["W2"], np.arange(V), np.zeros(V, np.uint64), 0,
                               w["temperature"])
        p = orc.softmax(T[0, k].astype(np.float64) * invT)
        for prev in range(V):
            q = orc.softmax(out["q_logits"][prev, 0])
            law, *_ = _law(orc, p, q)
            np.testing.assert_allclose(law, p, rtol=0, atol=1e-12)


@pytest.mark.parametrize("kind", ["one_hot", "uniform", "disjoint", "equal", "reversed"])
def test_exhaustive_law_adversarial_drafter(orc, kind):
    w, d, T = _tiny()
    V = w["V"]
    p = orc.softmax(T[0, 0].astype(np.float64))
    if kind == "one_hot":
        q = np.zeros(V); q[int(np.argmin(p))] = 1.0
    elif kind == "uniform":
        q = np.full(V, 1.0 / V)
    elif kind == "disjoint":
        top = np.argsort(p)[-V // 2:]
        p = np.zeros(V); p[top] = 1.0 / len(top)
        q = np.zeros(V); q[np.setdiff1d(np.arange(V), top)] = 2.0 / V
    elif kind == "equal":
        q = p.copy()
    else:
        q = orc.softmax(-T[0, 0].astype(np.float64))
    law, *_ = _law(orc, p, q)
    np.testing.assert_allclose(law, p, rtol=0, atol=1e-12)


def _run_cycles(orc, w, d, T, temperature, n_cycles, l=None):
    R, gamma = w["R"], w["gamma"]
    l = np.full(R, gamma, np.int32) if l is None else l
    cu = inputs.cu_from_lengths(l)
    target = inputs.pack_rows(T, l)
    outs = []
    for cyc in range(n_cycles):
        dr = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], cyc, temperature)
        v = orc.verify(target, cu, dr["y"], dr["q_logits"], d["seeds"], cyc, temperature)
        assert dr["status"] == 0 and v["status"] == 0
        outs.append((dr, v))
    return outs


def _gtest(counts, probs):
    """G-test of counts against probs, pooling cells with expected count < 5."""
    n = counts.sum()
    exp = probs * n
    order = np.argsort(exp)
    obs_c, exp_c = [], []
    acc_o = acc_e = 0.0
    for i in order:
        acc_o += counts[i]; acc_e += exp[i]
        if acc_e >= 5:
            obs_c.append(acc_o); exp_c.append(acc_e); acc_o = acc_e = 0.0
    if acc_e > 0 and exp_c:
        obs_c[-1] += acc_o; exp_c[-1] += acc_e
    obs_c, exp_c = np.array(obs_c), np.array(exp_c)
    mask = obs_c > 0
    G = 2.0 * (obs_c[mask] * np.log(obs_c[mask] / exp_c[mask])).sum()
    dof = max(len(obs_c) - 1, 1)
    return stats.chi2.sf(G, dof)


def test_empirical_committed_tokens_follow_target(orc):
    """2000 seeded cycles of the V=64 workload at T=1: at every slot the committed
    token's frequencies match the target row's p (G-test, p-value > 1e-3)."""
    w, d, T = _tiny()
    gamma, V = w["gamma"], w["V"]
    outs = _run_cycles(orc, w, d, T, w["temperature"], 2000)
    invT = float(np.float32(1.0) / np.float32(w["temperature"]))
    for slot in range(gamma + 1):
        toks = [v["out_tokens"][0, slot] for _, v in outs if v["n_acc"][0] >= slot]
        if len(toks) < 50:
            continue
        counts = np.bincount(np.array(toks), minlength=V).astype(np.float64)
        p = orc.softmax(T[0, slot].astype(np.float64) * invT)
        pv = _gtest(counts, p)
        assert pv > 1e-3, (slot, len(toks), pv)
    # the drafter is imperfect: some cycles reject, some accept everything
    n_acc = np.array([v["n_acc"][0] for _, v in outs])
    assert (n_acc < gamma).any() and (n_acc > 0).any()


def test_acceptance_ratio_direction(orc):
    """p = (0.9, 0.1), q = (0.5, 0.5), draft token 1: accepted with probability
    min(1, 0.1/0.5) = 0.2; draft token 0 always accepted."""
    V = 2
    target = np.log(np.array([[0.9, 0.1], [0.5, 0.5]], np.float32))
    ql = np.log(np.array([[[0.5, 0.5]]], np.float64))
    cu = np.array([0, 2], np.int32)
    seeds = np.array([77], np.uint64)
    acc1 = [orc.verify(target, cu, np.array([[1]]), ql, seeds, c, 1.0)["n_acc"][0] for c in range(4000)]
    acc0 = [orc.verify(target, cu, np.array([[0]]), ql, seeds, c, 1.0)["n_acc"][0] for c in range(200)]
    rate = np.mean(acc1)
    assert abs(rate - 0.2) < 4 * np.sqrt(0.2 * 0.8 / 4000), rate
    assert all(a == 1 for a in acc0)
    # on rejection of token 1 the residual max(0, p - q) = (0.4, 0) forces token 0
    for c in range(300):
        v = orc.verify(target, cu, np.array([[1]]), ql, seeds, c, 1.0)
        if v["n_acc"][0] == 0:
            assert v["out_tokens"][0, 0] == 0


def test_bonus_row_after_full_acceptance(orc):
    """Drafter equal to the target: every draft is accepted (ratio 1 > u) and
    the token after the block comes from row l (peaked on token 5)."""
    gamma, V = 3, 16
    g = np.random.default_rng(3)
    T = g.normal(0, 1, (gamma + 1, V)).astype(np.float32)
    T[gamma] = -30.0; T[gamma, 5] = 30.0
    T[gamma - 1, 9] = 40.0
    y = np.array([[int(np.argmax(T[j])) for j in range(gamma)]], np.int32)
    ql = T[None, :gamma].astype(np.float64)
    cu = np.array([0, gamma + 1], np.int32)
    for c in range(50):
        v = orc.verify(T, cu, y, ql, np.array([1], np.uint64), c, 1.0)
        assert v["n_acc"][0] == gamma
        assert list(v["out_tokens"][0]) == list(y[0]) + [5]


def test_greedy_equals_target_argmax_chain(orc):
    """Greedy: the committed tokens are the target-argmax chain of length commit_len."""
    for R, V, gamma, seed in [(1, 64, 5, 0), (6, 500, 4, 1), (3, 2000, 7, 2)]:
        w = inputs.workload("qwen3_8b_greedy", seed_offset=seed, R=R, V=V, gamma=gamma, rank=16,
                            w_sigma=0.3)
        d = inputs.draft_inputs(w)
        T = inputs.target_full(w, d["U"])
        dr = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], 0, 0.0)
        # make the drafter agree with the target on a prefix of some requests
        y = dr["y"].copy()
        for r in range(0, R, 2):
            y[r, : gamma // 2] = np.argmax(T[r, : gamma // 2], axis=1)
        l = np.full(R, gamma, np.int32)
        v = orc.verify(inputs.pack_rows(T, l), inputs.cu_from_lengths(l), y, None, d["seeds"], 0, 0.0)
        for r in range(R):
            n = v["n_acc"][r]
            chain = np.argmax(T[r, : n + 1], axis=1)
            assert list(v["out_tokens"][r, : n + 1]) == list(chain)
            assert all(v["out_tokens"][r, n + 1:] == -1)
            assert n == gamma or y[r, n] != chain[n]


def test_plain_decode_when_nothing_verified(orc):
    """l = 0 (target-only fallback): no draft is checked and the single token is
    drawn from row 0 with the bonus noise."""
    V = 8
    T = np.log(np.array([[0.05, 0.05, 0.6, 0.1, 0.05, 0.05, 0.05, 0.05]], np.float32))
    cu = np.array([0, 1], np.int32)
    toks = [orc.verify(T, cu, np.zeros((1, 3), np.int32), np.zeros((1, 3, V)), np.array([9], np.uint64),
                       c, 1.0) for c in range(3000)]
    assert all(t["n_acc"][0] == 0 for t in toks)
    counts = np.bincount([t["out_tokens"][0, 0] for t in toks], minlength=V).astype(float)
    assert _gtest(counts, np.exp(T[0].astype(np.float64))) > 1e-3


def test_variable_lengths_and_bad_inputs(orc):
    w = inputs.workload("varlen_verify", R=12, V=300, gamma=5, rank=16)
    d = inputs.draft_inputs(w)
    T = inputs.target_full(w, d["U"])
    l = inputs.verify_lengths(w)
    assert l.min() < w["gamma"] or l.max() > 0
    dr = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], 0, 1.0)
    v = orc.verify(inputs.pack_rows(T, l), inputs.cu_from_lengths(l), dr["y"], dr["q_logits"],
                   d["seeds"], 0, 1.0)
    assert v["status"] == 0
    assert ((v["n_acc"] >= 0) & (v["n_acc"] <= l)).all()
    # a verify length beyond gamma and an out-of-range draft token are flagged
    cu_bad = inputs.cu_from_lengths(l).copy()
    cu_bad[1:] += 0
    cu_bad[2:] += w["gamma"] + 3 - l[1]
    y_bad = dr["y"].copy(); y_bad[3, 0] = w["V"] + 5
    T_big = np.zeros((cu_bad[-1], w["V"]), np.float32)
    vb = orc.verify(T_big, cu_bad, y_bad, dr["q_logits"], d["seeds"], 0, 1.0)
    assert vb["status"] == -6
    assert vb["n_acc"][1] == -1
    if l[3] > 0:
        assert vb["n_acc"][3] == -1


def test_empty_residual_falls_back_to_target(orc):
    """The empty-residual branch (reading: when max(0, p - q) has no mass in the
    working precision after a rejection, the token is drawn from p with the
    residual's noise).  With exactly normalised p and q a rejection always
    leaves positive residual mass, so only rounding can reach this branch; these
    rows reach it.  Drafter row: 1024 zeros, the drafted token y at -40, seven
    entries at -inf; target row the same with -41 at y, so p(y)/q(y) = 1/e.  The
    true residual mass, q(y) - p(y) ~ (e^-40 - e^-41)/1024 ~ 2.6e-21, is below
    the resolution of ln(1024 + e^-40) in double, so the oracle's p and q agree
    bit for bit everywhere but y and its residual is empty."""
    V, y_tok = 1032, 1024
    s = np.zeros(V, np.float64)
    s[y_tok] = -40.0
    s[y_tok + 1:] = -np.inf
    t = s.copy()
    t[y_tok] = -41.0
    p, q = orc.softmax(t), orc.softmax(s)
    mask = np.arange(V) != y_tok
    np.testing.assert_array_equal(p[mask], q[mask])
    assert p[y_tok] < q[y_tok]
    exact_mass = (np.exp(-40.0) - np.exp(-41.0)) / 1024.0
    assert exact_mass > 0.0
    assert orc.residual_weights(p, q)[1] == 0.0

    target = np.stack([t, np.zeros(V)]).astype(np.float32)  # row 1: the bonus row
    cu = np.array([0, 2], np.int32)
    ql = s[None, None, :]
    seeds = np.array([0x5EED0042], np.uint64)
    rejections = distinct = 0
    for cycle in range(40):
        v = orc.verify(target, cu, np.array([[y_tok]], np.int32), ql, seeds, cycle, 1.0)
        u0 = orc.uniform_single(int(seeds[0]), cycle, 1, 0, 0)
        assert v["n_acc"][0] == (1 if u0 < np.exp(-1.0) else 0)
        if v["n_acc"][0] == 1:
            continue
        rejections += 1
        assert v["residual_empty"][0] == 1
        # the token is the Gumbel-max draw from p with the residual's noise
        # (purpose 2 at the rejected position), not the bonus noise (purpose 3)
        g2 = np.array([-np.log(-np.log(orc.uniform_vocab(int(seeds[0]), cycle, 2, 0, 0, j)))
                       for j in range(V)])
        g3 = np.array([-np.log(-np.log(orc.uniform_vocab(int(seeds[0]), cycle, 3, 0, 0, j)))
                       for j in range(V)])
        assert v["out_tokens"][0, 0] == int(np.argmax(t + g2))
        distinct += int(np.argmax(t + g2)) != int(np.argmax(t + g3))
        assert v["out_tokens"][0, 1] == -1
    assert rejections >= 15, rejections
    assert distinct >= rejections - 1  # the two noises almost never pick the same token
