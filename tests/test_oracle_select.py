"""Pins for the oracle's survival, capacity and prefix-closed selection.

Sources: DSpark explainer (papers.franksyz.com mainline topic 31) section 5
(a suffix position is worth the product of the conditional acceptance rates),
section 8 (survival a[r,k] from the confidences c[r,k]), section 9 (global
prefix-closed selection maximising predicted output times SPS(B); the causal
greedy stops when Theta stops improving) and section 10 (capacity K from the
confidences of two steps earlier, top-K of the current a within it).
"""
import itertools

import numpy as np
import pytest

from speculative_decoding_dspark_gb300 import inputs


def _brute_best(a, n):
    """max over prefix-closed sets of size n of sum(a); exhaustive over (l_0..l_{R-1})."""
    R, gamma = a.shape
    best = -1.0
    for ls in itertools.product(range(gamma + 1), repeat=R):
        if sum(ls) != n:
            continue
        s = sum(float(a[r, :ls[r]].astype(np.float64).sum()) for r in range(R))
        best = max(best, s)
    return best


def _conf(R, gamma, seed):
    w = inputs.workload("confidence_scheduled", seed_offset=seed, R=R, gamma=gamma)
    return inputs.confidence_inputs(w)


def test_survival_is_cumprod(orc):
    ci = _conf(64, 5, 0)
    out = orc.select_prefix(ci["c"], None, None, None, K_cap=64 * 6, mode=0)
    # numpy's float32 cumprod multiplies left to right in float32: bit-identical
    np.testing.assert_array_equal(out["a"], np.cumprod(ci["c"], axis=1, dtype=np.float32))
    assert (np.diff(out["a"], axis=1) <= 0).all()


@pytest.mark.parametrize("seed", range(4))
def test_topk_is_prefix_closed_and_optimal(orc, seed):
    R, gamma = 3, 3
    ci = _conf(R, gamma, seed)
    for n in range(R * gamma + 1):
        out = orc.select_prefix(ci["c"], None, None, None, K_cap=R + n, mode=0)
        assert out["status"] == 0
        l = out["l"]
        assert l.sum() == n and out["K_used"] == R + n
        assert (l >= 0).all() and (l <= gamma).all()
        np.testing.assert_array_equal(out["cu_seqlens"], inputs.cu_from_lengths(l))
        chosen = sum(float(out["a"][r, :l[r]].astype(np.float64).sum()) for r in range(R))
        assert chosen == pytest.approx(_brute_best(out["a"], n), rel=1e-12, abs=1e-15)


def _theta_table(a, sizes, sps, R, gamma, K_cap):
    th = []
    for S, v in zip(sizes, sps):
        if S < R:
            continue
        n = min(min(S, K_cap) - R, R * gamma)
        th.append((float(v) * (R + _brute_best(a, n)), S, n))
    return th


@pytest.mark.parametrize("seed", range(4))
def test_capacity_planning_is_exhaustive_argmax(orc, seed):
    R, gamma = 3, 3
    ci = _conf(R, gamma, seed)
    sizes = np.array([2, 3, 4, 6, 8, 12], np.int32)
    # a staircase steep enough that the best size varies with the confidences
    sps = (1.0 / (0.010 + 0.0016 * sizes)).astype(np.float32)
    for mode, plan_c in [(1, ci["c_hist"]), (2, ci["c"])]:
        for K_cap in [3, 7, 12]:
            out = orc.select_prefix(ci["c"], ci["c_hist"], sizes, sps, K_cap, mode)
            a_plan = np.cumprod(plan_c, axis=1, dtype=np.float32)
            table = _theta_table(a_plan, sizes, sps, R, gamma, K_cap)
            best = max(table, key=lambda t: (t[0], -t[1]))
            assert out["K_used"] == R + best[2], (mode, K_cap, table)
            # the selection itself always ranks the current a
            chosen = sum(float(out["a"][r, :out["l"][r]].astype(np.float64).sum()) for r in range(R))
            assert chosen == pytest.approx(_brute_best(out["a"], best[2]), rel=1e-12, abs=1e-15)


def test_first_stop_greedy(orc):
    """Mode 3 adds candidates in order of a while Theta strictly grows."""
    for seed in range(6):
        R, gamma = 3, 3
        ci = _conf(R, gamma, seed)
        sizes = np.array([3, 4, 5, 6, 8, 12], np.int32)
        sps = (1.0 / (0.010 + 0.0009 * sizes)).astype(np.float32)
        out = orc.select_prefix(ci["c"], None, sizes, sps, 12, 3)
        a = out["a"]
        n = 0
        pad = lambda B: min([i for i in range(len(sizes)) if sizes[i] >= B], key=lambda i: sizes[i])
        theta = float(sps[pad(R)]) * R
        while n < R * gamma:
            nxt = float(sps[pad(R + n + 1)]) * (R + _brute_best(a, n + 1))
            if not nxt > theta:
                break
            theta, n = nxt, n + 1
        assert out["K_used"] == R + n


def test_staircase_edge_selects_nothing_when_first_stop(orc):
    """At R = 512 (a capture-size edge) the first extra row doubles the padded
    batch, so the first-stop greedy verifies nothing, while the fixed capacity
    K = 1024 verifies the 512 best prefixes."""
    ci = _conf(512, 5, 0)
    g = orc.select_prefix(ci["c"], None, ci["capture_sizes"], ci["sps"], 1024, 3)
    assert g["K_used"] == 512 and (g["l"] == 0).all()
    f = orc.select_prefix(ci["c"], None, ci["capture_sizes"], ci["sps"], 1024, 0)
    assert f["K_used"] == 1024 and f["l"].sum() == 512
    h = orc.select_prefix(ci["c"], ci["c_hist"], ci["capture_sizes"], ci["sps"], 1024, 1)
    assert h["status"] == 0 and h["K_used"] in (512, 1024)


def test_tie_order_k_then_r(orc):
    """Equal survival values are taken in order of position, then request."""
    c = np.ones((3, 2), np.float32)
    out = orc.select_prefix(c, None, None, None, K_cap=3 + 4, mode=0)
    # order: (k0,r0),(k0,r1),(k0,r2),(k1,r0) -> l = [2,1,1]
    assert list(out["l"]) == [2, 1, 1]
    # position before request: a = [[1,1],[1,0.5]], two picks -> (k0,r0),(k0,r1)
    c = np.array([[1.0, 1.0], [1.0, 0.5]], np.float32)
    assert list(orc.select_prefix(c, None, None, None, K_cap=2 + 2, mode=0)["l"]) == [1, 1]
    # lower request first among equal (a, k)
    c = np.array([[0.7, 0.1], [0.7, 0.1], [0.7, 0.1]], np.float32)
    assert list(orc.select_prefix(c, None, None, None, K_cap=3 + 2, mode=0)["l"]) == [1, 1, 0]


def test_select_errors(orc):
    c = np.full((4, 3), 0.5, np.float32)
    assert orc.select_prefix(c, None, None, None, K_cap=3, mode=0)["status"] == -3
    bad = c.copy(); bad[1, 2] = 1.5
    assert orc.select_prefix(bad, None, None, None, K_cap=16, mode=0)["status"] == -6
    bad[1, 2] = np.nan
    assert orc.select_prefix(bad, None, None, None, K_cap=16, mode=0)["status"] == -6
    assert orc.select_prefix(c, None, [4, 8], [1.0, 2.0], 16, 1)["status"] == -1


def test_commit_lengths(orc):
    n_acc = np.array([0, 3, 5, 2], np.int32)
    l = np.array([2, 3, 5, 4], np.int32)
    out = orc.commit_lengths(n_acc, l, 5)
    assert out["status"] == 0
    assert list(out["commit_len"]) == [1, 4, 6, 3]
    assert list(out["cu_commit"]) == [0, 1, 5, 11, 14]
    assert list(out["discard"]) == [2, 0, 0, 2]
    assert out["total"] == 14
    out = orc.commit_lengths(n_acc, None, 5)
    assert list(out["discard"]) == [5, 2, 0, 3]
    bad = orc.commit_lengths(np.array([4], np.int32), np.array([3], np.int32), 5)
    assert bad["status"] == -6


def _brute_best_within(a, n, cap):
    """max over prefix-closed sets of size n with l[r] <= cap[r] of sum(a)."""
    R, gamma = a.shape
    best = -1.0
    for ls in itertools.product(*[range(int(c) + 1) for c in cap]):
        if sum(ls) != n:
            continue
        best = max(best, sum(float(a[r, :ls[r]].astype(np.float64).sum()) for r in range(R)))
    return best


@pytest.mark.parametrize("mode", [4, 5])
def test_cutoff_modes(orc, mode):
    """Static per-request cutoffs (the llama.cpp PR's conf_min confidence
    pruning on the per-position confidence, mode 4; a fixed threshold on the
    survival, mode 5).  With room for every eligible row, l counts the leading
    positions that pass (computed here with numpy); with less room, the kept
    set is the best prefix-closed one inside the eligible prefixes (brute force)."""
    for seed in range(3):
        ci = _conf(40, 6, seed)
        c = ci["c"]
        a = np.cumprod(c, axis=1, dtype=np.float32)
        for conf_min in (0.0, 0.3, 0.6, 0.9, 1.01):
            v = c if mode == 4 else a
            passed = v >= np.float32(conf_min)
            expect = np.where(passed.all(axis=1), c.shape[1], np.argmin(passed, axis=1))
            out = orc.select_prefix(c, None, None, None, 40 * 7, mode, conf_min)
            assert out["status"] == 0
            np.testing.assert_array_equal(out["l"], expect)
            assert out["K_used"] == 40 + expect.sum()
    R, gamma = 3, 3
    for seed in range(4):
        ci = _conf(R, gamma, seed)
        c, a = ci["c"], np.cumprod(ci["c"], axis=1, dtype=np.float32)
        for conf_min in (0.2, 0.5):
            v = c if mode == 4 else a
            passed = v >= np.float32(conf_min)
            cap = np.where(passed.all(axis=1), gamma, np.argmin(passed, axis=1))
            for n in range(int(cap.sum()) + 1):
                out = orc.select_prefix(c, None, None, None, R + n, mode, conf_min)
                l = out["l"]
                assert l.sum() == n and (l <= cap).all()
                got = sum(float(a[r, :l[r]].astype(np.float64).sum()) for r in range(R))
                assert got == pytest.approx(_brute_best_within(a, n, cap), rel=1e-12, abs=1e-15)


def _seq(T, R, gamma, seed):
    w = inputs.workload("confidence_scheduled", seed_offset=seed, R=R, gamma=gamma)
    return inputs.confidence_sequence(w, T)


def test_plan_cycles_accounting(orc):
    """A run of cycles: every cycle's accepted and wasted rows split its verified
    drafts (accepted + wasted = sum l, n_acc = min(n_full, l)); a drafter whose
    every draft is accepted wastes nothing; one whose every draft is rejected
    wastes every verified row and commits the guaranteed token alone."""
    T, R, gamma = 12, 64, 5
    seq = _seq(T, R, gamma, 0)
    sizes, sps = seq["capture_sizes"], seq["sps"]
    for mode in (0, 1, 2, 3, 4, 5):
        out = orc.plan_cycles(seq["c"], seq["n_full"], sizes, sps, 256, mode, 0.5)
        assert out["status"] == 0
        nacc = np.minimum(seq["n_full"], out["l"])
        np.testing.assert_array_equal(out["accepted"], nacc.sum(axis=1))
        np.testing.assert_array_equal(out["accepted"] + out["wasted"], out["l"].sum(axis=1))
        np.testing.assert_array_equal(out["K_used"], R + out["l"].sum(axis=1))
        rate = np.array([sps[np.argmax(sizes >= K)] for K in out["K_used"]], np.float64)
        np.testing.assert_allclose(out["theta_real"], rate * (R + out["accepted"]), rtol=1e-15)
    full = orc.plan_cycles(seq["c"], np.full((T, R), gamma, np.int32), sizes, sps, 256, 0)
    assert (full["wasted"] == 0).all() and (full["accepted"] == full["l"].sum(axis=1)).all()
    none = orc.plan_cycles(seq["c"], np.zeros((T, R), np.int32), sizes, sps, 256, 0)
    assert (none["accepted"] == 0).all() and (none["wasted"] == none["l"].sum(axis=1)).all()
    assert (none["theta_real"] == np.array([sps[np.argmax(sizes >= K)] for K in none["K_used"]]) * R).all()


def test_plan_cycles_history_is_causal(orc):
    """HISTORY takes cycle t's capacity from cycle t - lag: the first lag cycles
    use K_cap; later, the capacity is the one the single-cycle CURRENT mode
    picks on the confidences of cycle t - lag, while the logical selection is
    the top of cycle t's own survival; with every cycle's confidences equal
    the two modes coincide."""
    T, R, gamma = 10, 96, 5
    seq = _seq(T, R, gamma, 1)
    sizes, sps = seq["capture_sizes"], seq["sps"]
    K_cap = 512
    for lag in (1, 2, 3):
        h = orc.plan_cycles(seq["c"], seq["n_full"], sizes, sps, K_cap, 1, lag=lag)
        assert (h["K_used"][:lag] == min(K_cap, R * (gamma + 1))).all()
        for t in range(lag, T):
            cur = orc.select_prefix(seq["c"][t - lag], None, sizes, sps, K_cap, 2)
            assert h["K_used"][t] == cur["K_used"]
            top = orc.select_prefix(seq["c"][t], None, None, None, cur["K_used"], 0)
            np.testing.assert_array_equal(h["l"][t], top["l"])
    same = np.broadcast_to(seq["c"][0], seq["c"].shape).copy()
    h = orc.plan_cycles(same, None, sizes, sps, K_cap, 1)
    c = orc.plan_cycles(same, None, sizes, sps, K_cap, 2)
    np.testing.assert_array_equal(h["l"][2:], c["l"][2:])
    np.testing.assert_allclose(h["theta_pred"][2:], c["theta_pred"][2:], rtol=1e-15)


def _nll(beta, z, y):
    x = beta * z.astype(np.float64)
    return float(np.sum(np.logaddexp(0.0, x) - y * x))


def test_fit_temperatures_recovers_and_matches_library(orc):
    """Sequential temperature scaling: on labels drawn from known per-position
    temperatures the fit recovers them, and every position's temperature is the
    minimiser of its conditioned NLL found by scipy's bounded scalar search on
    the samples that reached the position."""
    from scipy.optimize import minimize_scalar
    w = inputs.workload("confidence_scheduled")
    cs = inputs.calibration_samples(w, 200_000)
    out = orc.fit_temperatures(cs["z"], cs["accepted"])
    assert out["status"] == 0
    np.testing.assert_allclose(out["tau"], cs["tau_true"], rtol=0.03)
    acc = cs["accepted"].astype(np.float64)
    for k in range(w["gamma"]):
        reached = np.ones(len(acc), bool) if k == 0 else acc[:, :k].all(axis=1)
        assert out["count"][k] == reached.sum()
        zk, yk = cs["z"][reached, k], acc[reached, k]
        res = minimize_scalar(lambda b: _nll(b, zk, yk), bounds=(1e-3, 1e3), method="bounded",
                              options={"xatol": 1e-12})
        assert 1.0 / out["tau"][k] == pytest.approx(res.x, rel=1e-5)
        assert out["nll"][k] == pytest.approx(_nll(res.x, zk, yk) / reached.sum(), rel=1e-9)


def test_fit_temperatures_conditions_on_reaching_the_position(orc):
    """Labels after a rejection do not enter the fit (setting them all to 1
    changes nothing), whereas fitting position 1 on every sample would give a
    different temperature; a position no sample reaches keeps tau = 1."""
    w = inputs.workload("confidence_scheduled", gamma=3)
    cs = inputs.calibration_samples(w, 50_000, tau_true=[1.0, 2.0, 0.5])
    base = orc.fit_temperatures(cs["z"], cs["accepted"])
    noisy = cs["accepted"].copy()
    reached = np.concatenate([np.ones((len(noisy), 1), bool),
                              np.cumprod(noisy, axis=1)[:, :-1].astype(bool)], axis=1)
    noisy[~reached] = 1
    alt = orc.fit_temperatures(cs["z"], noisy)
    np.testing.assert_array_equal(alt["tau"], base["tau"])
    wrong = orc.fit_temperatures(cs["z"][:, 1:2], noisy[:, 1:2])  # position 1 on every sample
    assert abs(wrong["tau"][0] - base["tau"][1]) > 0.05
    none = orc.fit_temperatures(cs["z"], np.zeros_like(cs["accepted"]))
    assert none["count"][1] == 0 and none["tau"][1] == 1.0 and none["tau"][2] == 1.0
