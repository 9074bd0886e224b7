"""Pins for the oracle's Markov-head block draft.

Sources: DSpark explainer (papers.franksyz.com mainline topic 31) section 6
(parallel backbone gives base logits, a light sequential head conditions on
the anchor and the sampled in-block prefix) and section 7 (drafter logits =
U_k + B_k; the Markov head looks only at the previous token through a low-rank
factorisation); llama.cpp PR 25173 description (anchor-first block, bias(prev)
= markov_w2 . markov_w1[prev], sampled left to right).
"""
import numpy as np
import pytest
from scipy import stats

from speculative_decoding_dspark_gb300 import inputs


def _bf16_decode(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_markov_bias_is_gemv(orc, dtype):
    """b = W2 @ W1[prev] (rows of both factors are rank-vectors), against numpy."""
    w = inputs.workload("batched_sampling", R=2, V=333, gamma=2, rank=24, w_dtype=dtype)
    d = inputs.draft_inputs(w)
    dec = _bf16_decode if dtype == "bf16" else (lambda a: a.astype(np.float64))
    W1, W2 = dec(d["W1"]), dec(d["W2"])
    for prev in [0, 7, 332]:
        ref = W2 @ W1[prev]
        np.testing.assert_allclose(orc.markov_bias(d["W1"], d["W2"], prev), ref, rtol=1e-12, atol=1e-15)
        # the transposed reading (W1 @ W2[prev]) is a different vector
        assert not np.allclose(W1 @ W2[prev], ref)
    assert np.all(orc.markov_bias(d["W1"], d["W2"], -1) == 0.0)


def test_logsumexp_closed_forms(orc):
    for V in [1, 64, 151936]:
        assert orc.logsumexp(np.full(V, 2.5)) == pytest.approx(2.5 + np.log(V), rel=1e-13)
    x = np.array([1000.0, -np.inf, 1000.0])
    assert orc.logsumexp(x) == pytest.approx(1000.0 + np.log(2.0), rel=1e-15)
    s = orc.softmax(np.array([0.0, np.log(3.0)]))
    np.testing.assert_allclose(s, [0.25, 0.75], rtol=1e-14)


def _draft_numpy_greedy(d, W1, W2, U):
    R, gamma, V = U.shape
    y = np.zeros((R, gamma), np.int64)
    for r in range(R):
        prev = int(d["anchor"][r])
        for k in range(gamma):
            s = U[r, k] + (W2 @ W1[prev] if prev >= 0 else 0.0)
            y[r, k] = int(np.argmax(s))
            prev = y[r, k]
    return y


def test_greedy_draft_is_semi_autoregressive_argmax(orc):
    """T = 0: y_k = argmax(U_k + W2 W1[y_{k-1}]), y_{-1} = anchor."""
    w = inputs.workload("qwen3_8b_greedy", R=4, V=700, gamma=6, rank=32, w_sigma=0.4)
    d = inputs.draft_inputs(w)
    out = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], 0, 0.0)
    ref = _draft_numpy_greedy(d, _bf16_decode(d["W1"]), _bf16_decode(d["W2"]), _bf16_decode(d["U"]))
    assert (out["y"] == ref).all()
    # the chain really depends on the previous token: a different anchor changes position 0
    d2 = dict(d, anchor=(d["anchor"] + 1) % w["V"])
    out2 = orc.markov_draft(d["U"], d["W1"], d["W2"], d2["anchor"], d["seeds"], 0, 0.0)
    assert not np.array_equal(out["q_logits"][:, 0], out2["q_logits"][:, 0])


def test_draft_logits_and_stats(orc):
    """q_logits = (U_k + bias(prev)) * invT, q_lse = logsumexp, q_tok = q(y)."""
    w = inputs.workload("batched_sampling", R=3, V=257, gamma=4, rank=16, w_sigma=0.3)
    d = inputs.draft_inputs(w)
    T = float(w["temperature"])
    invT = float(np.float32(1.0) / np.float32(T))
    out = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], 5, T)
    W1, W2, U = _bf16_decode(d["W1"]), _bf16_decode(d["W2"]), _bf16_decode(d["U"])
    for r in range(3):
        prev = int(d["anchor"][r])
        for k in range(4):
            s = (U[r, k] + W2 @ W1[prev]) * invT
            np.testing.assert_allclose(out["q_logits"][r, k], s, rtol=1e-12, atol=1e-12)
            lse = np.log(np.exp(s - s.max()).sum()) + s.max()
            assert out["q_lse"][r, k] == pytest.approx(lse, rel=1e-12)
            y = out["y"][r, k]
            assert out["q_tok"][r, k] == pytest.approx(np.exp(s[y] - lse), rel=1e-12)
            prev = int(y)
    # anchor < 0: no bias at position 0
    out0 = orc.markov_draft(d["U"], d["W1"], d["W2"], np.full(3, -1), d["seeds"], 5, T)
    np.testing.assert_allclose(out0["q_logits"][:, 0], U[:, 0] * invT, rtol=1e-13)


@pytest.mark.parametrize("V,n,sigma", [(12, 6000, 1.5), (40, 12000, 1.0), (300, 30000, 0.4)])
def test_gumbel_max_draws_follow_softmax(orc, V, n, sigma):
    """At T = 0.7 the drafted token's frequencies over n cycles match
    softmax(U * invT): chi-square over the entries and over the 16-entry
    segments whose race decides the draw.  V = 12 is one segment (the draw is
    the in-segment pick alone), V = 40 three (the last one ragged), V = 300 three
    128-entry blocks (segments j and j + 4 of a block share a Philox counter).
    A wrong word (race and pick from one word, or two segments from one word),
    an off-by-one in the running sum or a sign error in the noise fails here."""
    g = np.random.default_rng(11 + V)
    U = g.normal(0, sigma, (1, 1, V)).astype(np.float32)
    W = np.zeros((V, 4), np.float32)
    T = 0.7
    invT = float(np.float32(1.0) / np.float32(T))
    ys = np.array([orc.markov_draft(U, W, W, [-1], [123], c, T, want_logits=False)["y"][0, 0]
                   for c in range(n)])
    counts = np.bincount(ys, minlength=V)
    p = orc.softmax(U[0, 0].astype(np.float64) * invT)
    chi2 = ((counts - n * p) ** 2 / (n * p)).sum()
    assert stats.chi2.sf(chi2, V - 1) > 1e-3, chi2
    n_seg = (V + 15) // 16
    if n_seg > 1:
        seg_counts = np.add.reduceat(counts, np.arange(0, V, 16))
        seg_p = np.add.reduceat(p, np.arange(0, V, 16))
        chi2s = ((seg_counts - n * seg_p) ** 2 / (n * seg_p)).sum()
        assert stats.chi2.sf(chi2s, n_seg - 1) > 1e-3, chi2s
    # a sign error in the noise (argmin-like sampling) would favour the least likely token
    assert counts[np.argmax(p)] > counts[np.argmin(p)]


def test_draft_draw_is_argmax_of_its_segment_race(orc):
    """Where one entry holds nearly all of the weight, every draw is that entry
    (the race and the in-segment pick both follow the weight); where two
    segments hold equal weight and the rest none, each wins about half the
    time, independently of the block layout."""
    V = 256
    T = 1.0
    W = np.zeros((V, 4), np.float32)
    U = np.full((1, 1, V), -200.0, np.float32)
    U[0, 0, 77] = 0.0
    ys = [orc.markov_draft(U, W, W, [-1], [5], c, T, want_logits=False)["y"][0, 0] for c in range(200)]
    assert set(ys) == {77}
    for a, b in [(3, 200), (21, 85)]:  # slots of different blocks; slots j and j + 4 of one block
        U = np.full((1, 1, V), -200.0, np.float32)
        U[0, 0, a] = 0.0
        U[0, 0, b] = 0.0
        ys = np.array([orc.markov_draft(U, W, W, [-1], [9], c, T, want_logits=False)["y"][0, 0]
                       for c in range(4000)])
        assert set(np.unique(ys)) <= {a, b}
        frac = float(np.mean(ys == a))
        assert abs(frac - 0.5) < 4 * np.sqrt(0.25 / 4000), (a, b, frac)


def test_draft_margin_reports_near_decisions(orc):
    """The margin is the smaller of the race gap between the two best segments
    and the distance of the pick from the running sums around the drawn token:
    zero-margin cases cannot occur in general position, and an entry that
    holds all the weight of a one-segment vocabulary leaves the pick a margin
    equal to how far a W is from either end."""
    V = 8
    W = np.zeros((V, 4), np.float32)
    U = np.full((1, 1, V), -400.0, np.float32)
    U[0, 0, 5] = 0.0
    for c in range(20):
        out = orc.markov_draft(U, W, W, [-1], [3], c, 1.0, want_logits=False)
        assert out["y"][0, 0] == 5
        a = orc.philox4x32_10([0, 0, 0, (c << 4) | 0], 3)[1]
        a = orc.uniform_from_bits(int(a))
        assert out["margin"][0, 0] == pytest.approx(min(a, 1.0 - a), abs=1e-12)


def test_request_subset_replays_batch(orc):
    """req_ids lets a subset of requests be replayed with the batch's random counters."""
    w = inputs.workload("batched_sampling", R=5, V=200, gamma=3, rank=8)
    d = inputs.draft_inputs(w)
    full = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], 2, 0.7)
    sub = [1, 4]
    part = orc.markov_draft(d["U"][sub], d["W1"], d["W2"], d["anchor"][sub], d["seeds"][sub], 2, 0.7,
                            req_ids=sub)
    assert (part["y"] == full["y"][sub]).all()
    np.testing.assert_array_equal(part["q_lse"], full["q_lse"][sub])


# ---------------------------------------------------------------------------
# Fused drafter logits: the base logits come from the drafter's hidden states
# and the shared lm_head (explainer section 6: the parallel backbone gives every
# block position its hidden state in one pass; PR 25173 description: the drafter
# shares the target's lm_head), U[r,k,v] = <W_lm[v], h[r,k]>.

def _fused_case(V=520, d=64, R=3, gamma=4, rank=16, T=0.7, seed=0):
    w = inputs.workload("fused_logits", seed_offset=seed, R=R, V=V, gamma=gamma, rank=rank, d=d,
                        w_sigma=0.3, temperature=T)
    return w, inputs.fused_inputs(w)


@pytest.mark.parametrize("T", [0.7, 0.0])
def test_fused_draft_reduces_to_markov_draft_with_one_hot_lm_head(orc, T):
    """With W_lm[v] the unit vector e_{(3v+1) mod d}, U[r,k,v] = h[r,k,(3v+1) mod d] exactly:
    the fused draft must equal the pinned Markov draft given those base logits, output
    for output (a wrong position, a transposed lm_head or a dropped bias all break it)."""
    w, f = _fused_case(T=T)
    V, d = w["V"], w["d"]
    one = np.uint16(0x3F80)  # 1.0 in bf16
    col = (3 * np.arange(V) + 1) % d
    W_lm = np.zeros((V, d), np.uint16)
    W_lm[np.arange(V), col] = one
    U = np.ascontiguousarray(f["h"][:, :, col])  # bf16 bits, exact
    got = orc.fused_draft(f["h"], W_lm, f["W1"], f["W2"], f["anchor"], f["seeds"], 9, T)
    ref = orc.markov_draft(U, f["W1"], f["W2"], f["anchor"], f["seeds"], 9, T)
    assert got["status"] == 0 and ref["status"] == 0
    np.testing.assert_array_equal(got["y"], ref["y"])
    np.testing.assert_array_equal(got["q_logits"], ref["q_logits"])
    np.testing.assert_array_equal(got["q_lse"], ref["q_lse"])
    np.testing.assert_array_equal(got["margin"], ref["margin"])
    # the h of another position gives other base logits
    U_shift = np.ascontiguousarray(np.roll(f["h"], 1, axis=1)[:, :, col])
    other = orc.markov_draft(U_shift, f["W1"], f["W2"], f["anchor"], f["seeds"], 9, T)
    assert not np.array_equal(other["q_logits"], got["q_logits"])


def test_fused_draft_logits_are_one_contraction(orc):
    """q_logits[r,k] = ([W_lm | W2] @ [h[r,k]; W1[prev]]) * invT with prev the anchor or the
    previous draft, against numpy in float64; with V == d the transposed lm_head reading
    gives a different vector."""
    w, f = _fused_case(V=256, d=256, rank=32)
    T = float(w["temperature"])
    invT = float(np.float32(1.0) / np.float32(T))
    out = orc.fused_draft(f["h"], f["W_lm"], f["W1"], f["W2"], f["anchor"], f["seeds"], 4, T)
    h, Wl = _bf16_decode(f["h"]), _bf16_decode(f["W_lm"])
    W1, W2 = _bf16_decode(f["W1"]), _bf16_decode(f["W2"])
    K = np.concatenate([Wl, W2], axis=1)
    for r in range(w["R"]):
        prev = int(f["anchor"][r])
        for k in range(w["gamma"]):
            x = np.concatenate([h[r, k], W1[prev]])
            np.testing.assert_allclose(out["q_logits"][r, k], (K @ x) * invT, rtol=1e-12, atol=1e-12)
            wrong = (np.concatenate([Wl.T, W2], axis=1) @ x) * invT
            assert not np.allclose(out["q_logits"][r, k], wrong)
            prev = int(out["y"][r, k])


def test_fused_draft_subset_replays_requests(orc):
    """Rows given with req_ids draw the same tokens as in the whole batch (the subset mode the
    full-size GPU tests replay)."""
    w, f = _fused_case(R=5)
    T = float(w["temperature"])
    full = orc.fused_draft(f["h"], f["W_lm"], f["W1"], f["W2"], f["anchor"], f["seeds"], 2, T)
    ids = np.array([1, 4], np.int32)
    sub = orc.fused_draft(f["h"][ids], f["W_lm"], f["W1"], f["W2"], f["anchor"][ids], f["seeds"][ids], 2, T,
                          req_ids=ids)
    np.testing.assert_array_equal(sub["y"], full["y"][ids])
    np.testing.assert_array_equal(sub["q_logits"], full["q_logits"][ids])
