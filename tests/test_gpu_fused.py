"""GPU parity of the fused drafter logits (dspark_markov_draft_fused) against the
oracle's draft from hidden states: the drafter's logits of position k are
[W_lm | W2] . [h_k ; W1[prev]] in one contraction (explainer section 6: the
parallel backbone gives the hidden states, the base logits come from them;
PR 25173 description: the drafter shares the target's lm_head,
bias(prev) = markov_w2 . markov_w1[prev]).

The contraction is (d + rank) / 16 tensor-core MMAs into one fp32 accumulator
(288 at d = 4096, rank 512, against 32 for the Markov draft alone), so the
tolerances follow from a bound on that accumulation (parity_helpers.
fused_logit_tol): logits element by element within it, q_lse within its value
at the row's largest logit (delta), q(y) within 2 delta q(y) (at least 1e-5),
tokens exactly except where the oracle's margin is within 2 delta.
Markov factors at w_sigma 0.2 make the bias large enough to move the draws.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import parity_helpers as H  # noqa: E402
from speculative_decoding_dspark_gb300 import inputs  # noqa: E402


@pytest.fixture(scope="module")
def B():
    from speculative_decoding_dspark_gb300 import build
    build.build()
    from speculative_decoding_dspark_gb300 import binding
    return binding


def _case(seed=0, **over):
    w = inputs.workload("fused_logits", seed_offset=seed, **over)
    return w, inputs.fused_inputs(w)


def _compare(tally, g, o, T, w, rows=None, want_logits=True):
    """Tokens, q(y), log-normalisers and (if the GPU kept them) the scaled logits of the
    oracle's requests (o always holds the oracle's logits, which the bounds are taken on).  The tolerances follow from the logit bound of H.fused_logit_tol, taken
    at the row's largest logit (delta): a draw is exempt when the oracle's margin
    is within 2 delta (both sides of a near tie may move by delta); q_lse may move by
    delta, q(y) by 2 delta q(y) (and never needs to be closer than 1e-5)."""
    R, gamma = o["y"].shape
    invT = 1.0 if T == 0 else float(np.float32(1.0) / np.float32(T))
    sigma_s = w["u_sigma"] * invT
    ql = H.host(g["q_logits_dev"]) if want_logits else None
    clean = set()
    for i in range(R):
        gi = i if rows is None else rows[i]
        ok = True
        for k in range(gamma):
            tally.decisions += 1
            x = o["q_logits"][i, k]
            delta = float(H.fused_logit_tol(np.abs(x).max(), w["d"], w["rank"], sigma_s))
            if g["y"][gi, k] != o["y"][i, k]:
                if o["margin"][i, k] <= max(H.MARGIN, 2 * delta):
                    tally.exempt += 1
                else:
                    tally.errors.append(("draft token", gi, k, int(g["y"][gi, k]), int(o["y"][i, k]),
                                         float(o["margin"][i, k])))
                ok = False
                break
            if T > 0:
                qt = o["q_tok"][i, k]
                if abs(g["q_tok"][gi, k] - qt) > max(H.PROB_TOL, 2 * delta * qt):
                    tally.errors.append(("q_tok", gi, k, float(g["q_tok"][gi, k]), float(qt)))
                if abs(g["q_lse"][gi, k] - o["q_lse"][i, k]) > max(H.LSE_TOL * abs(o["q_lse"][i, k]), delta):
                    tally.errors.append(("q_lse", gi, k, float(g["q_lse"][gi, k]), float(o["q_lse"][i, k])))
            if want_logits:
                tol = H.fused_logit_tol(x, w["d"], w["rank"], sigma_s)
                err = np.abs(ql[gi, k].astype(np.float64) - x)
                if not (err <= tol).all():
                    v = int(np.argmax(err - tol))
                    tally.errors.append(("q_logits", gi, k, v, float(ql[gi, k, v]), float(x[v]),
                                         float(tol[v])))
        if ok:
            clean.add(i)
    return clean


@pytest.mark.parametrize("T", [0.7, 0.0])
@pytest.mark.parametrize("R,V,d,rank", [(8, 4104, 256, 64), (37, 2056, 64, 128), (3, 1032, 1024, 512)])
def test_fused_draft_small(B, orc, T, R, V, d, rank):
    """Every request and every vocabulary entry, ragged last tile (V % 128 == 8), two cycles;
    lm_head parts of 1 to 16 k-blocks ahead of 1 to 8 Markov k-blocks."""
    w, f = _case(R=R, V=V, gamma=3, rank=rank, d=d, w_sigma=0.2, temperature=T)
    tally = H.Tally()
    for cycle in range(2):
        g = H.gpu_fused_draft(f, T, cycle)
        assert g["status"] == 0
        o = orc.fused_draft(f["h"], f["W_lm"], f["W1"], f["W2"], f["anchor"], f["seeds"], cycle, T)
        clean = _compare(tally, g, o, T, w)
        assert len(clean) >= R - 1, (len(clean), R)
    tally.check()


def test_fused_draft_two_request_blocks(B, orc):
    """R = 130: two 128-request blocks (the second with two rows), rank 512, the h box past
    the last request zero-filled; called with q_logits and with q_logits = NULL."""
    R, V, d, rank, T = 130, 16392, 512, 512, 1.0
    w, f = _case(seed=1, R=R, V=V, gamma=3, rank=rank, d=d, w_sigma=0.2, temperature=T)
    bias = orc.markov_bias(f["W1"], f["W2"], int(f["anchor"][0]))
    assert bias.std() > 0.5, bias.std()
    tally = H.Tally()
    for cycle, want in ((0, True), (1, False)):
        g = H.gpu_fused_draft(f, T, cycle, want_logits=want)
        assert g["status"] == 0
        o = orc.fused_draft(f["h"], f["W_lm"], f["W1"], f["W2"], f["anchor"], f["seeds"], cycle, T)
        clean = _compare(tally, g, o, T, w, want_logits=want)
        assert len(clean) >= R - 2, len(clean)
    tally.check()


def test_fused_draft_full_size_sampled(B, orc):
    """The fused_logits workload at full size (R = 128, V = 151936, gamma = 7, d = 4096,
    rank 512, T = 0.7): the whole batch on the GPU, without and then with q_logits;
    requests from every tensor-memory lane quadrant replayed on the oracle, chosen per call."""
    w, f = _case()
    T = float(w["temperature"])
    t = {k: H.dev(f[k]) for k in ("h", "W_lm", "W1", "W2", "anchor", "seeds")}
    tally = H.Tally()
    for cycle, want, rows in ((0, False, [5, 70]), (1, True, [33, 127])):
        g = H.gpu_fused_draft(f, T, cycle, want_logits=want, dev_inputs=t)
        assert g["status"] == 0
        assert (g["y"] >= 0).all() and (g["y"] < w["V"]).all()
        assert np.isfinite(g["q_lse"]).all() and ((g["q_tok"] > 0) & (g["q_tok"] <= 1)).all()
        o = orc.fused_draft(f["h"][rows], f["W_lm"], f["W1"], f["W2"], f["anchor"][rows], f["seeds"][rows],
                            cycle, T, req_ids=rows)
        _compare(tally, g, o, T, w, rows=rows, want_logits=want)
    tally.check()


def test_fused_draft_refusals(B):
    """Shapes the tensor-core kernel does not take are refused before anything is enqueued."""
    import ctypes
    L = B.library()
    fake = ctypes.c_void_p(256)
    args = lambda d, rank, V: (fake, fake, d, fake, fake, fake, fake, 0, 1.0, 8, 3, V, rank,
                               fake, fake, fake, None, fake, 1 << 20, None, None)
    assert L.dspark_markov_draft_fused(*args(100, 64, 4096)) == B.DSPARK_ERR_UNSUPPORTED  # d % 64
    assert L.dspark_markov_draft_fused(*args(B.DSPARK_FUSED_MAX_D + 64, 64, 4096)) == B.DSPARK_ERR_UNSUPPORTED
    assert L.dspark_markov_draft_fused(*args(256, 576, 4096)) == B.DSPARK_ERR_UNSUPPORTED  # rank > 512
    assert L.dspark_markov_draft_fused(*args(256, 64, 4100)) == B.DSPARK_ERR_UNSUPPORTED  # V % 8
    assert L.dspark_markov_draft_fused(*args(0, 64, 4096)) == B.DSPARK_ERR_INVALID_ARG


def test_fused_draft_anchor_edge_cases(B, orc):
    """anchor -1: no bias at position 0 (the other reading of the anchor-first block); an
    anchor >= V: that request's tokens are -1 and DSPARK_ERR_DEVICE_INPUT is reported, while
    every other request is drafted as the oracle drafts it."""
    T = 0.7
    w, f = _case(seed=2, R=12, V=2056, gamma=3, rank=64, d=128, w_sigma=0.2, temperature=T)
    anchor = f["anchor"].copy()
    anchor[1] = -1
    anchor[5] = -1
    anchor[7] = w["V"] + 3
    g = H.gpu_fused_draft(dict(f, anchor=anchor), T, 0)
    assert g["status"] == B.DSPARK_ERR_DEVICE_INPUT
    assert (g["y"][7] == -1).all() and np.isnan(g["q_lse"][7]).all()
    rows = [i for i in range(w["R"]) if i != 7]
    o = orc.fused_draft(f["h"][rows], f["W_lm"], f["W1"], f["W2"], anchor[rows], f["seeds"][rows], 0, T,
                        req_ids=rows)
    tally = H.Tally()
    clean = _compare(tally, g, o, T, w, rows=rows)
    tally.check()
    assert len(clean) >= len(rows) - 1


def test_fused_draft_four_request_blocks_sampled(B, orc):
    """R = 512 (four request blocks over the same vocabulary tiles, the tensor-bound case the
    bench times), V = 129280, gamma = 5, d = 4096, rank 512, T = 1: the whole batch on the
    GPU, one request of every block replayed on the oracle."""
    w, f = _case(seed=3, R=512, V=129280, gamma=5, temperature=1.0)
    T = 1.0
    g = H.gpu_fused_draft(f, T, 4, want_logits=False)
    assert g["status"] == 0
    assert (g["y"] >= 0).all() and (g["y"] < w["V"]).all()
    rows = [1, 200, 300, 511]
    o = orc.fused_draft(f["h"][rows], f["W_lm"], f["W1"], f["W2"], f["anchor"][rows], f["seeds"][rows], 4, T,
                        req_ids=rows)
    tally = H.Tally()
    _compare(tally, g, o, T, w, rows=rows, want_logits=False)
    tally.check()
