"""Failure handling on the GPU without a fault: the grid-wide waits of the
cooperative launches give up after a limit and the call reports
DSPARK_ERR_TIMEOUT, leaves the outputs alone and keeps the context usable
(DSpark explainer section 16: a failure must fall back, not hang).

The waits are made to run out by the library's test injection: the barrier
counts one arrival more than the grid has, so nobody is released and every
CTA's wait ends at the limit (20 ms here).  Every test checks that a normal
call afterwards gives the same results as before.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import parity_helpers as H  # noqa: E402
from speculative_decoding_dspark_gb300 import inputs  # noqa: E402

LIMIT_NS = 20_000_000


@pytest.fixture(scope="module")
def B():
    from speculative_decoding_dspark_gb300 import build
    build.build()
    from speculative_decoding_dspark_gb300 import binding
    return binding


class injected:
    """Within the block: the named barrier never releases, waits give up after LIMIT_NS."""

    def __init__(self, B, mask):
        self.B, self.mask = B, mask

    def __enter__(self):
        self.B.dspark_set_wait_limit_ns(LIMIT_NS)
        self.B.dspark_set_fault_injection(self.mask)

    def __exit__(self, *exc):
        self.B.dspark_set_fault_injection(0)
        self.B.dspark_set_wait_limit_ns(0)
        return False


def _case(T):
    name = "batched_sampling" if T > 0 else "qwen3_8b_greedy"
    w, d = H.cycle_inputs(name, R=24, V=20000, gamma=4, rank=64, w_sigma=0.2)
    full = inputs.target_full(w, d["U"])
    l = inputs.verify_lengths(w)
    return w, d, H.dev(inputs.pack_rows(full, l)), H.dev(inputs.cu_from_lengths(l))


def _same(a, b):
    np.testing.assert_array_equal(a["n_acc"], b["n_acc"])
    np.testing.assert_array_equal(a["out_tokens"], b["out_tokens"])


@pytest.mark.parametrize("T", [0.7, 0.0])
def test_verify_barrier_timeout(B, T):
    w, d, target, cu = _case(T)
    g = H.gpu_draft(d, T, 0)
    samp = T > 0
    args = lambda: (target, cu, g["y_dev"], g["q_logits_dev"] if samp else None,
                    g["q_lse_dev"] if samp else None, g["q_tok_dev"] if samp else None,
                    H.dev(d["seeds"]) if samp else None, 0, T)
    ref = H.gpu_verify(*args())
    ref_m = H.gpu_verify_markov(target, cu, d, g, 0, T)
    assert ref["status"] == 0 and ref_m["status"] == 0
    with injected(B, B.DSPARK_INJECT_VERIFY_BARRIER):
        bad = H.gpu_verify(*args())
        bad_m = H.gpu_verify_markov(target, cu, d, g, 0, T)
    for b in (bad, bad_m):
        assert b["status"] == B.DSPARK_ERR_TIMEOUT
        # nothing was decided: the outputs keep the values they were filled with
        assert (b["n_acc"] == -7).all() and (b["out_tokens"] == -7).all()
    _same(H.gpu_verify(*args()), ref)
    _same(H.gpu_verify_markov(target, cu, d, g, 0, T), ref_m)


def test_draft_barrier_timeout(B):
    w, d, _, _ = _case(0.7)
    ref = H.gpu_draft(d, 0.7, 2, want_logits=False)
    assert ref["status"] == 0
    with injected(B, B.DSPARK_INJECT_DRAFT_BARRIER):
        bad = H.gpu_draft(d, 0.7, 2, want_logits=False)
    assert bad["status"] == B.DSPARK_ERR_TIMEOUT
    assert (bad["y"] == -7).all() and np.isnan(bad["q_lse"]).all() and np.isnan(bad["q_tok"]).all()
    again = H.gpu_draft(d, 0.7, 2, want_logits=False)
    assert again["status"] == 0
    np.testing.assert_array_equal(again["y"], ref["y"])
    np.testing.assert_array_equal(again["q_lse"], ref["q_lse"])


def test_fused_draft_barrier_timeout(B):
    """The fused drafter logits share the draft's grid barrier between positions."""
    w = inputs.workload("fused_logits", R=24, V=8192, gamma=4, rank=64, d=256, w_sigma=0.2)
    f = inputs.fused_inputs(w)
    ref = H.gpu_fused_draft(f, 0.7, 2, want_logits=False)
    assert ref["status"] == 0
    with injected(B, B.DSPARK_INJECT_DRAFT_BARRIER):
        bad = H.gpu_fused_draft(f, 0.7, 2, want_logits=False)
    assert bad["status"] == B.DSPARK_ERR_TIMEOUT
    assert (bad["y"] == -7).all() and np.isnan(bad["q_lse"]).all() and np.isnan(bad["q_tok"]).all()
    again = H.gpu_fused_draft(f, 0.7, 2, want_logits=False)
    assert again["status"] == 0
    np.testing.assert_array_equal(again["y"], ref["y"])
    np.testing.assert_array_equal(again["q_lse"], ref["q_lse"])


def test_static_scratch_timeout_after_a_normal_call(B):
    """The shared static scratch keeps the previous call's per-request rows; a
    call whose decision pass gives up must not draw from them."""
    T = 0.7
    w, d, target, cu = _case(T)
    g = H.gpu_draft(d, T, 1)
    R, gamma = g["y_dev"].shape
    max_rows = int(target.shape[0])

    def call():
        G = H.Guarded()
        n_acc = G.out((R,), torch.int32, -7)
        out = G.out((R, gamma + 1), torch.int32, -7)
        status = G.out((1,), torch.int32, 0)
        B.dspark_verify_static_scratch(target, cu, g["y_dev"], g["q_logits_dev"], g["q_lse_dev"],
                                       g["q_tok_dev"], H.dev(d["seeds"]), 1, T, max_rows, n_acc, out,
                                       dev_status=status)
        torch.cuda.synchronize()
        G.check()
        return dict(n_acc=H.host(n_acc), out_tokens=H.host(out), status=int(status.item()))

    ref = call()
    assert ref["status"] == 0
    with injected(B, B.DSPARK_INJECT_VERIFY_BARRIER):
        bad = call()
    assert bad["status"] == B.DSPARK_ERR_TIMEOUT
    assert (bad["n_acc"] == -7).all() and (bad["out_tokens"] == -7).all()
    _same(call(), ref)


def test_wait_settings_round_trip(B):
    assert B.dspark_set_wait_limit_ns(5_000_000) == 2_000_000_000
    assert B.dspark_set_wait_limit_ns(0) == 5_000_000
    assert B.dspark_set_wait_limit_ns(0) == 2_000_000_000
    assert B.dspark_set_fault_injection(3) == 0
    assert B.dspark_set_fault_injection(0) == 3
