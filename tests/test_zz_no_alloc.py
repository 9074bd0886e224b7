"""dspark_verify_static_scratch: verify for callers that cannot allocate.

Some callers are not allowed to allocate device memory (for example a plugin
inside a serving engine whose device memory all belongs to the engine's own
pool), so they cannot pass a workspace.  This entry point takes its scratch
from a fixed array compiled into the library.  The test calls it through the C
ABI twice in a row and checks each result against dspark_verify with a
caller-provided workspace on the same inputs.

This file is named so that pytest collects it after every other test file.
"""
import ctypes

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


def _case(seed_offset, varlen):
    name = "varlen_verify" if varlen else "batched_sampling"
    w, d = H.cycle_inputs(name, seed_offset=seed_offset, R=24, V=30000, gamma=5, rank=64, w_sigma=0.2)
    full = inputs.target_full(w, d["U"])
    l = inputs.verify_lengths(w)
    return w, d, H.dev(inputs.pack_rows(full, l)), H.dev(inputs.cu_from_lengths(l)), int(l.sum() + len(l))


def _verify_both(B, target, cu, g, seeds, cycle, T, max_rows):
    R, gamma = g["y_dev"].shape
    V = target.shape[1]
    outs = []
    for static in (False, True):
        n_acc = torch.full((R,), -7, dtype=torch.int32, device="cuda")
        out = torch.full((R, gamma + 1), -7, dtype=torch.int32, device="cuda")
        p_tok = torch.full((R, gamma), float("nan"), device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        args = (target, cu, g["y_dev"], g["q_logits_dev"] if T > 0 else None,
                g["q_lse_dev"] if T > 0 else None, g["q_tok_dev"] if T > 0 else None,
                seeds if T > 0 else None, cycle, T, max_rows, n_acc, out, p_tok)
        if static:
            B.dspark_verify_static_scratch(*args, dev_status=status)
        else:
            ws = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_VERIFY, R, gamma, V, 0, max_rows))
            B.dspark_verify(*args, ws=ws, dev_status=status)
        torch.cuda.synchronize()
        outs.append(dict(n_acc=H.host(n_acc), out=H.host(out), p_tok=H.host(p_tok), status=int(status.item())))
    return outs


def test_static_scratch_matches_workspace_verify_twice(B):
    # two sampling calls in a row, then a greedy one (which writes its tokens
    # from the decision pass and skips the draw kernel) on the array the
    # sampling calls left behind
    for call, (seed, varlen, T) in enumerate([(0, False, 0.7), (1, True, 1.0), (2, True, 0.0)]):
        w, d, target, cu, rows = _case(seed, varlen)
        g = H.gpu_draft(d, T, call)
        ref, got = _verify_both(B, target, cu, g, H.dev(d["seeds"]), call, T, rows)
        assert ref["status"] == 0 and got["status"] == 0
        np.testing.assert_array_equal(got["n_acc"], ref["n_acc"])
        np.testing.assert_array_equal(got["out"], ref["out"])
        if T == 0:
            assert set(np.unique(got["p_tok"][~np.isnan(got["p_tok"])])) <= {0.0, 1.0}
        examined = ~np.isnan(ref["p_tok"])
        np.testing.assert_array_equal(examined, ~np.isnan(got["p_tok"]))
        np.testing.assert_allclose(got["p_tok"][examined], ref["p_tok"][examined], rtol=0, atol=H.PROB_TOL)
        assert (ref["n_acc"] >= 0).all()


def test_static_scratch_rejects_oversized_requests(B):
    L = B.library()
    fake = ctypes.c_void_p(256)
    # 4096 requests of 7 drafts over a 151936-entry vocabulary need far more than 4 MiB
    st = L.dspark_verify_static_scratch(fake, fake, fake, fake, fake, fake, fake, 0, 1.0, 4096, 7,
                                        151936, 4096 * 8, fake, fake, None, None, None)
    assert st == B.DSPARK_ERR_CAPACITY
    assert B.dspark_workspace_size(B.DSPARK_OP_VERIFY, 4096, 7, 151936, 0, 4096 * 8) > 4 * 1024 * 1024
    # the largest batches that fit: 772 requests at V = 151936, 905 at V = 129280
    for R, V in ((772, 151936), (905, 129280)):
        assert B.dspark_workspace_size(B.DSPARK_OP_VERIFY, R, 7, V, 0, R * 8) <= 4 * 1024 * 1024
        assert B.dspark_workspace_size(B.DSPARK_OP_VERIFY, R + 1, 7, V, 0, (R + 1) * 8) > 4 * 1024 * 1024
