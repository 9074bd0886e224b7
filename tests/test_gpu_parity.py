"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.

Small cases compare every element; they span several vocabulary tiles and
chunks with a ragged tail.  The full-size workloads run the whole batch on the
GPU and replay a sample of requests on the oracle (the draft and verify of a
request depend only on that request's inputs and counters), while the
selection is compared on every candidate.
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


# ------------------------------------------------------------------ generator
def test_philox_bit_exact(B, orc):
    g = np.random.default_rng(5)
    n = 1 << 20
    ctr = g.integers(0, 1 << 32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    keys = g.integers(0, 1 << 63, size=n, dtype=np.uint64) * np.uint64(2) + np.uint64(1)
    out = torch.zeros((n, 4), dtype=torch.int32, device="cuda")
    B.dspark_philox4x32_10(H.dev(ctr).view(torch.int32), H.dev(keys), out)
    torch.cuda.synchronize()
    ref = orc.philox4x32_10_batch(ctr, keys)
    np.testing.assert_array_equal(H.host(out).view(np.uint32), ref)


# ------------------------------------------------------------------ draft
DRAFT_CASES = [
    # name, overrides, temperature, flags
    ("tiny_exhaustive", {}, 1.0, 0),
    ("tiny_exhaustive", {}, 0.0, 0),
    ("batched_sampling", dict(R=6, V=17416, gamma=4, rank=64, w_sigma=0.2), 0.7, 1),
    ("batched_sampling", dict(R=6, V=17416, gamma=4, rank=64, w_sigma=0.2), 0.7, 0),
    ("batched_sampling", dict(R=3, V=9001, gamma=3, rank=40, w_sigma=0.2), 1.0, 0),
    ("qwen3_8b_greedy", dict(R=5, V=20480, gamma=7, rank=128, w_sigma=0.2), 0.0, 0),
    ("qwen3_8b_greedy", dict(R=5, V=20480, gamma=7, rank=128, w_sigma=0.2), 0.0, 1),
    ("batched_sampling", dict(R=130, V=4096, gamma=2, rank=64, w_sigma=0.2), 0.7, 0),
]


@pytest.mark.parametrize("name,over,T,flags", DRAFT_CASES)
def test_draft_parity_small(B, orc, name, over, T, flags):
    w, d = H.cycle_inputs(name, **over)
    tally = H.Tally()
    for cycle in range(3):
        g = H.gpu_draft(d, T, cycle, flags=flags)
        o = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], cycle, T)
        assert g["status"] == 0
        clean = H.compare_draft(tally, g, o, T)
        # q_logits: the scaled logits of every vocabulary entry
        ql = H.host(g["q_logits_dev"])
        for r in clean:
            np.testing.assert_allclose(ql[r], o["q_logits"][r], rtol=2e-6, atol=2e-5)
    tally.check()


def test_draft_path_choice_resident_limit(B):
    """The tensor-core draft runs every position in one launch whose CTAs are
    resident together (one per SM per 128 requests): above that many requests
    the draft takes the CUDA-core kernels instead of failing to launch."""
    import torch
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    bf = B.DSPARK_BF16
    assert B.dspark_markov_draft_uses_tensor_cores(bf, bf, 128 * n_sm, 151936, 512)
    assert not B.dspark_markov_draft_uses_tensor_cores(bf, bf, 128 * n_sm + 1, 151936, 512)


@pytest.mark.parametrize("R,rank,T", [(128, 64, 0.7), (256, 128, 1.0), (100, 64, 0.0)])
def test_draft_multi_tile_elementwise(B, orc, R, rank, T):
    """Full vocabulary with every request row of the tile active: each CTA walks
    many vocabulary tiles, reusing its base-logit buffer and both accumulators.
    The scaled logits of sampled requests match the oracle element by element."""
    w, d = H.cycle_inputs("batched_sampling", R=R, V=151936, gamma=3, rank=rank, w_sigma=0.2)
    g = H.gpu_draft(d, T, 1)
    assert g["status"] == 0
    ql = H.host(g["q_logits_dev"])
    rows = [0, R // 2 + 1, R - 1]
    o = orc.markov_draft(d["U"][rows], d["W1"], d["W2"], d["anchor"][rows], d["seeds"][rows], 1, T,
                         req_ids=rows)
    tally = H.Tally()
    clean = H.compare_draft(tally, g, o, T, rows=rows)
    tally.check()
    for i in clean:
        np.testing.assert_allclose(ql[rows[i]], o["q_logits"][i], rtol=2e-6, atol=2e-5)


def test_draft_rank512_every_request(B, orc):
    """Rank 512 (the bench's Markov rank): A takes 128 KB of shared memory, so
    the W2 ring has four 16 KB stages and each tile's eight k-blocks wrap the
    ring inside the tile.  Factors at w_sigma 0.2 make the bias large enough to
    move the draws (|b| about 0.9 against U's sigma of 3; checked below), so a
    wrong k-block would change tokens and logits.  Every one of 128 requests
    (all four tensor-memory lane quadrants) over 129 vocabulary tiles with a
    ragged 8-column tail, called with q_logits (compared element by element)
    and with q_logits = NULL (the call the bench times)."""
    w, d = H.cycle_inputs("batched_sampling", R=128, V=16392, gamma=3, rank=512, w_sigma=0.2)
    assert B.dspark_markov_draft_uses_tensor_cores(B.DSPARK_BF16, B.DSPARK_BF16, 128, 16392, 512)
    bias = orc.markov_bias(d["W1"], d["W2"], int(d["anchor"][0]))
    assert bias.std() > 0.5, bias.std()
    T = 0.7
    tally = H.Tally()
    for cycle, want in ((0, True), (1, False)):
        g = H.gpu_draft(d, T, cycle, want_logits=want)
        assert g["status"] == 0
        o = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], cycle, T,
                             want_logits=want)
        clean = H.compare_draft(tally, g, o, T)
        assert len(clean) >= 120, len(clean)
        if want:
            ql = H.host(g["q_logits_dev"])
            for r in clean:
                np.testing.assert_allclose(ql[r], o["q_logits"][r], rtol=2e-6, atol=2e-5)
    tally.check()
    print(f"rank-512 draft: {tally.decisions} decisions, {tally.exempt} exempt near ties")


def test_draft_rank512_full_vocab_sampled(B, orc):
    """Rank 512 over the full 151936-entry vocabulary (each CTA walks about eight
    tiles per position, so the four-stage ring also wraps across tiles and
    positions), eight requests spread over the four lane quadrants compared with
    the oracle, with q_logits element by element and with q_logits = NULL."""
    w, d = H.cycle_inputs("batched_sampling", R=128, V=151936, gamma=2, rank=512, w_sigma=0.2)
    T = 0.7
    rows = [0, 9, 31, 32, 63, 64, 100, 127]
    tally = H.Tally()
    for cycle, want in ((0, True), (1, False)):
        g = H.gpu_draft(d, T, cycle, want_logits=want)
        assert g["status"] == 0
        o = orc.markov_draft(d["U"][rows], d["W1"], d["W2"], d["anchor"][rows], d["seeds"][rows], cycle,
                             T, req_ids=rows, want_logits=want)
        clean = H.compare_draft(tally, g, o, T, rows=rows)
        assert len(clean) >= 7, len(clean)
        if want:
            ql = H.host(g["q_logits_dev"])
            for i in clean:
                np.testing.assert_allclose(ql[rows[i]], o["q_logits"][i], rtol=2e-6, atol=2e-5)
    tally.check()


@pytest.mark.parametrize("rank", [64, 512])
def test_draft_w1_alignment_fallback(B, orc, rank):
    """W1 16 bytes past a 32-byte boundary: the tensor-core draft then reads the
    A rows 16 bytes a lane instead of 32.  The outputs equal the aligned call's
    bit for bit, and the oracle's."""
    w, d = H.cycle_inputs("batched_sampling", R=130, V=17416, gamma=3, rank=rank, w_sigma=0.2)
    assert B.dspark_markov_draft_uses_tensor_cores(B.DSPARK_BF16, B.DSPARK_BF16, 130, 17416, rank)
    T = 0.7
    ref = H.gpu_draft(d, T, 4, want_logits=False)
    W1 = H.dev(d["W1"])
    buf = torch.empty(W1.numel() + 8, dtype=torch.bfloat16, device="cuda")
    W1_off = buf[8:].view(W1.shape)
    W1_off.copy_(W1)
    assert W1_off.data_ptr() % 32 == 16
    U, W2 = H.dev(d["U"]), H.dev(d["W2"])
    R, gamma, V = U.shape
    y = torch.full((R, gamma), -7, dtype=torch.int32, device="cuda")
    q_lse = torch.full((R, gamma), float("nan"), device="cuda")
    q_tok = torch.full((R, gamma), float("nan"), device="cuda")
    ws = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_DRAFT, R, gamma, V, rank, 0, B.DSPARK_BF16, 0))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.dspark_markov_draft(U, W1_off, W2, H.dev(d["anchor"]), H.dev(d["seeds"]), 4, T, y, q_lse, q_tok, None, ws,
                          status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    np.testing.assert_array_equal(H.host(y), ref["y"])
    np.testing.assert_array_equal(H.host(q_lse), ref["q_lse"])
    np.testing.assert_array_equal(H.host(q_tok), ref["q_tok"])
    o = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], 4, T, want_logits=False)
    tally = H.Tally()
    H.compare_draft(tally, dict(y=H.host(y), q_lse=H.host(q_lse), q_tok=H.host(q_tok)), o, T)
    tally.check()


def test_draft_tiny_many_cycles(B, orc):
    """The V=64 workload: 2000 cycles at T=1 and 2000 greedy."""
    w, d = H.cycle_inputs("tiny_exhaustive")
    for T in (1.0, 0.0):
        tally = H.Tally()
        for cycle in range(2000):
            g = H.gpu_draft(d, T, cycle, want_logits=False)
            o = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], cycle, T,
                                 want_logits=False)
            H.compare_draft(tally, g, o, T)
        tally.check()


def test_draft_extreme_logit_scale(B, orc):
    """Logits far outside the usual range on the tensor-core draft: with
    u_sigma = 60 and T = 0.02 or 0.001 the base-2 scaled logits reach about 1.7e4
    and 3.5e5, so the weights of later passes sum past 2^32 (the race's reference
    moves) and at T = 0.001 the race records shared between a row's four threads
    saturate their half-precision slot (a looser bound, still a bound).  The
    tokens must match the oracle exactly (the draws are all but deterministic at
    this scale) and the log-normalisers to fp32 relative precision; q(y) is not
    compared here, since exp of the difference of two fp32 values near 1e5
    carries an absolute error of about 1e-2."""
    w, d = H.cycle_inputs("batched_sampling", R=6, V=17416, gamma=4, rank=64, w_sigma=0.2, u_sigma=60.0)
    assert B.dspark_markov_draft_uses_tensor_cores(B.DSPARK_BF16, B.DSPARK_BF16, 6, 17416, 64)
    for T in (0.02, 0.001):
        tally = H.Tally()
        for cycle in range(2):
            g = H.gpu_draft(d, T, cycle, want_logits=False)
            o = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], cycle, T,
                                 want_logits=False)
            assert g["status"] == 0
            clean = H.compare_draft(tally, g, o, 0.0)  # tokens only
            for r in clean:
                np.testing.assert_allclose(g["q_lse"][r], o["q_lse"][r], rtol=1e-5)
        tally.check()


# ------------------------------------------------------------------ verify
def _oracle_draft_as_inputs(o):
    return (o["y"].astype(np.int32), o["q_logits"].astype(np.float32),
            o["q_lse"].astype(np.float32), o["q_tok"].astype(np.float32))


VERIFY_CASES = [
    ("tiny_exhaustive", {}, 1.0),
    ("tiny_exhaustive", {}, 0.0),
    ("batched_sampling", dict(R=7, V=20000, gamma=5, rank=16, w_sigma=0.3), 0.7),
    ("varlen_verify", dict(R=24, V=10007, gamma=5, rank=16, w_sigma=0.3), 1.0),
    ("qwen3_8b_greedy", dict(R=9, V=16390, gamma=7, rank=16, w_sigma=0.3), 0.0),
]


@pytest.mark.parametrize("name,over,T", VERIFY_CASES)
def test_verify_parity_small(B, orc, name, over, T):
    """Verify alone, fed the oracle's own draft (rounded to fp32)."""
    w, d = H.cycle_inputs(name, **over)
    full = inputs.target_full(w, d["U"])
    l = inputs.verify_lengths(w)
    cu = inputs.cu_from_lengths(l)
    target = inputs.pack_rows(full, l)
    tally = H.Tally()
    for cycle in range(4):
        o_d = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], cycle, T)
        y, ql, qlse, qtok = _oracle_draft_as_inputs(o_d)
        o_v = orc.verify(target, cu, y, o_d["q_logits"], d["seeds"], cycle, T)
        g_v = H.gpu_verify(target, cu, y, ql if T > 0 else None, qlse if T > 0 else None,
                           qtok if T > 0 else None, d["seeds"] if T > 0 else None, cycle, T)
        assert g_v["status"] == 0 and o_v["status"] == 0
        H.compare_verify(tally, g_v, o_v, l)
    tally.check()


MARKOV_CASES = [
    ("batched_sampling", dict(R=7, V=20000, gamma=5, rank=64, w_sigma=0.3), 0.7, 4),
    ("varlen_verify", dict(R=24, V=10008, gamma=5, rank=64, w_sigma=0.3), 1.0, 4),
    ("batched_sampling", dict(R=130, V=4096, gamma=3, rank=128, w_sigma=0.3), 1.0, 4),
    ("qwen3_8b_greedy", dict(R=9, V=16392, gamma=7, rank=64, w_sigma=0.3), 0.0, 4),
    # rank 192: 24 sixteen-byte pieces per W1 row (not a power of two); V % 32 != 0
    ("batched_sampling", dict(R=11, V=12008, gamma=4, rank=192, w_sigma=0.3), 0.8, 4),
    # rank 512, the bench's: a four-stage W2 ring that wraps inside every tile,
    # 128 requests (every lane quadrant), a ragged last tile
    ("batched_sampling", dict(R=128, V=16392, gamma=3, rank=512, w_sigma=0.2), 0.7, 2),
]


@pytest.mark.parametrize("name,over,T,cycles", MARKOV_CASES)
def test_verify_markov_parity(B, orc, name, over, T, cycles):
    """Verify with the drafter's logits recomputed on the tensor cores: against
    the oracle, and identical to dspark_verify fed the stored logits."""
    w, d = H.cycle_inputs(name, **over)
    full = inputs.target_full(w, d["U"])
    l = inputs.verify_lengths(w)
    cu = inputs.cu_from_lengths(l)
    target = inputs.pack_rows(full, l)
    tD, cuD = H.dev(target), H.dev(cu)
    tally = H.Tally()
    for cycle in range(cycles):
        g = H.gpu_draft(d, T, cycle)
        gm = H.gpu_verify_markov(tD, cuD, d, g, cycle, T)
        gv = H.gpu_verify(tD, cuD, g["y_dev"], g["q_logits_dev"] if T > 0 else None,
                          g["q_lse_dev"] if T > 0 else None, g["q_tok_dev"] if T > 0 else None,
                          H.dev(d["seeds"]) if T > 0 else None, cycle, T)
        assert gm["status"] == 0 and gv["status"] == 0
        np.testing.assert_array_equal(gm["n_acc"], gv["n_acc"])
        np.testing.assert_array_equal(gm["out_tokens"], gv["out_tokens"])
        o = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], cycle, T)
        ov = orc.verify(target, cu, o["y"], o["q_logits"], d["seeds"], cycle, T)
        clean = H.compare_draft(tally, g, o, T)
        H.compare_verify(tally, gm, ov, l, only=clean)
    tally.check()


HOST_CASES = [
    ("batched_sampling", dict(R=128, V=16392, gamma=3, rank=512, w_sigma=0.2), 0.7),
    ("varlen_verify", dict(R=24, V=10008, gamma=5, rank=64, w_sigma=0.3), 1.0),
    ("qwen3_8b_greedy", dict(R=9, V=16392, gamma=7, rank=64, w_sigma=0.3), 0.0),
]


@pytest.mark.parametrize("name,over,T", HOST_CASES)
def test_verify_markov_host_target(B, orc, name, over, T):
    """Target rows left in pinned host memory, read by the kernels across the host
    link (only the rows up to each first rejection; the residual draw reads the
    device copy the decision pass keeps): the same accepted counts, tokens and
    p(y) as with the rows in device memory, bit for bit, and the same against the
    oracle."""
    w, d = H.cycle_inputs(name, **over)
    full = inputs.target_full(w, d["U"])
    l = inputs.verify_lengths(w)
    cu = inputs.cu_from_lengths(l)
    target = inputs.pack_rows(full, l)
    tD, cuD = H.dev(target), H.dev(cu)
    tH = torch.from_numpy(target).pin_memory()
    tally = H.Tally()
    for cycle in range(2):
        g = H.gpu_draft(d, T, cycle)
        on_dev = H.gpu_verify_markov(tD, cuD, d, g, cycle, T)
        on_host = H.gpu_verify_markov(tH, cuD, d, g, cycle, T, host_target=True)
        assert on_dev["status"] == 0 and on_host["status"] == 0
        for k in ("n_acc", "out_tokens"):
            np.testing.assert_array_equal(on_host[k], on_dev[k])
        np.testing.assert_array_equal(np.isnan(on_host["p_tok"]), np.isnan(on_dev["p_tok"]))
        ok = ~np.isnan(on_dev["p_tok"])
        np.testing.assert_array_equal(on_host["p_tok"][ok], on_dev["p_tok"][ok])
        o = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], cycle, T)
        ov = orc.verify(target, cu, o["y"], o["q_logits"], d["seeds"], cycle, T)
        clean = H.compare_draft(tally, g, o, T)
        H.compare_verify(tally, on_host, ov, l, only=clean)
    tally.check()


def test_host_target_refusals(B):
    """dspark_verify takes device rows only; pageable host memory is refused by
    both verify calls (the device cannot be trusted to read it)."""
    w, d = H.cycle_inputs("batched_sampling", R=4, V=1024, gamma=2, rank=64, w_sigma=0.2)
    full = inputs.target_full(w, d["U"])
    l = inputs.verify_lengths(w)
    target = inputs.pack_rows(full, l)
    g = H.gpu_draft(d, 0.7, 0)
    cuD = H.dev(inputs.cu_from_lengths(l))
    L = B.library()
    vp = ctypes.c_void_p
    n_acc = torch.empty(4, dtype=torch.int32, device="cuda")
    out = torch.empty((4, 3), dtype=torch.int32, device="cuda")
    pinned = torch.from_numpy(target).pin_memory()
    ws1 = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_VERIFY, 4, 2, 1024, 0, 12))
    st = L.dspark_verify(vp(pinned.data_ptr()), vp(cuD.data_ptr()), vp(g["y_dev"].data_ptr()),
                         vp(g["q_logits_dev"].data_ptr()), vp(g["q_lse_dev"].data_ptr()),
                         vp(g["q_tok_dev"].data_ptr()), vp(H.dev(d["seeds"]).data_ptr()), 0, 0.7, 4, 2, 1024, 12,
                         vp(n_acc.data_ptr()), vp(out.data_ptr()), None, vp(ws1.data_ptr()), ws1.numel(), None, None)
    assert st == B.DSPARK_ERR_UNSUPPORTED
    pageable = np.ascontiguousarray(target)
    ws = B.workspace(B.dspark_workspace_size(B.DSPARK_OP_VERIFY_MARKOV, 4, 2, 1024, 64, 12, B.DSPARK_BF16,
                                             B.DSPARK_VERIFY_HOST_TARGET))
    U, W1, W2, anc = H.dev(d["U"]), H.dev(d["W1"]), H.dev(d["W2"]), H.dev(d["anchor"])
    st = L.dspark_verify_markov(vp(pageable.ctypes.data), vp(cuD.data_ptr()), vp(g["y_dev"].data_ptr()),
                                vp(U.data_ptr()), vp(W1.data_ptr()), vp(W2.data_ptr()), vp(anc.data_ptr()), 64,
                                vp(g["q_lse_dev"].data_ptr()), vp(g["q_tok_dev"].data_ptr()),
                                vp(H.dev(d["seeds"]).data_ptr()), 0, 0.7, 4, 2, 1024, 12, vp(n_acc.data_ptr()),
                                vp(out.data_ptr()), None, vp(ws.data_ptr()), ws.numel(), None, None)
    assert st == B.DSPARK_ERR_UNSUPPORTED


def test_verify_tiny_many_cycles(B, orc):
    """The V=64 workload, 2000 full cycles draft -> verify on the GPU vs the oracle."""
    w, d = H.cycle_inputs("tiny_exhaustive")
    full = inputs.target_full(w, d["U"])
    l = inputs.verify_lengths(w)
    cu = inputs.cu_from_lengths(l)
    target = inputs.pack_rows(full, l)
    tD, cuD, seedsD = H.dev(target), H.dev(cu), H.dev(d["seeds"])
    for T in (1.0, 0.0):
        tally = H.Tally()
        for cycle in range(2000):
            g = H.gpu_draft(d, T, cycle)
            gv = H.gpu_verify(tD, cuD, g["y_dev"], g["q_logits_dev"] if T > 0 else None,
                              g["q_lse_dev"] if T > 0 else None, g["q_tok_dev"] if T > 0 else None,
                              seedsD if T > 0 else None, cycle, T)
            o = orc.markov_draft(d["U"], d["W1"], d["W2"], d["anchor"], d["seeds"], cycle, T)
            ov = orc.verify(target, cu, o["y"], o["q_logits"], d["seeds"], cycle, T)
            clean = H.compare_draft(tally, g, o, T)
            H.compare_verify(tally, gv, ov, l, only=clean)
        tally.check()


def test_verify_edge_cases(B, orc):
    # every request plain decode (l = 0), V not a multiple of 4 (scalar path)
    R, V, gamma = 5, 1001, 4
    g = np.random.default_rng(2)
    target = g.normal(0, 2, (R, V)).astype(np.float32)
    cu = np.arange(R + 1, dtype=np.int32)
    y = np.zeros((R, gamma), np.int32)
    seeds = inputs.request_seeds(99, R)
    ql = np.zeros((R, gamma, V), np.float32)
    for T in (1.0, 0.0):
        gv = H.gpu_verify(target, cu, y, ql, np.zeros((R, gamma), np.float32),
                          np.ones((R, gamma), np.float32), seeds, 3, T)
        ov = orc.verify(target, cu, y, ql.astype(np.float64), seeds, 3, T)
        assert (gv["n_acc"] == 0).all()
        np.testing.assert_array_equal(gv["out_tokens"], ov["out_tokens"])
    # a bad draft token and a bad length are reported, the request outputs are -1
    l = np.array([2, 3, 1, 0, 2], np.int32)
    cu = inputs.cu_from_lengths(l)
    target = g.normal(0, 2, (cu[-1], V)).astype(np.float32)
    y = g.integers(0, V, (R, gamma)).astype(np.int32)
    y[1, 1] = V + 3
    gv = H.gpu_verify(target, cu, y, ql, np.zeros((R, gamma), np.float32),
                      np.ones((R, gamma), np.float32), seeds, 0, 1.0)
    assert gv["status"] == -6 and gv["n_acc"][1] == -1 and (gv["out_tokens"][1] == -1).all()
    assert (gv["n_acc"][[0, 2, 3, 4]] >= 0).all()
    bad_cu = cu.copy(); bad_cu[3] = bad_cu[2] - 1
    gv = H.gpu_verify(target, bad_cu, y, ql, np.zeros((R, gamma), np.float32),
                      np.ones((R, gamma), np.float32), seeds, 0, 1.0)
    assert gv["status"] == -6 and (gv["n_acc"] == -1).all()


def _empty_residual_case(R=16, V=1032):
    """Rows whose residual max(0, p - q) is empty in floating point although a
    rejection is likely.  Drafter row: 1024 zeros, the drafted token y at -40,
    seven entries at -inf; target row: the same but -41 at y, so p(y)/q(y) =
    1/e (rejected when u >= 0.37).  Both log-normalisers round to ln 1024 (the
    mass at y is 1e-18 of the total), so p == q on every other entry, in double
    and in fp32 alike: the exact residual mass, (q(y) - p(y)) ~ 3e-21, is far
    below either precision."""
    s = np.zeros(V, np.float32)
    s[1024] = -40.0
    s[1025:] = -np.inf
    t = s.copy()
    t[1024] = -41.0
    g = np.random.default_rng(11)
    target = np.zeros((2 * R, V), np.float32)
    target[0::2] = t
    target[1::2] = 3.0 * g.standard_normal((R, V)).astype(np.float32)  # bonus rows
    cu = inputs.cu_from_lengths(np.ones(R, np.int32))
    y = np.full((R, 1), 1024, np.int32)
    q_logits = np.broadcast_to(s, (R, 1, V)).copy()
    return s, target, cu, y, q_logits


def test_empty_residual_fallback(B, orc):
    """The empty-residual branch (a rejection whose max(0, p - q) has no mass in
    the working precision draws from p with the residual's noise): the oracle
    takes it on these rows, and both GPU verify paths -- stored drafter logits
    (dspark_verify) and recomputed ones (dspark_verify_markov: zero factors,
    anchor -1, so the recomputed logits are U itself) -- commit the same tokens."""
    R, V = 16, 1032
    s, target, cu, y, q_logits = _empty_residual_case(R, V)
    seeds = inputs.request_seeds(0x5EED0100, R)
    lse = orc.logsumexp(s.astype(np.float64))
    q_lse = np.full((R, 1), np.float32(lse), np.float32)
    q_tok = np.full((R, 1), np.float32(np.exp(-40.0 - lse)), np.float32)
    zeros_w = np.zeros((V, 64), np.uint16)
    d = dict(U=inputs.bf16_bits(q_logits), W1=zeros_w, W2=zeros_w, anchor=np.full(R, -1, np.int32),
             seeds=seeds)
    tally = H.Tally()
    empties = 0
    for cycle in range(3):
        ov = orc.verify(target, cu, y, q_logits.astype(np.float64), seeds, cycle, 1.0)
        empties += int(ov["residual_empty"].sum())
        gv = H.gpu_verify(target, cu, y, q_logits, q_lse, q_tok, seeds, cycle, 1.0)
        g = dict(y_dev=H.dev(y), q_lse_dev=H.dev(q_lse), q_tok_dev=H.dev(q_tok))
        gm = H.gpu_verify_markov(target, cu, d, g, cycle, 1.0)
        assert gv["status"] == 0 and gm["status"] == 0
        H.compare_verify(tally, gv, ov, np.ones(R, np.int32))
        H.compare_verify(tally, gm, ov, np.ones(R, np.int32))
    tally.check()
    assert empties >= 10, empties  # about 63% of 48 draws are rejections


# ------------------------------------------------------------------ select / commit
@pytest.mark.parametrize("mode", [0, 1, 2, 3])
@pytest.mark.parametrize("R,gamma,seed", [(512, 5, 0), (3, 3, 1), (97, 7, 2), (1000, 8, 3)])
def test_select_parity(B, orc, mode, R, gamma, seed):
    w = inputs.workload("confidence_scheduled", seed_offset=seed, R=R, gamma=gamma)
    ci = inputs.confidence_inputs(w)
    sizes, sps = ci["capture_sizes"], ci["sps"]
    if R < 64:
        sizes = np.array([3, 4, 5, 6, 8, 12], np.int32)
        sps = (1.0 / (0.010 + 0.0009 * sizes)).astype(np.float32)
    for K_cap in sorted({R, R + (R * gamma) // 3, 2 * R, R * (gamma + 1)}):
        o = orc.select_prefix(ci["c"], ci["c_hist"], sizes, sps, K_cap, mode)
        g = H.gpu_select(ci["c"], ci["c_hist"], sizes, sps, K_cap, mode)
        assert o["status"] == 0 and g["status"] == 0
        np.testing.assert_array_equal(g["a"].view(np.uint32), o["a"].view(np.uint32))
        if o["theta_gap"] > 1e-9:
            np.testing.assert_array_equal(g["l"], o["l"])
            np.testing.assert_array_equal(g["cu_seqlens"], o["cu_seqlens"])
            assert g["K_used"] == o["K_used"]


@pytest.mark.parametrize("mode", [4, 5])
@pytest.mark.parametrize("R,gamma,seed", [(512, 5, 0), (3, 3, 1), (97, 7, 2), (1000, 8, 3)])
def test_select_cutoff_parity(B, orc, mode, R, gamma, seed):
    """The static cutoffs (per-position confidence, survival), with room for
    every eligible row and with less: bit-exact a, l, cu_seqlens and K."""
    w = inputs.workload("confidence_scheduled", seed_offset=seed, R=R, gamma=gamma)
    c = inputs.confidence_inputs(w)["c"]
    for conf_min in (0.0, 0.3, 0.6, 0.95):
        for K_cap in sorted({R, R + (R * gamma) // 3, R * (gamma + 1)}):
            o = orc.select_prefix(c, None, None, None, K_cap, mode, conf_min)
            g = H.gpu_select(c, None, None, None, K_cap, mode, conf_min)
            assert o["status"] == 0 and g["status"] == 0
            np.testing.assert_array_equal(g["a"].view(np.uint32), o["a"].view(np.uint32))
            np.testing.assert_array_equal(g["l"], o["l"])
            np.testing.assert_array_equal(g["cu_seqlens"], o["cu_seqlens"])
            assert g["K_used"] == o["K_used"]


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4, 5])
def test_plan_cycles_parity(B, orc, mode):
    """A run of 64 cycles of the confidence-scheduled workload (R = 512,
    gamma = 5, K_cap = 1024), one CTA per cycle: lengths, capacities, accepted
    drafts and wasted rows bit-exact (cycles whose capacity choice is a
    rounding-level Theta tie exempt), Theta to fp64 rounding."""
    w = inputs.workload("confidence_scheduled")
    seq = inputs.confidence_sequence(w, 64)
    o = orc.plan_cycles(seq["c"], seq["n_full"], seq["capture_sizes"], seq["sps"], seq["K_cap"], mode, 0.6)
    g = H.gpu_plan(seq["c"], seq["n_full"], seq["capture_sizes"], seq["sps"], seq["K_cap"], mode, 0.6)
    assert o["status"] == 0 and g["status"] == 0
    keep = o["theta_gap"] > 1e-9
    assert keep.mean() > 0.99
    np.testing.assert_array_equal(g["l"][keep], o["l"][keep])
    np.testing.assert_array_equal(g["K_used"][keep], o["K_used"][keep])
    np.testing.assert_array_equal(g["accepted"][keep], o["accepted"][keep])
    np.testing.assert_array_equal(g["wasted"][keep], o["wasted"][keep])
    np.testing.assert_allclose(g["theta_pred"][keep], o["theta_pred"][keep], rtol=1e-12)
    np.testing.assert_allclose(g["theta_real"][keep], o["theta_real"][keep], rtol=1e-12)


@pytest.mark.parametrize("N,gamma,tau,zero", [(200_000, 5, None, False), (1000, 3, [1.0, 2.0, 0.5], False),
                                               (37, 4, None, False), (5000, 3, None, True)])
def test_fit_temperatures_parity(B, orc, N, gamma, tau, zero):
    """Sequential temperature scaling on the GPU against the oracle: the samples
    per position exactly, the temperatures and mean NLL to fp64 rounding of two
    Newton iterations converged to the same minimiser (relative 1e-6 and 1e-9);
    with every label 0 the later positions keep tau = 1."""
    w = inputs.workload("confidence_scheduled", gamma=gamma)
    cs = inputs.calibration_samples(w, N, tau_true=tau)
    if zero:
        cs["accepted"][:] = 0
    o = orc.fit_temperatures(cs["z"], cs["accepted"])
    G = H.Guarded()
    t = G.out((gamma,), torch.float32, float("nan"))
    nll = G.out((gamma,), torch.float64, float("nan"))
    cnt = G.out((gamma,), torch.int32, -7)
    ws = G.workspace(B.dspark_workspace_size(B.DSPARK_OP_CALIBRATE, 0, gamma, 0))
    status = G.out((1,), torch.int32, 0)
    B.dspark_fit_temperatures(H.dev(cs["z"]), H.dev(cs["accepted"]), t, nll, cnt, ws, status)
    torch.cuda.synchronize()
    G.check()
    assert int(status.item()) == 0 and o["status"] == 0
    np.testing.assert_array_equal(H.host(cnt), o["count"])
    np.testing.assert_allclose(H.host(t), o["tau"], rtol=1e-6)
    np.testing.assert_allclose(H.host(nll), o["nll"], rtol=1e-9, atol=1e-12)
    if zero:
        assert (H.host(t)[1:] == 1.0).all()


def test_kv_reserve_commit_parity(B, orc):
    """Forty cycles of reserve -> verify outcome -> commit on a 512-request paged
    KV cache (page size 16) against the oracle: lengths, block table, the whole
    free stack and its top bit-exact after every call (the stack order is a
    scan over the requests, so it is unique); then the two failure cases."""
    w = inputs.workload("confidence_scheduled")
    kv = inputs.kv_state(w, page_size=16, max_len=4096, spare_pages=3)
    st = orc.KvState(kv["kv_len"], kv["block_table"], kv["free_pages"], kv["free_top"], kv["page_size"])
    G = H.Guarded()
    d_len = G.out((w["R"],), torch.int32, 0); d_len.copy_(H.dev(st.kv_len))
    d_bt = G.out(st.block_table.shape, torch.int32, 0); d_bt.copy_(H.dev(st.block_table))
    d_free = G.out(st.free_pages.shape, torch.int32, 0); d_free.copy_(H.dev(st.free_pages))
    d_top = G.out((1,), torch.int32, 0); d_top.copy_(H.dev(st.free_top))
    d_res = G.out((w["R"],), torch.int32, -7)
    status = G.out((1,), torch.int32, 0)
    g = np.random.default_rng(7)
    P = kv["page_size"]

    def same():
        torch.cuda.synchronize()
        np.testing.assert_array_equal(H.host(d_len), st.kv_len)
        np.testing.assert_array_equal(H.host(d_bt), st.block_table)
        np.testing.assert_array_equal(H.host(d_free), st.free_pages)
        assert int(d_top.item()) == int(st.free_top[0])

    for cycle in range(40):
        l = g.integers(0, w["gamma"] + 1, size=w["R"]).astype(np.int32)
        n_acc = (g.random(w["R"]) * (l + 1)).astype(np.int32)
        rc, res = orc.kv_reserve(st, l)
        assert rc == 0
        B.dspark_kv_reserve(d_len, H.dev(l), P, d_bt, d_free, d_top, d_res, status)
        same()
        np.testing.assert_array_equal(H.host(d_res), res)
        assert orc.kv_commit(st, l, n_acc) == 0
        B.dspark_kv_commit(d_len, H.dev(l), H.dev(n_acc), P, d_bt, d_free, d_top, status)
        same()
        # requests past 3000 tokens finish: their pages go back (the same on both sides)
        for r in np.nonzero(st.kv_len > 3000)[0]:
            pages = st.block_table[r][st.block_table[r] >= 0]
            st.free_pages[st.free_top[0]: st.free_top[0] + len(pages)] = pages
            st.free_top[0] += len(pages)
            st.block_table[r] = -1
            st.kv_len[r] = 0
        d_len.copy_(H.dev(st.kv_len)); d_bt.copy_(H.dev(st.block_table))
        d_free.copy_(H.dev(st.free_pages)); d_top.copy_(H.dev(st.free_top))
    assert int(status.item()) == 0
    # too few free pages: nothing changes and the capacity error is reported
    d_top.fill_(0); st.free_top[0] = 0
    B.dspark_kv_reserve(d_len, H.dev(np.full(w["R"], w["gamma"], np.int32)), P, d_bt, d_free, d_top, None, status)
    same()
    assert int(status.item()) == B.DSPARK_ERR_CAPACITY
    G.check()


def test_select_ties_and_errors(B, orc):
    c = np.array([[1.0, 1.0], [1.0, 0.5], [0.7, 0.7]], np.float32)
    for K_cap in range(3, 10):
        o = orc.select_prefix(c, None, None, None, K_cap, 0)
        g = H.gpu_select(c, None, None, None, K_cap, 0)
        np.testing.assert_array_equal(g["l"], o["l"])
    # a confidence of -0 is a survival of 0: it ties with +0 (position, then request order)
    cz = np.array([[-0.0, 0.5], [0.0, 1.0], [0.3, -0.0], [0.0, 0.0]], np.float32)
    for K_cap in range(4, 13):
        o = orc.select_prefix(cz, None, None, None, K_cap, 0)
        g = H.gpu_select(cz, None, None, None, K_cap, 0)
        np.testing.assert_array_equal(g["l"], o["l"])
        np.testing.assert_array_equal(g["cu_seqlens"], o["cu_seqlens"])
    bad = c.copy(); bad[2, 1] = np.nan
    for K_cap in (6, 9):  # a ranked selection; a capacity that admits every candidate
        g = H.gpu_select(bad, None, None, None, K_cap, 0)
        assert g["status"] == -6 and (g["l"] == -1).all() and (g["cu_seqlens"] == -1).all()
        assert g["K_used"] == -1
    with pytest.raises(B.DSparkError):
        H.gpu_select(c, None, None, None, 2, 0)


def test_commit_parity(B, orc):
    g = np.random.default_rng(0)
    for R, gamma in [(1, 5), (700, 7), (3000, 5)]:
        l = g.integers(0, gamma + 1, R).astype(np.int32)
        n_acc = (g.random(R) * (l + 1)).astype(np.int32)
        for ll in (l, None):
            o = orc.commit_lengths(n_acc if ll is not None else np.minimum(n_acc, gamma), ll, gamma)
            gg = H.gpu_commit(n_acc if ll is not None else np.minimum(n_acc, gamma), ll, gamma)
            for key in ("commit_len", "cu_commit", "discard"):
                np.testing.assert_array_equal(gg[key], o[key])
            assert gg["total"] == o["total"] and gg["status"] == 0


# ------------------------------------------------------------------ full-size workloads
FULL = [
    ("qwen3_8b_greedy", 4),
    ("batched_sampling", 2),
    ("varlen_verify", 1),
    ("confidence_scheduled", 1),
]


def _sample_rows(R, cycle, l, n=8):
    """n requests replayed on the oracle, drawn afresh each cycle, always with
    the first and last request and, for variable lengths, the shortest and
    longest verify length."""
    g = np.random.default_rng(1000 + cycle)
    rows = {0, R - 1, int(np.argmin(l)), int(np.argmax(l))}
    rest = [r for r in g.permutation(R) if r not in rows]
    rows.update(int(r) for r in rest[: max(0, n - len(rows))])
    return sorted(rows)


@pytest.mark.parametrize("name,cycles", FULL)
def test_full_size_cycle_sampled(B, orc, name, cycles):
    w, d = H.cycle_inputs(name)
    T = float(w["temperature"])
    full = inputs.target_full(w, d["U"])
    R, gamma = w["R"], w["gamma"]
    tally = H.Tally()
    for cycle in range(cycles):
        if w.get("confidence"):
            ci = inputs.confidence_inputs(w)
            o_s = orc.select_prefix(ci["c"], ci["c_hist"], ci["capture_sizes"], ci["sps"], ci["K_cap"], 1)
            g_s = H.gpu_select(ci["c"], ci["c_hist"], ci["capture_sizes"], ci["sps"], ci["K_cap"], 1)
            np.testing.assert_array_equal(g_s["l"], o_s["l"])
            l = o_s["l"]
        else:
            l = inputs.verify_lengths(w)
        cu = inputs.cu_from_lengths(l)
        target = inputs.pack_rows(full, l)
        g = H.gpu_draft(d, T, cycle)
        gv = H.gpu_verify(target, cu, g["y_dev"], g["q_logits_dev"] if T > 0 else None,
                          g["q_lse_dev"] if T > 0 else None, g["q_tok_dev"] if T > 0 else None,
                          H.dev(d["seeds"]) if T > 0 else None, cycle, T)
        assert g["status"] == 0 and gv["status"] == 0
        rows = _sample_rows(R, cycle, l)
        sub = dict(U=d["U"][rows], anchor=d["anchor"][rows], seeds=d["seeds"][rows])
        o = orc.markov_draft(sub["U"], d["W1"], d["W2"], sub["anchor"], sub["seeds"], cycle, T,
                             req_ids=rows)
        lsub = l[rows]
        ov = orc.verify(inputs.pack_rows(full[rows], lsub), inputs.cu_from_lengths(lsub), o["y"],
                        o["q_logits"], sub["seeds"], cycle, T, req_ids=rows)
        clean = H.compare_draft(tally, g, o, T, rows=rows)
        H.compare_verify(tally, gv, ov, lsub, rows=rows, only=clean)
        # the same verify with the drafter's rejected rows recomputed from its factors
        gm = H.gpu_verify_markov(H.dev(target), H.dev(cu), d, g, cycle, T)
        assert gm["status"] == 0
        np.testing.assert_array_equal(gm["n_acc"], gv["n_acc"])
        np.testing.assert_array_equal(gm["out_tokens"], gv["out_tokens"])
        # properties that hold for every request of the batch
        assert ((gv["n_acc"] >= 0) & (gv["n_acc"] <= l)).all()
        for r in range(R):
            n = gv["n_acc"][r]
            assert (gv["out_tokens"][r, :n] == g["y"][r, :n]).all()
            assert 0 <= gv["out_tokens"][r, n] < w["V"]
            assert (gv["out_tokens"][r, n + 1:] == -1).all()
    tally.check()
