"""Helpers for the GPU parity tests: run the CUDA library through its C ABI on
seeded inputs and compare with the CPU oracle.

Comparison rule: token ids, accepted counts, verify lengths and row offsets
must agree exactly, except where the oracle itself records a rounding-level
near tie -- the top two Gumbel (or greedy logit) scores of a draw within
MARGIN, or |u - p/q| within MARGIN for an acceptance -- such decisions are
counted as exempt and the rest of that request is left out; exempt decisions
must stay under 0.1% of all decisions.  Probabilities (q(y), p(y)) agree to
PROB_TOL absolute, log-normalisers to LSE_TOL relative.

Every output and workspace passed to the library is surrounded by guard bytes
that are checked after the call (no write outside a buffer).
"""
from __future__ import annotations

import numpy as np
import torch

from speculative_decoding_dspark_gb300 import binding as B
from speculative_decoding_dspark_gb300 import inputs

MARGIN = 1e-5
PROB_TOL = 1e-5
LSE_TOL = 1e-5
EXEMPT_FRACTION = 1e-3


# ---------------------------------------------------------------- guard words
# Every output and workspace the helpers hand to the library sits between two
# 256-byte guard regions filled with GUARD_BYTE; after each call the guards are
# compared, so a kernel writing past either end of a buffer fails the test.
GUARD_BYTES = 256
GUARD_BYTE = 0xA5


class Guarded:
    """Outputs and workspaces of one library call, each between guard regions."""

    def __init__(self):
        self.raw = []

    def _alloc(self, nbytes):
        nbytes = int(nbytes)
        raw = torch.empty(GUARD_BYTES + nbytes + GUARD_BYTES, dtype=torch.uint8, device="cuda")
        raw.fill_(GUARD_BYTE)
        self.raw.append((raw, nbytes))
        return raw[GUARD_BYTES:GUARD_BYTES + nbytes]

    def out(self, shape, dtype, fill):
        """A contiguous tensor of `shape` filled with `fill` (its data 256-byte aligned)."""
        n = int(np.prod(shape))
        item = torch.empty((), dtype=dtype).element_size()
        t = self._alloc(max(n, 1) * item).view(dtype)[:n].view(shape)
        t.fill_(fill)
        return t

    def workspace(self, nbytes):
        return self._alloc(max(int(nbytes), 256))

    def check(self):
        """Call after the device has finished the call."""
        for raw, nbytes in self.raw:
            head = raw[:GUARD_BYTES]
            tail = raw[GUARD_BYTES + nbytes:]
            assert bool((head == GUARD_BYTE).all()), "write before the start of an output or workspace"
            assert bool((tail == GUARD_BYTE).all()), "write past the end of an output or workspace"


def dev(x: np.ndarray) -> torch.Tensor:
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    if x.dtype == np.uint64:
        return torch.from_numpy(x.view(np.int64)).cuda()
    if x.dtype == np.uint32:
        return torch.from_numpy(x.view(np.int32)).cuda()
    return torch.from_numpy(x).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def gpu_draft(d: dict, temperature: float, cycle: int, flags: int = 0, want_logits: bool = True):
    U, W1, W2 = dev(d["U"]), dev(d["W1"]), dev(d["W2"])
    R, gamma, V = U.shape
    rank = W1.shape[1]
    G = Guarded()
    y = G.out((R, gamma), torch.int32, -7)
    q_lse = G.out((R, gamma), torch.float32, float("nan"))
    q_tok = G.out((R, gamma), torch.float32, float("nan"))
    q_logits = G.out((R, gamma, V), torch.float32, float("nan")) if want_logits else None
    w_dtype = B.DSPARK_BF16 if W1.dtype == torch.bfloat16 else B.DSPARK_F32
    ws = G.workspace(B.dspark_workspace_size(B.DSPARK_OP_DRAFT, R, gamma, V, rank, 0, w_dtype, flags))
    status = G.out((1,), torch.int32, 0)
    B.dspark_markov_draft(U, W1, W2, dev(d["anchor"]), dev(d["seeds"]), cycle, temperature, y,
                          q_lse, q_tok, q_logits, ws, status, flags=flags)
    torch.cuda.synchronize()
    G.check()
    out = dict(y=host(y), q_lse=host(q_lse), q_tok=host(q_tok), status=int(status.item()))
    out["q_logits_dev"] = q_logits
    out["q_lse_dev"], out["q_tok_dev"], out["y_dev"] = q_lse, q_tok, y
    return out


def gpu_fused_draft(f: dict, temperature: float, cycle: int, want_logits: bool = True, dev_inputs=None):
    """dspark_markov_draft_fused on the inputs of inputs.fused_inputs (dev_inputs: the same
    arrays already on the device, keyed alike)."""
    t = dev_inputs or {k: dev(f[k]) for k in ("h", "W_lm", "W1", "W2", "anchor", "seeds")}
    R, gamma, d = t["h"].shape
    V = t["W_lm"].shape[0]
    rank = t["W1"].shape[1]
    G = Guarded()
    y = G.out((R, gamma), torch.int32, -7)
    q_lse = G.out((R, gamma), torch.float32, float("nan"))
    q_tok = G.out((R, gamma), torch.float32, float("nan"))
    q_logits = G.out((R, gamma, V), torch.float32, float("nan")) if want_logits else None
    ws = G.workspace(B.dspark_workspace_size(B.DSPARK_OP_DRAFT_FUSED, R, gamma, V, rank, 0, B.DSPARK_BF16, 0))
    status = G.out((1,), torch.int32, 0)
    B.dspark_markov_draft_fused(t["h"], t["W_lm"], t["W1"], t["W2"], t["anchor"], t["seeds"], cycle, temperature,
                                y, q_lse, q_tok, q_logits, ws, status)
    torch.cuda.synchronize()
    G.check()
    out = dict(y=host(y), q_lse=host(q_lse), q_tok=host(q_tok), status=int(status.item()))
    out["q_logits_dev"] = q_logits
    return out


def fused_logit_tol(x: np.ndarray, d: int, rank: int, sigma_s: float) -> np.ndarray:
    """Elementwise bound on |GPU - oracle| for the fused draft's scaled logits x (the
    oracle's, in double).  The contraction runs as (d + rank) / 16 tensor-core MMAs
    of K = 16 adding into one fp32 accumulator; allowing each addition to lose one
    unit in the last place (2^-23 relative, an accumulator that truncates) at a
    partial-sum magnitude up to |x| + sigma_s (sigma_s: the scale of the logits'
    law, the partial sums' typical excursion past the final value) gives
    ((d + rank) / 16 + 2) * 2^-23 * (|x| + sigma_s).  A dropped or repeated 64-wide
    k-block, or one wrong operand element, moves a logit by far more."""
    n_mma = (d + rank) // 16
    return (n_mma + 2) * 2.0 ** -23 * (np.abs(x) + sigma_s)


def gpu_verify(target, cu, y, q_logits, q_lse, q_tok, seeds, cycle, temperature, max_rows=None):
    """All array arguments may be numpy (copied) or CUDA tensors (used as is)."""
    t = lambda a: None if a is None else (a if isinstance(a, torch.Tensor) else dev(a))
    target_d, cu_d, y_d = t(target), t(cu), t(y)
    R, gamma = y_d.shape
    V = target_d.shape[1]
    max_rows = int(target_d.shape[0]) if max_rows is None else max_rows
    G = Guarded()
    n_acc = G.out((R,), torch.int32, -7)
    out = G.out((R, gamma + 1), torch.int32, -7)
    p_tok = G.out((R, gamma), torch.float32, float("nan"))
    ws = G.workspace(B.dspark_workspace_size(B.DSPARK_OP_VERIFY, R, gamma, V, 0, max_rows))
    status = G.out((1,), torch.int32, 0)
    B.dspark_verify(target_d, cu_d, y_d, t(q_logits), t(q_lse), t(q_tok), t(seeds), cycle,
                    temperature, max_rows, n_acc, out, p_tok, ws, status)
    torch.cuda.synchronize()
    G.check()
    return dict(n_acc=host(n_acc), out_tokens=host(out), p_tok=host(p_tok), status=int(status.item()))


def gpu_verify_markov(target, cu, d, g, cycle, temperature, max_rows=None, host_target=False):
    """dspark_verify_markov on the GPU draft g of inputs d (drafter logits recomputed);
    host_target: target is a pinned host tensor read by the kernels across the link."""
    t = lambda a: a if isinstance(a, torch.Tensor) else dev(a)
    target_d, cu_d = t(target), t(cu)
    y_d = g["y_dev"]
    R, gamma = y_d.shape
    V = target_d.shape[1]
    W1 = dev(d["W1"])
    rank = W1.shape[1]
    max_rows = int(target_d.shape[0]) if max_rows is None else max_rows
    G = Guarded()
    n_acc = G.out((R,), torch.int32, -7)
    out = G.out((R, gamma + 1), torch.int32, -7)
    p_tok = G.out((R, gamma), torch.float32, float("nan"))
    ws = G.workspace(B.dspark_workspace_size(B.DSPARK_OP_VERIFY_MARKOV, R, gamma, V, rank, max_rows, B.DSPARK_BF16,
                                             B.DSPARK_VERIFY_HOST_TARGET if host_target else 0))
    status = G.out((1,), torch.int32, 0)
    samp = temperature > 0
    B.dspark_verify_markov(target_d, cu_d, y_d, dev(d["U"]), W1, dev(d["W2"]), dev(d["anchor"]),
                           g["q_lse_dev"] if samp else None, g["q_tok_dev"] if samp else None,
                           dev(d["seeds"]) if samp else None, cycle, temperature, max_rows, n_acc, out,
                           p_tok, ws, status)
    torch.cuda.synchronize()
    G.check()
    return dict(n_acc=host(n_acc), out_tokens=host(out), p_tok=host(p_tok), status=int(status.item()))


def gpu_select(c, c_hist, sizes, sps, K_cap, mode, conf_min=0.0):
    R, gamma = c.shape
    G = Guarded()
    a = G.out((R, gamma), torch.float32, float("nan"))
    l = G.out((R,), torch.int32, -7)
    cu = G.out((R + 1,), torch.int32, -7)
    K = G.out((1,), torch.int32, 0)
    status = G.out((1,), torch.int32, 0)
    t = lambda x: None if x is None else dev(x)
    try:
        B.dspark_select_prefix(dev(c), t(c_hist), t(sizes), t(sps), K_cap, mode, a, l, cu, K, None, status,
                               conf_min=conf_min)
    finally:
        torch.cuda.synchronize()
        G.check()
    return dict(a=host(a), l=host(l), cu_seqlens=host(cu), K_used=int(K.item()), status=int(status.item()))


def gpu_plan(c_seq, n_full, sizes, sps, K_cap, mode, conf_min=0.0, lag=2):
    T, R, gamma = c_seq.shape
    G = Guarded()
    l = G.out((T, R), torch.int32, -7)
    K = G.out((T,), torch.int32, -7)
    stats = G.out((T, 4), torch.float64, float("nan"))
    status = G.out((1,), torch.int32, 0)
    B.dspark_plan_cycles(dev(c_seq), None if n_full is None else dev(n_full), dev(sizes), dev(sps), K_cap, mode,
                         l, K, stats, conf_min=conf_min, lag=lag, dev_status=status)
    torch.cuda.synchronize()
    G.check()
    st = host(stats)
    return dict(l=host(l), K_used=host(K), theta_pred=st[:, 0], theta_real=st[:, 1],
                accepted=st[:, 2].astype(np.int64), wasted=st[:, 3].astype(np.int64), status=int(status.item()))


def gpu_commit(n_acc, l, gamma):
    R = len(n_acc)
    G = Guarded()
    cl = G.out((R,), torch.int32, -7)
    cu = G.out((R + 1,), torch.int32, -7)
    disc = G.out((R,), torch.int32, -7)
    tot = G.out((1,), torch.int32, 0)
    status = G.out((1,), torch.int32, 0)
    B.dspark_commit_lengths(dev(np.asarray(n_acc, np.int32)), None if l is None else dev(np.asarray(l, np.int32)),
                            gamma, cl, cu, disc, tot, status)
    torch.cuda.synchronize()
    G.check()
    return dict(commit_len=host(cl), cu_commit=host(cu), discard=host(disc), total=int(tot.item()),
                status=int(status.item()))


class Tally:
    """Counts decisions and exempt near ties across a test."""

    def __init__(self):
        self.decisions = 0
        self.exempt = 0
        self.errors = []

    def check(self):
        assert not self.errors, self.errors[:10]
        assert self.exempt <= max(1, EXEMPT_FRACTION * self.decisions) or self.decisions == 0, \
            (self.exempt, self.decisions)


def compare_draft(tally: Tally, g: dict, o: dict, temperature: float, rows=None):
    """Returns the set of request rows whose drafts matched completely."""
    R, gamma = o["y"].shape
    clean = set()
    for i in range(R):
        gi = i if rows is None else rows[i]
        ok = True
        for k in range(gamma):
            tally.decisions += 1
            if g["y"][gi, k] != o["y"][i, k]:
                if o["margin"][i, k] <= MARGIN:
                    tally.exempt += 1
                else:
                    tally.errors.append(("draft token", gi, k, int(g["y"][gi, k]), int(o["y"][i, k]),
                                         float(o["margin"][i, k])))
                ok = False
                break
            if temperature > 0:
                if abs(g["q_tok"][gi, k] - o["q_tok"][i, k]) > PROB_TOL:
                    tally.errors.append(("q_tok", gi, k, float(g["q_tok"][gi, k]), float(o["q_tok"][i, k])))
                lse = o["q_lse"][i, k]
                if abs(g["q_lse"][gi, k] - lse) > LSE_TOL * max(1.0, abs(lse)):
                    tally.errors.append(("q_lse", gi, k, float(g["q_lse"][gi, k]), float(lse)))
        if ok:
            clean.add(i)
    return clean


def compare_verify(tally: Tally, g: dict, o: dict, l, rows=None, only=None):
    """Compare n_acc, out_tokens and p_tok of the oracle's requests (optionally a
    subset); l = the verify length of each oracle request."""
    R = len(o["n_acc"])
    for i in range(R):
        if only is not None and i not in only:
            continue
        gi = i if rows is None else rows[i]
        n_o, n_g = int(o["n_acc"][i]), int(g["n_acc"][gi])
        tally.decisions += max(n_o, 0) + 1
        if n_o != n_g:
            j = min(n_o, n_g)
            if j >= 0 and o["accept_margin"][i, j] <= MARGIN:
                tally.exempt += 1
            else:
                tally.errors.append(("n_acc", gi, n_g, n_o))
            continue
        if list(g["out_tokens"][gi]) != list(o["out_tokens"][i]):
            if o["sample_margin"][i] <= MARGIN:
                tally.exempt += 1
            else:
                tally.errors.append(("out_tokens", gi, list(g["out_tokens"][gi]), list(o["out_tokens"][i]),
                                     float(o["sample_margin"][i])))
            continue
        if n_o < 0:
            continue
        for j in range(min(n_o + 1, int(l[i]))):  # the drafts examined
            if abs(g["p_tok"][gi, j] - o["p_tok"][i, j]) > PROB_TOL:
                tally.errors.append(("p_tok", gi, j, float(g["p_tok"][gi, j]), float(o["p_tok"][i, j])))


def cycle_inputs(name: str, seed_offset: int = 0, **overrides):
    w = inputs.workload(name, seed_offset=seed_offset, **overrides)
    d = inputs.draft_inputs(w)
    return w, d
