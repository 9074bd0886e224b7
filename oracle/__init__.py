"""CPU oracle for the DSpark decode-cycle hot path -- TEST INFRASTRUCTURE ONLY.

A thin numpy/ctypes wrapper over ``dspark_oracle.cpp``, a plain single-threaded
C++ restatement of the cycle in double precision (Markov-head draft, from given
base logits or from the drafter's hidden states and shared lm_head, lossless
verify with residual and bonus, survival and prefix selection, commit
lengths, and the Philox4x32-10 generator they draw from).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it and
shares no code with it; the product path fails loudly instead of falling back
here.

Every function is pinned by a CPU test against something other than itself
(closed forms, brute force, an independent library Philox and empirical
laws); none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.cpp")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libdspark_oracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16 = 0, 1
PURPOSE_DRAFT, PURPOSE_ACCEPT, PURPOSE_RESIDUAL, PURPOSE_BONUS = 0, 1, 2, 3
MODE_FIXED, MODE_HISTORY, MODE_CURRENT, MODE_FIRST_STOP = 0, 1, 2, 3
MODE_CONF_CUTOFF, MODE_SURVIVAL_CUTOFF = 4, 5


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (plain -O2, no FP contraction) and return the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            vp, i32, u32, u64, f32, dbl = (ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32,
                                           ctypes.c_uint64, ctypes.c_float, ctypes.c_double)
            L.orc_philox4x32_10.argtypes = [vp, u64, vp]
            L.orc_philox4x32_10_batch.argtypes = [vp, vp, i32, vp]
            L.orc_uniform_from_bits.argtypes = [u32]
            L.orc_uniform_from_bits.restype = dbl
            L.orc_uniform_vocab.argtypes = [u64, u32, i32, i32, i32, i32]
            L.orc_uniform_vocab.restype = dbl
            L.orc_uniform_single.argtypes = [u64, u32, i32, i32, i32]
            L.orc_uniform_single.restype = dbl
            L.orc_markov_bias.argtypes = [vp, vp, i32, i32, i32, i32, vp]
            L.orc_logsumexp.argtypes = [vp, i32]
            L.orc_logsumexp.restype = dbl
            L.orc_softmax.argtypes = [vp, i32, vp]
            L.orc_residual_weights.argtypes = [vp, vp, i32, vp]
            L.orc_residual_weights.restype = dbl
            L.orc_markov_draft.argtypes = [vp, i32, vp, vp, i32, vp, vp, vp, u32, f32,
                                           i32, i32, i32, i32, vp, vp, vp, vp, vp]
            L.orc_markov_draft.restype = i32
            L.orc_fused_draft.argtypes = [vp, vp, i32, i32, vp, vp, i32, vp, vp, vp, u32, f32,
                                          i32, i32, i32, i32, vp, vp, vp, vp, vp]
            L.orc_fused_draft.restype = i32
            L.orc_verify.argtypes = [vp, vp, vp, vp, vp, vp, u32, f32, i32, i32, i32,
                                     vp, vp, vp, vp, vp, vp]
            L.orc_verify.restype = i32
            L.orc_select_prefix.argtypes = [vp, vp, vp, vp, i32, i32, i32, f32, i32, i32,
                                            vp, vp, vp, vp, vp]
            L.orc_select_prefix.restype = i32
            L.orc_plan_cycles.argtypes = [vp, vp, vp, vp, i32, i32, i32, f32, i32, i32, i32, i32,
                                          vp, vp, vp, vp]
            L.orc_plan_cycles.restype = i32
            L.orc_fit_temperatures.argtypes = [vp, vp, i32, i32, vp, vp, vp]
            L.orc_fit_temperatures.restype = i32
            L.orc_kv_reserve.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp, i32, vp]
            L.orc_kv_reserve.restype = i32
            L.orc_kv_commit.argtypes = [vp, vp, vp, i32, i32, vp, i32, vp, vp, i32]
            L.orc_kv_commit.restype = i32
            L.orc_commit_lengths.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp]
            L.orc_commit_lengths.restype = i32
            _lib = L
    return _lib


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _wdtype(a):
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"weights/logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


# ---------------------------------------------------------------- generator
def philox4x32_10(ctr, seed: int) -> np.ndarray:
    ctr = _c(ctr, np.uint32)
    out = np.zeros(4, np.uint32)
    lib().orc_philox4x32_10(_p(ctr), ctypes.c_uint64(seed), _p(out))
    return out


def philox4x32_10_batch(ctr, keys) -> np.ndarray:
    """ctr [n, 4] uint32, keys [n] uint64 -> [n, 4] uint32."""
    ctr = _c(ctr, np.uint32)
    keys = _c(keys, np.uint64)
    out = np.zeros_like(ctr)
    lib().orc_philox4x32_10_batch(_p(ctr), _p(keys), keys.size, _p(out))
    return out


def uniform_from_bits(x: int) -> float:
    return lib().orc_uniform_from_bits(x)


def uniform_vocab(seed, cycle, purpose, req, pos, v) -> float:
    return lib().orc_uniform_vocab(seed, cycle, purpose, req, pos, v)


def uniform_single(seed, cycle, purpose, req, pos) -> float:
    return lib().orc_uniform_single(seed, cycle, purpose, req, pos)


# ---------------------------------------------------------------- row helpers
def markov_bias(W1, W2, prev: int) -> np.ndarray:
    W1 = np.ascontiguousarray(W1)
    W2 = np.ascontiguousarray(W2)
    V, rank = W2.shape
    b = np.zeros(V, np.float64)
    lib().orc_markov_bias(_p(W1), _p(W2), _wdtype(W2), V, rank, prev, _p(b))
    return b


def logsumexp(x) -> float:
    x = _c(x, np.float64)
    return lib().orc_logsumexp(_p(x), x.size)


def softmax(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.zeros_like(x)
    lib().orc_softmax(_p(x), x.size, _p(out))
    return out


def residual_weights(p, q):
    p = _c(p, np.float64)
    q = _c(q, np.float64)
    res = np.zeros_like(p)
    total = lib().orc_residual_weights(_p(p), _p(q), p.size, _p(res))
    return res, total


# ---------------------------------------------------------------- cycle steps
def markov_draft(U, W1, W2, anchor, seeds, cycle, temperature, req_ids=None,
                 want_logits=True):
    """Draft gamma tokens per request. U: [R,gamma,V] float32 or bf16 bits."""
    U = np.ascontiguousarray(U)
    W1 = np.ascontiguousarray(W1)
    W2 = np.ascontiguousarray(W2)
    assert W1.dtype == W2.dtype
    R, gamma, V = U.shape
    rank = W2.shape[1]
    anchor = _c(anchor, np.int32)
    seeds = _c(seeds, np.uint64)
    rid = None if req_ids is None else _c(req_ids, np.int32)
    y = np.zeros((R, gamma), np.int32)
    q_lse = np.zeros((R, gamma), np.float64)
    q_tok = np.zeros((R, gamma), np.float64)
    margin = np.zeros((R, gamma), np.float64)
    q_logits = np.zeros((R, gamma, V), np.float64) if want_logits else None
    st = lib().orc_markov_draft(_p(U), _wdtype(U), _p(W1), _p(W2), _wdtype(W2), _p(anchor),
                                _p(seeds), _p(rid), cycle, temperature, R, gamma, V, rank,
                                _p(y), _p(q_lse), _p(q_tok), _p(q_logits), _p(margin))
    return dict(status=st, y=y, q_lse=q_lse, q_tok=q_tok, q_logits=q_logits, margin=margin)


def fused_draft(h, W_lm, W1, W2, anchor, seeds, cycle, temperature, req_ids=None,
                want_logits=True):
    """Draft gamma tokens per request with the base logits formed from the
    drafter's hidden states and the shared lm_head: U[r,k,v] = <W_lm[v], h[r,k]>.
    h: [R,gamma,d], W_lm: [V,d], both float32 or both bf16 bits."""
    h = np.ascontiguousarray(h)
    W_lm = np.ascontiguousarray(W_lm)
    W1 = np.ascontiguousarray(W1)
    W2 = np.ascontiguousarray(W2)
    assert W1.dtype == W2.dtype and h.dtype == W_lm.dtype
    R, gamma, d = h.shape
    V = W_lm.shape[0]
    assert W_lm.shape[1] == d and W2.shape[0] == V
    rank = W2.shape[1]
    anchor = _c(anchor, np.int32)
    seeds = _c(seeds, np.uint64)
    rid = None if req_ids is None else _c(req_ids, np.int32)
    y = np.zeros((R, gamma), np.int32)
    q_lse = np.zeros((R, gamma), np.float64)
    q_tok = np.zeros((R, gamma), np.float64)
    margin = np.zeros((R, gamma), np.float64)
    q_logits = np.zeros((R, gamma, V), np.float64) if want_logits else None
    st = lib().orc_fused_draft(_p(h), _p(W_lm), _wdtype(h), d, _p(W1), _p(W2), _wdtype(W2), _p(anchor),
                               _p(seeds), _p(rid), cycle, temperature, R, gamma, V, rank,
                               _p(y), _p(q_lse), _p(q_tok), _p(q_logits), _p(margin))
    return dict(status=st, y=y, q_lse=q_lse, q_tok=q_tok, q_logits=q_logits, margin=margin)


def verify(target, cu_seqlens, y, q_logits, seeds, cycle, temperature, req_ids=None):
    """Verify drafted blocks against packed target rows [sum(l+1), V] float32."""
    target = _c(target, np.float32)
    cu = _c(cu_seqlens, np.int32)
    y = _c(y, np.int32)
    R, gamma = y.shape
    V = target.shape[1]
    ql = None if q_logits is None else _c(q_logits, np.float64)
    if ql is None and temperature != 0.0:
        raise ValueError("sampling verify needs the drafter's q_logits")
    seeds = _c(seeds, np.uint64)
    rid = None if req_ids is None else _c(req_ids, np.int32)
    n_acc = np.zeros(R, np.int32)
    out = np.zeros((R, gamma + 1), np.int32)
    p_tok = np.zeros((R, gamma), np.float64)
    am = np.zeros((R, gamma), np.float64)
    sm = np.zeros(R, np.float64)
    empty = np.zeros(R, np.int32)
    st = lib().orc_verify(_p(target), _p(cu), _p(y), _p(ql), _p(seeds), _p(rid), cycle,
                          temperature, R, gamma, V, _p(n_acc), _p(out), _p(p_tok), _p(am),
                          _p(sm), _p(empty))
    return dict(status=st, n_acc=n_acc, out_tokens=out, p_tok=p_tok, accept_margin=am,
                sample_margin=sm, residual_empty=empty)


def select_prefix(c, c_hist, capture_sizes, sps, K_cap, mode, conf_min=0.0):
    c = _c(c, np.float32)
    R, gamma = c.shape
    ch = None if c_hist is None else _c(c_hist, np.float32)
    cs = None if capture_sizes is None else _c(capture_sizes, np.int32)
    sp = None if sps is None else _c(sps, np.float32)
    n_steps = 0 if cs is None else cs.size
    a = np.zeros((R, gamma), np.float32)
    l = np.zeros(R, np.int32)
    cu = np.zeros(R + 1, np.int32)
    K_used = np.zeros(1, np.int32)
    gap = np.zeros(1, np.float64)
    st = lib().orc_select_prefix(_p(c), _p(ch), _p(cs), _p(sp), n_steps, K_cap, mode, conf_min, R,
                                 gamma, _p(a), _p(l), _p(cu), _p(K_used), _p(gap))
    return dict(status=st, a=a, l=l, cu_seqlens=cu, K_used=int(K_used[0]), theta_gap=float(gap[0]))


def plan_cycles(c_seq, n_full, capture_sizes, sps, K_cap, mode, conf_min=0.0, lag=2):
    """A run of scheduling cycles: c_seq [n_cycles, R, gamma] float32, n_full
    [n_cycles, R] int32 (leading drafts the target would accept) or None."""
    c_seq = _c(c_seq, np.float32)
    T, R, gamma = c_seq.shape
    nf = None if n_full is None else _c(n_full, np.int32)
    cs = _c(capture_sizes, np.int32)
    sp = _c(sps, np.float32)
    l_seq = np.zeros((T, R), np.int32)
    K_seq = np.zeros(T, np.int32)
    stats = np.zeros((T, 4), np.float64)
    gap = np.zeros(T, np.float64)
    st = lib().orc_plan_cycles(_p(c_seq), _p(nf), _p(cs), _p(sp), cs.size, K_cap, mode, conf_min, lag,
                               T, R, gamma, _p(l_seq), _p(K_seq), _p(stats), _p(gap))
    return dict(status=st, l=l_seq, K_used=K_seq, theta_pred=stats[:, 0], theta_real=stats[:, 1],
                accepted=stats[:, 2].astype(np.int64), wasted=stats[:, 3].astype(np.int64), theta_gap=gap)


def fit_temperatures(z, accepted):
    """Sequential temperature scaling: z [N, gamma] float32 confidence logits,
    accepted [N, gamma] 0/1 labels -> tau, mean NLL and samples per position."""
    z = _c(z, np.float32)
    acc = _c(accepted, np.uint8)
    N, gamma = z.shape
    tau = np.zeros(gamma, np.float32)
    nll = np.zeros(gamma, np.float64)
    cnt = np.zeros(gamma, np.int32)
    st = lib().orc_fit_temperatures(_p(z), _p(acc), N, gamma, _p(tau), _p(nll), _p(cnt))
    return dict(status=st, tau=tau, nll=nll, count=cnt)


class KvState:
    """A paged KV cache's bookkeeping: committed lengths, block table, free stack."""

    def __init__(self, kv_len, block_table, free_pages, free_top, page_size):
        self.kv_len = _c(kv_len, np.int32).copy()
        self.block_table = _c(block_table, np.int32).copy()
        self.free_pages = _c(free_pages, np.int32).copy()
        self.free_top = np.array([free_top], np.int32)
        self.P = int(page_size)

    def copy(self):
        return KvState(self.kv_len, self.block_table, self.free_pages, int(self.free_top[0]), self.P)


def kv_reserve(st: KvState, l):
    l = _c(l, np.int32)
    R, max_blocks = st.block_table.shape
    reserved = np.zeros(R, np.int32)
    rc = lib().orc_kv_reserve(_p(st.kv_len), _p(l), R, st.P, _p(st.block_table), max_blocks,
                              _p(st.free_pages), _p(st.free_top), st.free_pages.size, _p(reserved))
    return rc, reserved


def kv_commit(st: KvState, l, n_acc):
    l = _c(l, np.int32)
    n_acc = _c(n_acc, np.int32)
    R, max_blocks = st.block_table.shape
    return lib().orc_kv_commit(_p(st.kv_len), _p(l), _p(n_acc), R, st.P, _p(st.block_table), max_blocks,
                               _p(st.free_pages), _p(st.free_top), st.free_pages.size)


def commit_lengths(n_acc, l, gamma):
    n_acc = _c(n_acc, np.int32)
    R = n_acc.size
    lp = None if l is None else _c(l, np.int32)
    cl = np.zeros(R, np.int32)
    cu = np.zeros(R + 1, np.int32)
    disc = np.zeros(R, np.int32)
    tot = np.zeros(1, np.int32)
    st = lib().orc_commit_lengths(_p(n_acc), _p(lp), R, gamma, _p(cl), _p(cu), _p(disc), _p(tot))
    return dict(status=st, commit_len=cl, cu_commit=cu, discard=disc, total=int(tot[0]))
