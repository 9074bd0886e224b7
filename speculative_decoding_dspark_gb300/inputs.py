"""Seeded synthetic inputs for the DSpark decode-cycle hot path.

This module only makes input tensors (numpy, host memory) with the shapes and
value laws of the workloads the library is measured on; it contains none of
the cycle's arithmetic (no bias, softmax, sampling, acceptance or selection),
so the CUDA path and the CPU oracle can both consume its bytes without sharing
any of the method's code.  Random numbers the method itself draws come from
the per-request Philox seeds produced here, which each side expands with its
own generator.

Workloads (sizes and laws; the model weights and benchmark prompts of the
pages are not available, so every tensor is synthetic):

* ``tiny_exhaustive``  R=1, V=64, gamma=5, rank=8, fp32 W1/W2 ~ N(0,0.5^2),
  U[5,64] ~ N(0,2^2), target row j = 0.7*U_j + 0.3*N(0,2^2); the row after the
  block uses an extra U-law row.  T = 1.0 and greedy.
* ``qwen3_8b_greedy``  R=16, V=151936 (Qwen3 vocabulary), gamma=7 (the released
  block-7 drafts), rank=256; bf16 W ~ N(0,0.02^2), bf16 U ~ N(0,3^2); fp32
  target row j = 0.6*U_j + 0.8*3*Z (correlation 0.6, sigma 3), row 7 = 3*Z.
  Greedy.
* ``batched_sampling``  R=128, V=151936, gamma=7, rank=512, T=0.7, the same laws,
  an independent Philox seed per request.
* ``varlen_verify``  R=256, V=129280 (DeepSeek-V4 vocabulary), gamma=5 (V4 block
  size), rank=512 (V4-Pro Markov rank); verify lengths l[r] uniform in 0..5,
  packed rows with cu_seqlens, T=1.0.
* ``confidence_scheduled``  R=512, V=129280, gamma=5, rank=512; confidences
  c = sigmoid(N(1,1.5^2) / tau_k), tau = [1.0, 1.1, 1.2, 1.3, 1.4]; history
  confidences from an independent stream; capture sizes 64..1024 with the
  synthetic step-rate staircase SPS(S) = 1/(10 ms + 20 us * S); K_cap = 1024;
  T = 1.0.
* ``fused_logits``  the batched-sampling shape (R=128, V=151936, gamma=7,
  rank=512, T=0.7) with the base logits formed from the drafter's hidden
  states instead of given: h[R, gamma, d] ~ N(0, 1) bf16 with d = 4096 (the
  hidden size of Qwen3-8B, whose vocabulary V is) and a shared lm_head
  W_lm[V, d] ~ N(0, (3 / sqrt(d))^2) bf16, so that U = W_lm . h keeps the
  N(0, 3^2) law of the other workloads; Markov factors as there.
"""
from __future__ import annotations

import numpy as np

GOLDEN_RATIO_64 = 0x9E3779B97F4A7C15
BASE_SEED = 0x5EED0000

WORKLOADS = {
    "tiny_exhaustive": dict(index=0, R=1, V=64, gamma=5, rank=8, w_dtype="f32", w_sigma=0.5,
                            u_dtype="f32", u_sigma=2.0, t_u=0.7, t_z=0.3 * 2.0,
                            bonus_law="extra_u", temperature=1.0),
    "qwen3_8b_greedy": dict(index=1, R=16, V=151936, gamma=7, rank=256, w_dtype="bf16",
                            w_sigma=0.02, u_dtype="bf16", u_sigma=3.0, t_u=0.6, t_z=0.8 * 3.0,
                            bonus_law="z", temperature=0.0),
    "batched_sampling": dict(index=2, R=128, V=151936, gamma=7, rank=512, w_dtype="bf16",
                             w_sigma=0.02, u_dtype="bf16", u_sigma=3.0, t_u=0.6, t_z=0.8 * 3.0,
                             bonus_law="z", temperature=0.7),
    "varlen_verify": dict(index=3, R=256, V=129280, gamma=5, rank=512, w_dtype="bf16",
                          w_sigma=0.02, u_dtype="bf16", u_sigma=3.0, t_u=0.6, t_z=0.8 * 3.0,
                          bonus_law="z", temperature=1.0, varlen=True),
    "confidence_scheduled": dict(index=4, R=512, V=129280, gamma=5, rank=512, w_dtype="bf16",
                                 w_sigma=0.02, u_dtype="bf16", u_sigma=3.0, t_u=0.6,
                                 t_z=0.8 * 3.0, bonus_law="z", temperature=1.0,
                                 confidence=True, K_cap=1024,
                                 tau=[1.0, 1.1, 1.2, 1.3, 1.4],
                                 capture_sizes=[64, 128, 256, 512, 1024]),
    "fused_logits": dict(index=5, R=128, V=151936, gamma=7, rank=512, d=4096, w_dtype="bf16",
                         w_sigma=0.02, u_dtype="bf16", u_sigma=3.0, t_u=0.6, t_z=0.8 * 3.0,
                         bonus_law="z", temperature=0.7),
}


def rng(seed: int, stream: int) -> np.random.Generator:
    """Independent numpy stream ``stream`` of base seed ``seed``."""
    return np.random.default_rng([int(seed) & 0xFFFFFFFFFFFFFFFF, int(stream)])


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def as_f32(x: np.ndarray) -> np.ndarray:
    return bf16_to_f32(x) if x.dtype == np.uint16 else np.asarray(x, np.float32)


def request_seeds(base: int, R: int) -> np.ndarray:
    """Per-request 64-bit Philox keys: base + r * golden-ratio constant (mod 2^64)."""
    r = np.arange(R, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return (np.uint64(base) + r * np.uint64(GOLDEN_RATIO_64)).astype(np.uint64)


def sps_staircase(capture_sizes) -> np.ndarray:
    """Synthetic engine step rate per capture size: 1 / (10 ms + 20 us * size)."""
    s = np.asarray(capture_sizes, np.float64)
    return (1.0 / (0.010 + 20e-6 * s)).astype(np.float32)


def _normal(g: np.random.Generator, shape, sigma: float) -> np.ndarray:
    out = g.standard_normal(size=shape, dtype=np.float32)
    out *= np.float32(sigma)
    return out


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits(x) if dtype == "bf16" else np.ascontiguousarray(x, np.float32)


def workload(name: str, seed_offset: int = 0, **overrides) -> dict:
    """The size and law parameters of a workload, with optional size overrides
    (R, V, gamma, rank, temperature) for reduced-size test cases."""
    w = dict(WORKLOADS[name])
    w.update(overrides)
    w["name"] = name
    w["seed"] = BASE_SEED + w["index"] + 7919 * int(seed_offset)
    return w


def draft_inputs(w: dict) -> dict:
    """Markov-head factors, base logits, anchors and per-request seeds."""
    R, V, gamma, rank, seed = w["R"], w["V"], w["gamma"], w["rank"], w["seed"]
    W1 = _store(_normal(rng(seed, 1), (V, rank), w["w_sigma"]), w["w_dtype"])
    W2 = _store(_normal(rng(seed, 2), (V, rank), w["w_sigma"]), w["w_dtype"])
    U = _store(_normal(rng(seed, 3), (R, gamma, V), w["u_sigma"]), w["u_dtype"])
    anchor = rng(seed, 4).integers(0, V, size=R, dtype=np.int64).astype(np.int32)
    return dict(W1=W1, W2=W2, U=U, anchor=anchor, seeds=request_seeds(seed, R),
                temperature=np.float32(w["temperature"]))


def fused_inputs(w: dict) -> dict:
    """Drafter hidden states h [R, gamma, d] ~ N(0, 1) and the shared lm_head
    W_lm [V, d] ~ N(0, (u_sigma / sqrt(d))^2), both bf16, with the Markov factors,
    anchors and seeds of draft_inputs (streams 1, 2, 4 as there; h and W_lm from
    streams 13 and 14, so no U is drawn)."""
    R, V, gamma, rank, d, seed = w["R"], w["V"], w["gamma"], w["rank"], w["d"], w["seed"]
    W1 = _store(_normal(rng(seed, 1), (V, rank), w["w_sigma"]), w["w_dtype"])
    W2 = _store(_normal(rng(seed, 2), (V, rank), w["w_sigma"]), w["w_dtype"])
    h = bf16_bits(_normal(rng(seed, 13), (R, gamma, d), 1.0))
    W_lm = np.empty((V, d), np.uint16)
    g = rng(seed, 14)
    sig = w["u_sigma"] / np.sqrt(d)
    for v0 in range(0, V, 8192):  # in slices: the fp32 draw of a full lm_head would double the memory
        W_lm[v0:v0 + 8192] = bf16_bits(_normal(g, (min(8192, V - v0), d), sig))
    anchor = rng(seed, 4).integers(0, V, size=R, dtype=np.int64).astype(np.int32)
    return dict(W1=W1, W2=W2, h=h, W_lm=W_lm, anchor=anchor, seeds=request_seeds(seed, R),
                temperature=np.float32(w["temperature"]))


def target_full(w: dict, U: np.ndarray) -> np.ndarray:
    """Target logits for every position 0..gamma of every request, [R, gamma+1, V] fp32.
    Row j < gamma correlates with the drafter's base logits U_j; row gamma (after
    the block) follows the bonus law."""
    R, V, gamma, seed = w["R"], w["V"], w["gamma"], w["seed"]
    g = rng(seed, 5)
    T = np.empty((R, gamma + 1, V), np.float32)
    Uf = as_f32(U)
    for r in range(R):
        z = _normal(g, (gamma + 1, V), 1.0)
        T[r, :gamma] = np.float32(w["t_u"]) * Uf[r] + np.float32(w["t_z"]) * z[:gamma]
        if w["bonus_law"] == "extra_u":
            extra = _normal(g, (V,), w["u_sigma"])
            T[r, gamma] = np.float32(w["t_u"]) * extra + np.float32(w["t_z"]) * z[gamma]
        else:
            T[r, gamma] = np.float32(w["u_sigma"]) * z[gamma]
    return T


def verify_lengths(w: dict) -> np.ndarray:
    """Per-request verify lengths: uniform in 0..gamma for the variable-length
    workload, gamma for every request otherwise."""
    R, gamma = w["R"], w["gamma"]
    if w.get("varlen"):
        return rng(w["seed"], 7).integers(0, gamma + 1, size=R, dtype=np.int64).astype(np.int32)
    return np.full(R, gamma, np.int32)


def cu_from_lengths(l: np.ndarray) -> np.ndarray:
    """Row boundaries of the packed verify rows: request r owns l[r] + 1 rows."""
    cu = np.zeros(len(l) + 1, np.int32)
    cu[1:] = np.cumsum(np.asarray(l, np.int64) + 1)
    return cu


def pack_rows(full: np.ndarray, l: np.ndarray) -> np.ndarray:
    """Pack rows 0..l[r] of every request back to back (no padding)."""
    return np.ascontiguousarray(np.concatenate([full[r, : int(l[r]) + 1] for r in range(len(l))], 0))


def confidence_inputs(w: dict) -> dict:
    """Calibrated per-position confidences c = sigmoid(z / tau_k), z ~ N(1, 1.5^2),
    for the current cycle and, from an independent stream, for the cycle whose
    confidences fix the physical capacity."""
    R, gamma, seed = w["R"], w["gamma"], w["seed"]
    # per-position calibration temperatures; positions past the given list
    # continue the workload's +0.1 step
    given = list(w.get("tau", []))
    tau = np.asarray([given[k] if k < len(given) else 1.0 + 0.1 * k for k in range(gamma)],
                     np.float64)

    def conf(stream):
        z = 1.0 + 1.5 * rng(seed, stream).standard_normal((R, gamma))
        return (1.0 / (1.0 + np.exp(-z / tau[None, :]))).astype(np.float32)

    sizes = np.asarray(w.get("capture_sizes", [64, 128, 256, 512, 1024]), np.int32)
    return dict(c=conf(8), c_hist=conf(9), capture_sizes=sizes, sps=sps_staircase(sizes),
                K_cap=int(w.get("K_cap", R * (gamma + 1))), tau=tau)


def confidence_sequence(w: dict, n_cycles: int, drift: float = 0.0) -> dict:
    """Confidences of n_cycles consecutive cycles of the same R request slots
    ([n_cycles, R, gamma], each cycle drawn from the workload's law) and, as the
    synthetic stand-in for the target's verdicts, n_full [n_cycles, R]: how many
    leading drafts the target accepts, drawn so that draft k survives with
    probability c[t, r, k] given the ones before it (the confidences are
    calibrated conditional acceptance rates).  drift > 0 adds a batch-wide shift
    of the confidence logits that wanders from cycle to cycle (a random walk of
    step `drift` pulled back towards 0 by 10% a cycle: the batch's mix of easy and
    hard text changing over time)."""
    R, gamma, seed = w["R"], w["gamma"], w["seed"]
    tau = confidence_inputs(w)["tau"]
    z = 1.0 + 1.5 * rng(seed, 10).standard_normal((n_cycles, R, gamma))
    if drift > 0.0:
        steps = drift * rng(seed, 12).standard_normal(n_cycles)
        shift = np.zeros(n_cycles)
        for t in range(1, n_cycles):
            shift[t] = 0.9 * shift[t - 1] + steps[t]
        z = z + shift[:, None, None]
    c = (1.0 / (1.0 + np.exp(-z / tau[None, None, :]))).astype(np.float32)
    u = rng(seed, 11).random((n_cycles, R, gamma), dtype=np.float32)
    ok = u < c
    n_full = np.where(ok.all(axis=2), gamma, np.argmin(ok, axis=2)).astype(np.int32)
    sizes = np.asarray(w.get("capture_sizes", [64, 128, 256, 512, 1024]), np.int32)
    return dict(c=c, n_full=n_full, capture_sizes=sizes, sps=sps_staircase(sizes),
                K_cap=int(w.get("K_cap", R * (gamma + 1))))


def calibration_samples(w: dict, n_samples: int, tau_true=None) -> dict:
    """Labelled samples for the confidence calibration: the confidence head's raw
    logits z [n_samples, gamma] (the workload's law, N(1, 1.5^2)) and 0/1
    acceptance labels drawn left to right, position k accepted with
    probability sigmoid(z_k / tau_true_k) when every earlier position was
    (later positions of a rejected sample are labelled 0, as a verify that
    stopped there would record).  tau_true defaults to the workload's
    per-position temperatures."""
    gamma, seed = w["gamma"], w["seed"]
    tau = np.asarray(confidence_inputs(w)["tau"] if tau_true is None else tau_true, np.float64)
    z = (1.0 + 1.5 * rng(seed, 13).standard_normal((n_samples, gamma))).astype(np.float32)
    u = rng(seed, 14).random((n_samples, gamma))
    p = 1.0 / (1.0 + np.exp(-z.astype(np.float64) / tau[None, :]))
    ok = u < p
    reached = np.cumprod(ok, axis=1).astype(bool)
    return dict(z=z, accepted=reached.astype(np.uint8), tau_true=tau.astype(np.float32))


def kv_state(w: dict, page_size: int = 16, max_len: int = 4096, spare_pages: int = 0,
             headroom: int = 0) -> dict:
    """A paged KV cache's bookkeeping before a cycle: committed lengths
    kv_len [R] uniform in 0 .. max_len - (gamma + 1) * 2 tokens, a block table
    [R, max_blocks] (room for max_len + headroom tokens) holding each request's
    committed pages (page ids a random permutation, -1 past the committed
    ones), and a stack of free pages with enough room for every request to
    verify gamma + 1 more rows (plus spare_pages)."""
    R, gamma, seed = w["R"], w["gamma"], w["seed"]
    g = rng(seed, 15)
    max_blocks = -(-(max_len + headroom) // page_size)
    kv_len = g.integers(0, max_len - 2 * (gamma + 1), size=R, dtype=np.int64).astype(np.int32)
    held = -(-kv_len.astype(np.int64) // page_size)
    extra = -(-(kv_len.astype(np.int64) + gamma + 1) // page_size) - held
    n_pages = int(held.sum() + extra.sum()) + spare_pages
    perm = g.permutation(n_pages).astype(np.int32)
    bt = np.full((R, max_blocks), -1, np.int32)
    o = 0
    for r in range(R):
        bt[r, : held[r]] = perm[o: o + held[r]]
        o += int(held[r])
    free = np.zeros(n_pages, np.int32)
    free[: n_pages - o] = perm[o:]
    return dict(kv_len=kv_len, block_table=bt, free_pages=free, free_top=n_pages - o,
                page_size=page_size, n_pages=n_pages)
