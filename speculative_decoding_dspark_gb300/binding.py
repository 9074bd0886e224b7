"""Python binding of libdspark.so: the C ABI in include/dspark.h, one function per
entry point with the same name.

Argument marshalling only -- shapes are read from the tensors, pointers and the
current CUDA stream are passed through, and a negative status raises
DSparkError.  Every step of the cycle runs in the library's CUDA kernels; there
is no CPU or PyTorch fallback: if the shared library is missing the import of
this module fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# DSPARK_LIBRARY may name another build of the library (the DSPARK_DEBUG one)
LIB_PATH = os.environ.get("DSPARK_LIBRARY") or os.path.join(_HERE, "libdspark.so")

DSPARK_OK = 0
DSPARK_ERR_INVALID_ARG = -1
DSPARK_ERR_UNSUPPORTED = -2
DSPARK_ERR_CAPACITY = -3
DSPARK_ERR_CUDA = -4
DSPARK_ERR_TIMEOUT = -5
DSPARK_ERR_DEVICE_INPUT = -6
DSPARK_ERR_WORKSPACE = -7
DSPARK_ERR_BOUNDS = -8

DSPARK_F32, DSPARK_BF16 = 0, 1
DSPARK_OP_DRAFT, DSPARK_OP_VERIFY, DSPARK_OP_SELECT, DSPARK_OP_VERIFY_MARKOV, DSPARK_OP_CALIBRATE = 0, 1, 2, 3, 4
DSPARK_OP_DRAFT_FUSED = 5
DSPARK_FUSED_MAX_D = 16384
DSPARK_DRAFT_FORCE_SIMT = 1
DSPARK_VERIFY_HOST_TARGET = 1
DSPARK_SELECT_FIXED, DSPARK_SELECT_HISTORY, DSPARK_SELECT_CURRENT, DSPARK_SELECT_FIRST_STOP = 0, 1, 2, 3
DSPARK_SELECT_CONF_CUTOFF, DSPARK_SELECT_SURVIVAL_CUTOFF = 4, 5
DSPARK_INJECT_VERIFY_BARRIER, DSPARK_INJECT_DRAFT_BARRIER = 1, 2

EXPORTED = ["dspark_status_string", "dspark_version", "dspark_workspace_size", "dspark_philox4x32_10",
            "dspark_markov_draft_uses_tensor_cores", "dspark_markov_draft", "dspark_verify",
            "dspark_select_prefix", "dspark_commit_lengths", "dspark_verify_static_scratch",
            "dspark_verify_markov", "dspark_set_wait_limit_ns", "dspark_set_fault_injection",
            "dspark_plan_cycles", "dspark_fit_temperatures", "dspark_kv_reserve", "dspark_kv_commit",
            "dspark_markov_draft_fused"]


class DSparkError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({_status_string(status)})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() "
                          "(or python -m speculative_decoding_dspark_gb300.build)")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, u32, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t
    L.dspark_status_string.argtypes = [i32]
    L.dspark_status_string.restype = ctypes.c_char_p
    L.dspark_version.restype = i32
    L.dspark_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, ctypes.c_uint]
    L.dspark_workspace_size.restype = sz
    L.dspark_markov_draft_uses_tensor_cores.argtypes = [i32, i32, i32, i32, i32, ctypes.c_uint]
    L.dspark_markov_draft_uses_tensor_cores.restype = i32
    L.dspark_markov_draft.argtypes = [vp, i32, vp, vp, i32, vp, vp, u32, f32, i32, i32, i32, i32,
                                      vp, vp, vp, vp, ctypes.c_uint, vp, sz, vp, vp]
    L.dspark_markov_draft.restype = i32
    L.dspark_markov_draft_fused.argtypes = [vp, vp, i32, vp, vp, vp, vp, u32, f32, i32, i32, i32, i32,
                                            vp, vp, vp, vp, vp, sz, vp, vp]
    L.dspark_markov_draft_fused.restype = i32
    L.dspark_verify.argtypes = [vp, vp, vp, vp, vp, vp, vp, u32, f32, i32, i32, i32, i32,
                                vp, vp, vp, vp, sz, vp, vp]
    L.dspark_verify.restype = i32
    L.dspark_select_prefix.argtypes = [vp, vp, vp, vp, i32, i32, i32, f32, i32, i32, vp, vp, vp, vp,
                                       vp, sz, vp, vp]
    L.dspark_select_prefix.restype = i32
    L.dspark_plan_cycles.argtypes = [vp, vp, vp, vp, i32, i32, i32, f32, i32, i32, i32, i32, vp, vp, vp,
                                     vp, vp]
    L.dspark_plan_cycles.restype = i32
    L.dspark_verify_markov.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, u32, f32, i32, i32,
                                       i32, i32, vp, vp, vp, vp, sz, vp, vp]
    L.dspark_verify_markov.restype = i32
    L.dspark_verify_static_scratch.argtypes = [vp, vp, vp, vp, vp, vp, vp, u32, f32, i32, i32, i32,
                                               i32, vp, vp, vp, vp, vp]
    L.dspark_verify_static_scratch.restype = i32
    L.dspark_philox4x32_10.argtypes = [vp, vp, i32, vp, vp]
    L.dspark_philox4x32_10.restype = i32
    L.dspark_commit_lengths.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, vp, vp]
    L.dspark_commit_lengths.restype = i32
    L.dspark_fit_temperatures.argtypes = [vp, vp, i32, i32, vp, vp, vp, vp, sz, vp, vp]
    L.dspark_fit_temperatures.restype = i32
    L.dspark_kv_reserve.argtypes = [vp, vp, i32, i32, vp, i32, vp, vp, i32, vp, vp, vp]
    L.dspark_kv_reserve.restype = i32
    L.dspark_kv_commit.argtypes = [vp, vp, vp, i32, i32, vp, i32, vp, vp, i32, vp, vp]
    L.dspark_kv_commit.restype = i32
    L.dspark_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.dspark_set_wait_limit_ns.restype = ctypes.c_uint64
    L.dspark_set_fault_injection.argtypes = [ctypes.c_uint]
    L.dspark_set_fault_injection.restype = ctypes.c_uint
    return L


_L = _load()


def library() -> ctypes.CDLL:
    return _L


def _status_string(status: int) -> str:
    return _L.dspark_status_string(int(status)).decode()


def dspark_status_string(status: int) -> str:
    return _status_string(status)


def dspark_version() -> int:
    return _L.dspark_version()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t):
    if t.dtype == torch.float32:
        return DSPARK_F32
    if t.dtype == torch.bfloat16:
        return DSPARK_BF16
    raise TypeError(f"expected float32 or bfloat16, got {t.dtype}")


def _check(t, name, dtype=None, shape=None, allow_none=False, allow_pinned=False):
    if t is None:
        if allow_none:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda and not (allow_pinned and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor" + (" or pinned host memory" if allow_pinned else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _raise(fn, st):
    if st != DSPARK_OK:
        raise DSparkError(fn, st)


def dspark_workspace_size(op, R, gamma, V, rank=0, max_rows=0, w_dtype=DSPARK_BF16, flags=0) -> int:
    return int(_L.dspark_workspace_size(op, R, gamma, V, rank, max_rows, w_dtype, flags))


def dspark_markov_draft_uses_tensor_cores(u_dtype, w_dtype, R, V, rank, flags=0) -> bool:
    return bool(_L.dspark_markov_draft_uses_tensor_cores(u_dtype, w_dtype, R, V, rank, flags))


def dspark_set_wait_limit_ns(limit_ns: int) -> int:
    """Limit of the grid-wide device waits for later calls (0: the 2 s default);
    returns the previous limit."""
    return int(_L.dspark_set_wait_limit_ns(int(limit_ns)))


def dspark_set_fault_injection(mask: int) -> int:
    """Test hook: make the named grid-wide waits run out (see dspark.h); returns
    the previous mask."""
    return int(_L.dspark_set_fault_injection(int(mask)))


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A caller-owned workspace buffer (torch allocations are 256-byte aligned)."""
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def dspark_markov_draft(U, W1, W2, anchor, seeds, cycle, temperature, draft_tokens, q_lse=None,
                        q_tok=None, q_logits=None, ws=None, dev_status=None, flags=0, stream=None):
    R, gamma, V = U.shape
    rank = W1.shape[1]
    _check(U, "U", shape=(R, gamma, V))
    _check(W1, "W1", dtype=W2.dtype, shape=(V, rank))
    _check(W2, "W2", shape=(V, rank))
    _check(anchor, "anchor", torch.int32, (R,))
    _check(seeds, "seeds", torch.int64, (R,), allow_none=True)
    _check(draft_tokens, "draft_tokens", torch.int32, (R, gamma))
    _check(q_lse, "q_lse", torch.float32, (R, gamma), allow_none=True)
    _check(q_tok, "q_tok", torch.float32, (R, gamma), allow_none=True)
    _check(q_logits, "q_logits", torch.float32, (R, gamma, V), allow_none=True)
    _check(ws, "ws", torch.uint8)
    _check(dev_status, "dev_status", torch.int32, allow_none=True)
    st = _L.dspark_markov_draft(_ptr(U), _dtype_code(U), _ptr(W1), _ptr(W2), _dtype_code(W2),
                                _ptr(anchor), _ptr(seeds), int(cycle), float(temperature), R,
                                gamma, V, rank, _ptr(draft_tokens), _ptr(q_lse), _ptr(q_tok),
                                _ptr(q_logits), int(flags), _ptr(ws), ws.numel(),
                                _ptr(dev_status), _stream(stream))
    _raise("dspark_markov_draft", st)


def dspark_markov_draft_fused(h, W_lm, W1, W2, anchor, seeds, cycle, temperature, draft_tokens, q_lse=None,
                              q_tok=None, q_logits=None, ws=None, dev_status=None, stream=None):
    R, gamma, d = h.shape
    V = W_lm.shape[0]
    rank = W1.shape[1]
    _check(h, "h", torch.bfloat16, (R, gamma, d))
    _check(W_lm, "W_lm", torch.bfloat16, (V, d))
    _check(W1, "W1", torch.bfloat16, (V, rank))
    _check(W2, "W2", torch.bfloat16, (V, rank))
    _check(anchor, "anchor", torch.int32, (R,))
    _check(seeds, "seeds", torch.int64, (R,), allow_none=True)
    _check(draft_tokens, "draft_tokens", torch.int32, (R, gamma))
    _check(q_lse, "q_lse", torch.float32, (R, gamma), allow_none=True)
    _check(q_tok, "q_tok", torch.float32, (R, gamma), allow_none=True)
    _check(q_logits, "q_logits", torch.float32, (R, gamma, V), allow_none=True)
    _check(ws, "ws", torch.uint8)
    _check(dev_status, "dev_status", torch.int32, allow_none=True)
    st = _L.dspark_markov_draft_fused(_ptr(h), _ptr(W_lm), d, _ptr(W1), _ptr(W2), _ptr(anchor), _ptr(seeds),
                                      int(cycle), float(temperature), R, gamma, V, rank, _ptr(draft_tokens),
                                      _ptr(q_lse), _ptr(q_tok), _ptr(q_logits), _ptr(ws), ws.numel(),
                                      _ptr(dev_status), _stream(stream))
    _raise("dspark_markov_draft_fused", st)


def dspark_verify(target_logits, cu_seqlens, draft_tokens, q_logits, q_lse, q_tok, seeds, cycle,
                  temperature, max_rows, n_accepted, out_tokens, p_tok=None, ws=None,
                  dev_status=None, stream=None):
    R, gamma = draft_tokens.shape
    V = target_logits.shape[1]
    _check(target_logits, "target_logits", torch.float32)
    _check(cu_seqlens, "cu_seqlens", torch.int32, (R + 1,))
    _check(draft_tokens, "draft_tokens", torch.int32)
    _check(q_logits, "q_logits", torch.float32, (R, gamma, V), allow_none=True)
    _check(q_lse, "q_lse", torch.float32, (R, gamma), allow_none=True)
    _check(q_tok, "q_tok", torch.float32, (R, gamma), allow_none=True)
    _check(seeds, "seeds", torch.int64, (R,), allow_none=True)
    _check(n_accepted, "n_accepted", torch.int32, (R,))
    _check(out_tokens, "out_tokens", torch.int32, (R, gamma + 1))
    _check(p_tok, "p_tok", torch.float32, (R, gamma), allow_none=True)
    _check(ws, "ws", torch.uint8)
    _check(dev_status, "dev_status", torch.int32, allow_none=True)
    if target_logits.shape[0] < max_rows:
        raise ValueError("target_logits has fewer rows than max_rows")
    st = _L.dspark_verify(_ptr(target_logits), _ptr(cu_seqlens), _ptr(draft_tokens), _ptr(q_logits),
                          _ptr(q_lse), _ptr(q_tok), _ptr(seeds), int(cycle), float(temperature), R,
                          gamma, V, int(max_rows), _ptr(n_accepted), _ptr(out_tokens), _ptr(p_tok),
                          _ptr(ws), ws.numel(), _ptr(dev_status), _stream(stream))
    _raise("dspark_verify", st)


def dspark_verify_markov(target_logits, cu_seqlens, draft_tokens, U, W1, W2, anchor, q_lse, q_tok, seeds,
                         cycle, temperature, max_rows, n_accepted, out_tokens, p_tok=None, ws=None,
                         dev_status=None, stream=None):
    R, gamma = draft_tokens.shape
    V = target_logits.shape[1]
    rank = W1.shape[1]
    _check(target_logits, "target_logits", torch.float32, allow_pinned=True)
    _check(cu_seqlens, "cu_seqlens", torch.int32, (R + 1,))
    _check(draft_tokens, "draft_tokens", torch.int32)
    _check(U, "U", torch.bfloat16, (R, gamma, V))
    _check(W1, "W1", torch.bfloat16, (V, rank))
    _check(W2, "W2", torch.bfloat16, (V, rank))
    _check(anchor, "anchor", torch.int32, (R,))
    _check(q_lse, "q_lse", torch.float32, (R, gamma), allow_none=True)
    _check(q_tok, "q_tok", torch.float32, (R, gamma), allow_none=True)
    _check(seeds, "seeds", torch.int64, (R,), allow_none=True)
    _check(n_accepted, "n_accepted", torch.int32, (R,))
    _check(out_tokens, "out_tokens", torch.int32, (R, gamma + 1))
    _check(p_tok, "p_tok", torch.float32, (R, gamma), allow_none=True)
    _check(ws, "ws", torch.uint8)
    _check(dev_status, "dev_status", torch.int32, allow_none=True)
    if target_logits.shape[0] < max_rows:
        raise ValueError("target_logits has fewer rows than max_rows")
    st = _L.dspark_verify_markov(_ptr(target_logits), _ptr(cu_seqlens), _ptr(draft_tokens), _ptr(U), _ptr(W1),
                                 _ptr(W2), _ptr(anchor), rank, _ptr(q_lse), _ptr(q_tok), _ptr(seeds),
                                 int(cycle), float(temperature), R, gamma, V, int(max_rows),
                                 _ptr(n_accepted), _ptr(out_tokens), _ptr(p_tok), _ptr(ws), ws.numel(),
                                 _ptr(dev_status), _stream(stream))
    _raise("dspark_verify_markov", st)


def dspark_verify_static_scratch(target_logits, cu_seqlens, draft_tokens, q_logits, q_lse, q_tok,
                                 seeds, cycle, temperature, max_rows, n_accepted, out_tokens,
                                 p_tok=None, dev_status=None, stream=None):
    """dspark_verify without a workspace argument, for callers that are not
    allowed to allocate device memory (for example a plugin inside a serving
    engine whose device memory all belongs to the engine's pool).  The scratch
    is a fixed 4 MiB array inside the library, shared by every call on a
    device: calls must not overlap on the GPU, the first call on a device
    (which looks the array up) should happen before any stream capture, and
    the entry point must not be used after a cudaDeviceReset."""
    R, gamma = draft_tokens.shape
    V = target_logits.shape[1]
    _check(target_logits, "target_logits", torch.float32)
    _check(cu_seqlens, "cu_seqlens", torch.int32, (R + 1,))
    _check(draft_tokens, "draft_tokens", torch.int32)
    _check(q_logits, "q_logits", torch.float32, (R, gamma, V), allow_none=True)
    _check(q_lse, "q_lse", torch.float32, (R, gamma), allow_none=True)
    _check(q_tok, "q_tok", torch.float32, (R, gamma), allow_none=True)
    _check(seeds, "seeds", torch.int64, (R,), allow_none=True)
    _check(n_accepted, "n_accepted", torch.int32, (R,))
    _check(out_tokens, "out_tokens", torch.int32, (R, gamma + 1))
    _check(p_tok, "p_tok", torch.float32, (R, gamma), allow_none=True)
    _check(dev_status, "dev_status", torch.int32, allow_none=True)
    if target_logits.shape[0] < max_rows:
        raise ValueError("target_logits has fewer rows than max_rows")
    st = _L.dspark_verify_static_scratch(_ptr(target_logits), _ptr(cu_seqlens), _ptr(draft_tokens),
                                         _ptr(q_logits), _ptr(q_lse), _ptr(q_tok), _ptr(seeds),
                                         int(cycle), float(temperature), R, gamma, V, int(max_rows),
                                         _ptr(n_accepted), _ptr(out_tokens), _ptr(p_tok),
                                         _ptr(dev_status), _stream(stream))
    _raise("dspark_verify_static_scratch", st)


def dspark_select_prefix(c, c_hist, capture_sizes, sps, K_cap, mode, a, l, cu_seqlens, K_used,
                         ws=None, dev_status=None, stream=None, conf_min=0.0):
    R, gamma = c.shape
    _check(c, "c", torch.float32)
    _check(c_hist, "c_hist", torch.float32, (R, gamma), allow_none=True)
    _check(capture_sizes, "capture_sizes", torch.int32, allow_none=True)
    _check(sps, "sps", torch.float32, allow_none=True)
    _check(a, "a", torch.float32, (R, gamma))
    _check(l, "l", torch.int32, (R,))
    _check(cu_seqlens, "cu_seqlens", torch.int32, (R + 1,))
    _check(K_used, "K_used", torch.int32, (1,))
    _check(dev_status, "dev_status", torch.int32, allow_none=True)
    n_steps = 0 if capture_sizes is None else capture_sizes.numel()
    if sps is not None and sps.numel() != n_steps:
        raise ValueError("sps and capture_sizes differ in length")
    st = _L.dspark_select_prefix(_ptr(c), _ptr(c_hist), _ptr(capture_sizes), _ptr(sps), n_steps,
                                 int(K_cap), int(mode), float(conf_min), R, gamma, _ptr(a), _ptr(l),
                                 _ptr(cu_seqlens), _ptr(K_used), _ptr(ws),
                                 0 if ws is None else ws.numel(), _ptr(dev_status), _stream(stream))
    _raise("dspark_select_prefix", st)


def dspark_plan_cycles(c_seq, n_full, capture_sizes, sps, K_cap, mode, l_seq, K_seq, stats, conf_min=0.0,
                       lag=2, dev_status=None, stream=None):
    T, R, gamma = c_seq.shape
    _check(c_seq, "c_seq", torch.float32)
    _check(n_full, "n_full", torch.int32, (T, R), allow_none=True)
    _check(capture_sizes, "capture_sizes", torch.int32)
    _check(sps, "sps", torch.float32, (capture_sizes.numel(),))
    _check(l_seq, "l_seq", torch.int32, (T, R))
    _check(K_seq, "K_seq", torch.int32, (T,))
    _check(stats, "stats", torch.float64, (T, 4))
    _check(dev_status, "dev_status", torch.int32, allow_none=True)
    st = _L.dspark_plan_cycles(_ptr(c_seq), _ptr(n_full), _ptr(capture_sizes), _ptr(sps), capture_sizes.numel(),
                               int(K_cap), int(mode), float(conf_min), int(lag), T, R, gamma, _ptr(l_seq),
                               _ptr(K_seq), _ptr(stats), _ptr(dev_status), _stream(stream))
    _raise("dspark_plan_cycles", st)


def dspark_fit_temperatures(z, accepted, tau, nll=None, count=None, ws=None, dev_status=None, stream=None):
    N, gamma = z.shape
    _check(z, "z", torch.float32)
    _check(accepted, "accepted", torch.uint8, (N, gamma))
    _check(tau, "tau", torch.float32, (gamma,))
    _check(nll, "nll", torch.float64, (gamma,), allow_none=True)
    _check(count, "count", torch.int32, (gamma,), allow_none=True)
    _check(ws, "ws", torch.uint8)
    _check(dev_status, "dev_status", torch.int32, allow_none=True)
    st = _L.dspark_fit_temperatures(_ptr(z), _ptr(accepted), N, gamma, _ptr(tau), _ptr(nll), _ptr(count),
                                    _ptr(ws), ws.numel(), _ptr(dev_status), _stream(stream))
    _raise("dspark_fit_temperatures", st)


def dspark_kv_reserve(kv_len, l, page_size, block_table, free_pages, free_top, reserved=None, dev_status=None,
                      stream=None):
    R, max_blocks = block_table.shape
    _check(kv_len, "kv_len", torch.int32, (R,))
    _check(l, "l", torch.int32, (R,))
    _check(block_table, "block_table", torch.int32)
    _check(free_pages, "free_pages", torch.int32)
    _check(free_top, "free_top", torch.int32, (1,))
    _check(reserved, "reserved", torch.int32, (R,), allow_none=True)
    _check(dev_status, "dev_status", torch.int32, allow_none=True)
    _raise("dspark_kv_reserve",
           _L.dspark_kv_reserve(_ptr(kv_len), _ptr(l), R, int(page_size), _ptr(block_table), max_blocks,
                                _ptr(free_pages), _ptr(free_top), free_pages.numel(), _ptr(reserved),
                                _ptr(dev_status), _stream(stream)))


def dspark_kv_commit(kv_len, l, n_accepted, page_size, block_table, free_pages, free_top, dev_status=None,
                     stream=None):
    R, max_blocks = block_table.shape
    _check(kv_len, "kv_len", torch.int32, (R,))
    _check(l, "l", torch.int32, (R,))
    _check(n_accepted, "n_accepted", torch.int32, (R,))
    _check(block_table, "block_table", torch.int32)
    _check(free_pages, "free_pages", torch.int32)
    _check(free_top, "free_top", torch.int32, (1,))
    _check(dev_status, "dev_status", torch.int32, allow_none=True)
    _raise("dspark_kv_commit",
           _L.dspark_kv_commit(_ptr(kv_len), _ptr(l), _ptr(n_accepted), R, int(page_size), _ptr(block_table),
                               max_blocks, _ptr(free_pages), _ptr(free_top), free_pages.numel(), _ptr(dev_status),
                               _stream(stream)))


def dspark_philox4x32_10(ctr, keys, out, stream=None):
    n = keys.shape[0]
    _check(ctr, "ctr", torch.int32, (n, 4))
    _check(keys, "keys", torch.int64, (n,))
    _check(out, "out", torch.int32, (n, 4))
    _raise("dspark_philox4x32_10",
           _L.dspark_philox4x32_10(_ptr(ctr), _ptr(keys), n, _ptr(out), _stream(stream)))


def dspark_commit_lengths(n_accepted, l, gamma, commit_len, cu_commit, discard, total=None,
                          dev_status=None, stream=None):
    R = n_accepted.shape[0]
    _check(n_accepted, "n_accepted", torch.int32, (R,))
    _check(l, "l", torch.int32, (R,), allow_none=True)
    _check(commit_len, "commit_len", torch.int32, (R,))
    _check(cu_commit, "cu_commit", torch.int32, (R + 1,))
    _check(discard, "discard", torch.int32, (R,))
    _check(total, "total", torch.int32, (1,), allow_none=True)
    _check(dev_status, "dev_status", torch.int32, allow_none=True)
    st = _L.dspark_commit_lengths(_ptr(n_accepted), _ptr(l), R, int(gamma), _ptr(commit_len),
                                  _ptr(cu_commit), _ptr(discard), _ptr(total), _ptr(dev_status),
                                  _stream(stream))
    _raise("dspark_commit_lengths", st)
