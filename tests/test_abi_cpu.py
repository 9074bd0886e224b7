"""CPU-only checks of the C ABI: the library builds and loads without a GPU,
exports every function include/dspark.h declares, and its host-side argument
checks answer without touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_dspark_gb300 import build
    try:
        build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dspark_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n
    from speculative_decoding_dspark_gb300 import binding
    assert set(binding.EXPORTED) == set(names)


def test_debug_build_exports_every_declared_symbol():
    """The DSPARK_DEBUG build (device-side bounds checks) compiles and exports the
    same functions."""
    from speculative_decoding_dspark_gb300 import build
    try:
        build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    dbg = ctypes.CDLL(build.build(debug=True))
    for n in declared_functions():
        assert hasattr(dbg, n), n
    dbg.dspark_status_string.restype = ctypes.c_char_p
    assert b"bounds" in dbg.dspark_status_string(-8)


def test_status_strings_and_version(lib):
    lib.dspark_status_string.restype = ctypes.c_char_p
    for code in range(0, -9, -1):
        s = lib.dspark_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.dspark_status_string(-99).decode() == "unknown status"
    assert lib.dspark_version() >= 100


def test_workspace_sizes(lib):
    ws = lib.dspark_workspace_size
    ws.restype = ctypes.c_size_t
    ws.argtypes = [ctypes.c_int] * 7 + [ctypes.c_uint]
    # verify: counters + statistics of every request's first row (1024-element
    # units) + extra-token partials (8192-element chunks), 256-byte aligned pieces
    v = ws(1, 128, 7, 151936, 0, 1024, 0, 0)
    nchunk = (151936 + 8191) // 8192
    nsub = (151936 + 1023) // 1024
    assert v >= 128 * nsub * 16 + 128 * nchunk * 32
    assert v % 256 == 0
    assert ws(1, 0, 7, 151936, 0, 1024, 0, 0) == 0
    assert ws(2, 512, 5, 0, 0, 0, 0, 0) == 0
    # draft on the CUDA cores keeps an fp32 bias row per request
    d = ws(0, 4, 5, 64, 8, 0, 0, 1)
    assert d >= 4 * 64 * 4
    assert ws(0, 4, 0, 64, 8, 0, 0, 0) == 0
    # calibration: partial sums per position, independent of the sample count
    assert ws(4, 0, 5, 0, 0, 0, 0, 0) > 0 and ws(4, 0, 17, 0, 0, 0, 0, 0) == 0
    # fused drafter logits: the tensor-core draft's keys, step counters and pieces
    f = ws(5, 128, 7, 151936, 512, 0, 1, 0)
    assert f >= 7 * 128 * 8 and f % 256 == 0
    assert ws(5, 128, 0, 151936, 512, 0, 1, 0) == 0 and ws(5, 0, 7, 151936, 512, 0, 1, 0) == 0


def test_host_argument_checks(lib):
    vp = ctypes.c_void_p
    f = lib.dspark_markov_draft
    f.restype = ctypes.c_int
    f.argtypes = [vp, ctypes.c_int, vp, vp, ctypes.c_int, vp, vp, ctypes.c_uint32, ctypes.c_float,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp,
                  ctypes.c_uint, vp, ctypes.c_size_t, vp, vp]
    fake = vp(4096)
    args = [fake, 1, fake, fake, 1, fake, fake, 0, 0.7, 4, 5, 64, 8, fake, fake, fake, None, 0,
            vp(256 * 64), 1 << 20, None, None]
    a = list(args); a[0] = None
    assert f(*a) == -1          # NULL U
    a = list(args); a[10] = 17
    assert f(*a) == -1          # gamma > 16
    a = list(args); a[8] = -1.0
    assert f(*a) == -1          # negative temperature
    a = list(args); a[6] = None
    assert f(*a) == -1          # sampling without seeds
    a = list(args); a[18] = vp(4100)
    assert f(*a) == -7          # misaligned workspace
    a = list(args); a[19] = 16
    assert f(*a) == -7          # workspace too small

    fd = lib.dspark_markov_draft_fused
    fd.restype = ctypes.c_int
    fd.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp, vp, ctypes.c_uint32, ctypes.c_float,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp,
                   vp, ctypes.c_size_t, vp, vp]
    # h, W_lm, d, W1, W2, anchor, seeds, cycle, T, R, gamma, V, rank, y, q_lse, q_tok, q_logits, ws, bytes, status, stream
    fargs = [fake, fake, 256, fake, fake, fake, fake, 0, 0.7, 4, 5, 4096, 64, fake, fake, fake, None,
             vp(256 * 64), 1 << 20, None, None]
    a = list(fargs); a[1] = None
    assert fd(*a) == -1         # NULL lm_head
    a = list(fargs); a[2] = 0
    assert fd(*a) == -1         # no hidden size
    a = list(fargs); a[6] = None
    assert fd(*a) == -1         # sampling without seeds
    a = list(fargs); a[10] = 17
    assert fd(*a) == -1         # gamma > 16
    a = list(fargs); a[17] = vp(4100)
    assert fd(*a) == -7         # misaligned workspace
    a = list(fargs); a[2] = 100
    assert fd(*a) == -2         # hidden size not a multiple of 64
    a = list(fargs); a[2] = 16384 + 64
    assert fd(*a) == -2         # hidden size above DSPARK_FUSED_MAX_D

    s = lib.dspark_select_prefix
    s.restype = ctypes.c_int
    s.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                  ctypes.c_int, vp, vp, vp, vp, vp, ctypes.c_size_t, vp, vp]
    base = [fake, None, None, None, 0, 16, 0, 0.0, 4, 3, fake, fake, fake, fake, None, 0, None, None]
    a = list(base); a[5] = 3
    assert s(*a) == -3          # K_cap < R
    a = list(base); a[6] = 1
    assert s(*a) == -1          # history mode without c_hist
    a = list(base); a[8] = 4096; a[9] = 3; a[5] = 1 << 20
    assert s(*a) == -2          # more candidates than one CTA sorts
    a = list(base); a[6] = 6
    assert s(*a) == -1          # no such mode
    a = list(base); a[6] = 4; a[7] = float("nan")
    assert s(*a) == -1          # NaN cutoff

    pc = lib.dspark_plan_cycles
    pc.restype = ctypes.c_int
    pc.argtypes = [vp] * 4 + [ctypes.c_int] * 3 + [ctypes.c_float] + [ctypes.c_int] * 4 + [vp] * 5
    # c_seq, n_full, sizes, sps, n_steps, K_cap, mode, conf_min, lag, n_cycles, R, gamma, l, K, stats, status, stream
    base = [fake, None, fake, fake, 5, 1024, 1, 0.0, 2, 100, 512, 5, fake, fake, fake, None, None]
    a = list(base); a[8] = 0
    assert pc(*a) == -1         # lag < 1
    a = list(base); a[4] = 0
    assert pc(*a) == -1         # no capture sizes
    a = list(base); a[5] = 100
    assert pc(*a) == -3         # K_cap < R
    a = list(base); a[9] = 0
    assert pc(*a) == -1         # no cycles

    v = lib.dspark_verify
    v.restype = ctypes.c_int
    v.argtypes = [vp] * 7 + [ctypes.c_uint32, ctypes.c_float] + [ctypes.c_int] * 4 + \
        [vp, vp, vp, vp, ctypes.c_size_t, vp, vp]
    base = [fake] * 7 + [0, 1.0, 4, 5, 1000, 24, fake, fake, None, vp(256 * 64), 1 << 26, None, None]
    a = list(base); a[12] = 3
    assert v(*a) == -1          # max_rows < R
    a = list(base); a[12] = 25
    assert v(*a) == -1          # max_rows > R * (gamma + 1)
    a = list(base); a[3] = None
    assert v(*a) == -1          # sampling without q_logits
    a = list(base); a[17] = 100
    assert v(*a) == -7          # workspace too small

    mk = lib.dspark_verify_markov
    mk.restype = ctypes.c_int
    mk.argtypes = [vp] * 7 + [ctypes.c_int] + [vp] * 3 + [ctypes.c_uint32, ctypes.c_float] + \
        [ctypes.c_int] * 4 + [vp] * 4 + [ctypes.c_size_t, vp, vp]
    # target, cu, y, U, W1, W2, anchor, rank, q_lse, q_tok, seeds, cycle, T, R, gamma, V, max_rows,
    # n_acc, out, p_tok, ws, ws_bytes, status, stream
    base = [fake] * 7 + [64] + [fake] * 3 + [0, 1.0, 4, 5, 1024, 24] + [fake] * 3 + \
        [vp(256 * 64), 1 << 30, None, None]
    a = list(base); a[0] = vp(4096 + 4)
    assert mk(*a) == -2         # target logits not 16-byte aligned (sampling)
    a = list(base); a[3] = vp(4096 + 8)
    assert mk(*a) == -2         # U not 16-byte aligned
    a = list(base); a[7] = 100
    assert mk(*a) == -2         # rank not a multiple of 64


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """The Python binding refuses to import when the shared library is absent."""
    import importlib.util
    import shutil
    pkg = tmp_path / "speculative_decoding_dspark_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "speculative_decoding_dspark_gb300", "binding.py"), pkg / "binding.py")
    spec = importlib.util.spec_from_file_location("binding_copy", pkg / "binding.py")
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)
