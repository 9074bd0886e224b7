"""The DSPARK_DEBUG build (device-side bounds checks of computed indices).

Each case runs in a child process that loads the chosen build through
DSPARK_LIBRARY, so that this process keeps the normal library.  On valid
inputs the debug build's outputs equal the normal build's bit for bit with
status 0; a free-page stack holding a page id outside the pool (a value the
normal build does not check) is reported as DSPARK_ERR_BOUNDS, and the page is
not handed out.  One verify case accepts every draft, so each bonus draw sits at
position gamma, the largest position the checks must let through.
"""
import json
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")

CHILD = textwrap.dedent(r"""
    import json, sys
    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    sys.path.insert(0, TESTS)
    import parity_helpers as H
    from speculative_decoding_dspark_gb300 import binding as B, inputs
    out = {"lib": B.LIB_PATH}
    # tensor-core draft (two request blocks) and both verify calls, sampling and greedy
    for T, name, over in [(0.7, "batched_sampling", dict(R=130, V=17416, gamma=3, rank=64, w_sigma=0.2)),
                          (0.0, "qwen3_8b_greedy", dict(R=9, V=16392, gamma=5, rank=64, w_sigma=0.3))]:
        w, d = H.cycle_inputs(name, **over)
        g = H.gpu_draft(d, T, 3)
        full = inputs.target_full(w, d["U"])
        l = inputs.verify_lengths(w)
        cu = inputs.cu_from_lengths(l)
        tD, cuD = H.dev(inputs.pack_rows(full, l)), H.dev(cu)
        gm = H.gpu_verify_markov(tD, cuD, d, g, 3, T)
        gv = H.gpu_verify(tD, cuD, g["y_dev"], g["q_logits_dev"] if T > 0 else None,
                          g["q_lse_dev"] if T > 0 else None, g["q_tok_dev"] if T > 0 else None,
                          H.dev(d["seeds"]) if T > 0 else None, 3, T)
        out[f"draft_{T}"] = [g["status"], g["y"].tolist(), g["q_lse"].tolist(), g["q_tok"].tolist()]
        out[f"markov_{T}"] = [gm["status"], gm["n_acc"].tolist(), gm["out_tokens"].tolist(), gm["p_tok"].tolist()]
        out[f"verify_{T}"] = [gv["status"], gv["n_acc"].tolist(), gv["out_tokens"].tolist(), gv["p_tok"].tolist()]
    # stored-logits verify where every request accepts all gamma drafts, so the
    # bonus draw sits at position gamma (the last row of each request)
    R, V, gamma = 8, 1032, 3
    rng = np.random.default_rng(5)
    y = rng.integers(0, V, (R, gamma)).astype(np.int32)
    ql = rng.standard_normal((R, gamma, V)).astype(np.float32)
    m = ql.max(axis=2, keepdims=True)
    q_lse = (m[..., 0] + np.log(np.exp(ql - m).sum(axis=2))).astype(np.float32)
    q_tok = np.exp(np.take_along_axis(ql, y[..., None], 2)[..., 0] - q_lse).astype(np.float32)
    target = np.zeros((R * (gamma + 1), V), np.float32)
    for r in range(R):
        for j in range(gamma):
            target[r * (gamma + 1) + j, y[r, j]] = 60.0  # p(y) = 1: accepted
        target[r * (gamma + 1) + gamma] = rng.standard_normal(V).astype(np.float32)
    cu = inputs.cu_from_lengths(np.full(R, gamma, np.int32))
    seeds = inputs.request_seeds(0x5EED0300, R)
    gv = H.gpu_verify(target, cu, y, ql, q_lse, q_tok, seeds, 0, 1.0)
    out["verify_bonus"] = [gv["status"], gv["n_acc"].tolist(), gv["out_tokens"].tolist(), gv["p_tok"].tolist()]
    # paged KV: a valid reserve and commit, then a stack with a page id outside the pool
    R, P, pool = 4, 16, 64
    kv_len = np.array([5, 16, 0, 31], np.int32)
    lv = np.array([3, 5, 7, 1], np.int32)
    n_acc = np.array([1, 5, 0, 0], np.int32)
    max_blocks = 8
    for bad in (False, True):
        bt = np.full((R, max_blocks), -1, np.int32)
        free = list(range(pool))
        for r in range(R):
            for b in range((int(kv_len[r]) + P - 1) // P):
                bt[r, b] = free.pop()
        if bad:
            free[-1] = pool + 5  # the next page handed out is outside the pool
        stack = np.array(free + [0] * (pool - len(free)), np.int32)
        kv_d, l_d, na_d = H.dev(kv_len), H.dev(lv), H.dev(n_acc)
        bt_d, st_d = H.dev(bt), H.dev(stack)
        top = torch.tensor([len(free)], dtype=torch.int32, device="cuda")
        res = torch.zeros(R, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        B.dspark_kv_reserve(kv_d, l_d, P, bt_d, st_d, top, res, status)
        r1 = int(status.item())
        if not bad:
            B.dspark_kv_commit(kv_d, l_d, na_d, P, bt_d, st_d, top, status)
        torch.cuda.synchronize()
        out[f"kv_{bad}"] = [r1, int(status.item()), H.host(bt_d).tolist(), H.host(kv_d).tolist(), int(top.item())]
    print("RESULT " + json.dumps(out))
""")


def _run(lib):
    env = dict(os.environ)
    if lib:
        env["DSPARK_LIBRARY"] = lib
    else:
        env.pop("DSPARK_LIBRARY", None)
    code = f"ROOT = {ROOT!r}\nTESTS = {TESTS!r}\n" + CHILD
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    line = [x for x in r.stdout.splitlines() if x.startswith("RESULT ")][-1]
    return json.loads(line[len("RESULT "):])


def test_debug_build_matches_and_checks():
    from speculative_decoding_dspark_gb300 import build
    build.build()
    dbg = build.build(debug=True)
    normal = _run(None)
    debug = _run(dbg)
    assert debug["lib"].endswith("libdspark_debug.so") and normal["lib"].endswith("libdspark.so")
    for key in normal:
        if key in ("lib", "kv_True"):
            continue
        assert debug[key] == normal[key], key
        if key.startswith(("draft", "markov", "verify")):
            assert normal[key][0] == 0, (key, normal[key][0])
    assert normal["verify_bonus"][1] == [3] * 8  # every request took the bonus draw at position gamma
    assert normal["kv_False"][:2] == [0, 0]
    # the bad page id: handed out silently by the normal build, refused by the debug one
    B_ERR_BOUNDS = -8
    assert normal["kv_True"][0] == 0
    assert debug["kv_True"][0] == B_ERR_BOUNDS
    bad_page = 64 + 5
    assert bad_page in np.array(normal["kv_True"][2]).ravel().tolist()
    assert bad_page not in np.array(debug["kv_True"][2]).ravel().tolist()
