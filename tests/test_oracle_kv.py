"""Pins for the oracle's paged-KV reserve and commit/rollback.

Source: DSpark explainer (papers.franksyz.com mainline topic 31) section 11
(verify writes candidates into temporary pages; after the first rejection only
the accepted prefix is promoted and every other candidate's state is released)
and section 15 (leaked or double-freed temporary state among the failure
classes).  The pins: a hand-worked example, conservation of pages (every page
exactly once in a block table or on the free stack) and the page counts the
lengths imply, over a many-cycle run; failure cases leave the state unchanged
or commit nothing.
"""
import numpy as np

from speculative_decoding_dspark_gb300 import inputs


def _ceil(a, b):
    return -(-np.asarray(a, np.int64) // b)


def test_hand_worked_example(orc):
    # P = 4; request 0 holds 5 tokens (pages 2, 3), request 1 holds 8 (pages 0, 1)
    st = orc.KvState([5, 8], [[2, 3, -1], [0, 1, -1]], [10, 11, 12, 13], 4, 4)
    rc, res = orc.kv_reserve(st, [3, 0])  # rows at 5..8 and at 8: one page more each
    assert rc == 0 and list(res) == [1, 1]
    # the top two pages of the stack, in request order
    assert st.block_table.tolist() == [[2, 3, 12], [0, 1, 13]] and st.free_top[0] == 2
    rc = orc.kv_commit(st, [3, 0], [1, 0])  # request 0 keeps 5 + 2 = 7 tokens, request 1 8 + 1 = 9
    assert rc == 0
    assert st.kv_len.tolist() == [7, 9]
    assert st.block_table.tolist() == [[2, 3, -1], [0, 1, 13]]
    assert st.free_top[0] == 3 and st.free_pages[2] == 12


def _check_conservation(st, n_pages):
    held = st.block_table[st.block_table >= 0]
    free = st.free_pages[: st.free_top[0]]
    allp = np.concatenate([held, free])
    assert len(allp) == n_pages and len(np.unique(allp)) == n_pages


def test_many_cycles_conserve_pages(orc):
    w = inputs.workload("confidence_scheduled", R=64)
    kv = inputs.kv_state(w, page_size=16, max_len=4096, spare_pages=5)
    st = orc.KvState(kv["kv_len"], kv["block_table"], kv["free_pages"], kv["free_top"], kv["page_size"])
    g = np.random.default_rng(0)
    P = kv["page_size"]
    for cycle in range(40):
        l = g.integers(0, w["gamma"] + 1, size=w["R"]).astype(np.int32)
        before = st.kv_len.copy()
        rc, res = orc.kv_reserve(st, l)
        assert rc == 0
        np.testing.assert_array_equal(res, _ceil(before + l + 1, P) - _ceil(before, P))
        _check_conservation(st, kv["n_pages"])
        held = (st.block_table >= 0).sum(axis=1)
        np.testing.assert_array_equal(held, _ceil(before + l + 1, P))
        n_acc = (g.random(w["R"]) * (l + 1)).astype(np.int32)
        assert orc.kv_commit(st, l, n_acc) == 0
        np.testing.assert_array_equal(st.kv_len, before + n_acc + 1)
        _check_conservation(st, kv["n_pages"])
        held = (st.block_table >= 0).sum(axis=1)
        np.testing.assert_array_equal(held, _ceil(st.kv_len, P))
        # the held pages are the leading block-table entries
        for r in range(w["R"]):
            assert (st.block_table[r, : held[r]] >= 0).all() and (st.block_table[r, held[r]:] == -1).all()
        # make room for the next cycle: requests that grew past 3000 tokens finish and free everything
        done = st.kv_len > 3000
        for r in np.nonzero(done)[0]:
            pages = st.block_table[r][st.block_table[r] >= 0]
            st.free_pages[st.free_top[0]: st.free_top[0] + len(pages)] = pages
            st.free_top[0] += len(pages)
            st.block_table[r] = -1
            st.kv_len[r] = 0


def test_failures(orc):
    st = orc.KvState([5, 8], [[2, 3, -1], [0, 1, -1]], [10, 11, 12, 13], 1, 4)
    snap = st.copy()
    rc, _ = orc.kv_reserve(st, [3, 0])  # needs two pages, one is free
    assert rc == -3
    for a in ("kv_len", "block_table", "free_pages", "free_top"):
        np.testing.assert_array_equal(getattr(st, a), getattr(snap, a))
    rc, _ = orc.kv_reserve(st, [20, 0])  # past max_blocks
    assert rc == -3
    # a request whose accepted count is out of range commits nothing and frees its temporary pages
    st = orc.KvState([5, 8], [[2, 3, -1], [0, 1, -1]], [10, 11, 12, 13], 4, 4)
    assert orc.kv_reserve(st, [3, 0])[0] == 0
    assert orc.kv_commit(st, [3, 0], [4, 0]) == -6
    assert st.kv_len.tolist() == [5, 9]
    assert st.block_table.tolist() == [[2, 3, -1], [0, 1, 13]] and st.free_top[0] == 3
