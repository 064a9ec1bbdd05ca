"""Host-side page accounting for two-family paged KV serving (include/pg_kv.h), on CPU.

What is checked follows "feat(gemma4): paged KV serving across both attention families",
Description and Verification: admission atomic across both pools, the page count as the exact
frontier account, a forced partial failure leaving both pools at their pre-request occupancy,
checks before any state change, page ids valid only against the issuing server, and failing
closed at the sliding window; and its review finding "Commit KV frontiers only after a
successful step": admission reserves, the frontier moves only on commit, and an aborted step
leaves both pools and the frontier as they were before admission.
"""
import numpy as np
import pytest

from paged_sliding_window_qkv_gb300 import pg

L, G = pg.PG_KV_LOCAL, pg.PG_KV_GLOBAL


def server(pages_local=64, pages_global=64, ps=16, window=1023, fail_closed=1, rope_rows=1 << 20):
    rc, s = pg.pg_kv_server_create(pages_local, pages_global, ps, window, fail_closed, rope_rows)
    assert rc == pg.PG_KV_OK
    return s


def free(s):
    return pg.pg_kv_free_pages(s, L)[1], pg.pg_kv_free_pages(s, G)[1]


def state(s, rid):
    rc, f, nl, ng = pg.pg_kv_request_info(s, rid)
    assert rc == pg.PG_KV_OK
    return f, nl, ng, tuple(pg.pg_kv_request_pages(s, rid, L)[1]), tuple(pg.pg_kv_request_pages(s, rid, G)[1])


def open_req(s):
    rc, rid = pg.pg_kv_request_open(s)
    assert rc == pg.PG_KV_OK and rid > 0
    return rid


def step(s, rid, n):
    """Admit a step and commit it (the step's launches succeeded); returns the admit status."""
    rc = pg.pg_kv_admit_step(s, rid, n)
    if rc == pg.PG_KV_OK:
        assert pg.pg_kv_commit_step(s, rid) == pg.PG_KV_OK
    return rc


def test_page_count_is_the_exact_frontier_account():
    s = server(ps=16)
    rid = open_req(s)
    frontier = 0
    for n in [1, 15, 1, 16, 17, 3, 64, 1]:
        assert step(s, rid, n) == pg.PG_KV_OK
        frontier += n
        f, nl, ng, _, _ = state(s, rid)
        assert f == frontier
        assert nl == ng == -(-frontier // 16)        # ceil(frontier / page_size) in both pools
    assert free(s) == (64 - nl, 64 - ng)
    pg.pg_kv_server_destroy(s)


def test_forced_partial_failure_leaves_both_pools_untouched():
    # the pages' verification: a refused second family must drop the first family's grant
    for refused in (G, L):
        s = server()
        rid = open_req(s)
        assert step(s, rid, 20) == pg.PG_KV_OK
        before_free, before_state = free(s), state(s, rid)
        assert pg.pg_kv_inject_refusal(s, refused, 1) == pg.PG_KV_OK
        assert step(s, rid, 30) == pg.PG_KV_ERR_NO_PAGES
        assert free(s) == before_free
        assert state(s, rid) == before_state
        # the refusal was one-shot: the same step is admitted next
        assert step(s, rid, 30) == pg.PG_KV_OK
        assert state(s, rid)[0] == 50
        pg.pg_kv_server_destroy(s)


def test_exhausted_family_refuses_without_stranding_the_other():
    s = server(pages_local=64, pages_global=3, ps=16)
    rid = open_req(s)
    assert step(s, rid, 48) == pg.PG_KV_OK       # 3 pages each
    before = free(s), state(s, rid)
    assert step(s, rid, 1) == pg.PG_KV_ERR_NO_PAGES   # global has no 4th page
    assert (free(s), state(s, rid)) == before
    assert free(s) == (61, 0)
    pg.pg_kv_server_destroy(s)


def test_window_fails_closed_and_rope_bound():
    s = server(window=31, fail_closed=1, rope_rows=40)
    rid = open_req(s)
    assert step(s, rid, 32) == pg.PG_KV_OK        # window_left + 1 positions
    before = free(s), state(s, rid)
    assert step(s, rid, 1) == pg.PG_KV_ERR_WINDOW
    assert (free(s), state(s, rid)) == before
    pg.pg_kv_server_destroy(s)
    s = server(window=31, fail_closed=0, rope_rows=40)
    rid = open_req(s)
    assert step(s, rid, 40) == pg.PG_KV_OK        # positions 0..39 < rope_rows
    assert step(s, rid, 1) == pg.PG_KV_ERR_ROPE
    assert state(s, rid)[0] == 40
    pg.pg_kv_server_destroy(s)


def test_foreign_and_closed_requests_are_refused():
    s1, s2 = server(), server()
    r1 = open_req(s1)
    assert step(s2, r1 + 1000, 1) == pg.PG_KV_ERR_FOREIGN
    assert step(s1, r1, 17) == pg.PG_KV_OK
    assert free(s1) == (62, 62)
    assert pg.pg_kv_request_close(s1, r1) == pg.PG_KV_OK
    assert free(s1) == (64, 64)                                   # pages returned to both pools
    assert step(s1, r1, 1) == pg.PG_KV_ERR_FOREIGN
    assert pg.pg_kv_request_close(s1, r1) == pg.PG_KV_ERR_FOREIGN
    assert step(s1, 0, 1) == pg.PG_KV_ERR_FOREIGN
    for s in (s1, s2):
        pg.pg_kv_server_destroy(s)


def test_bad_arguments():
    assert pg.pg_kv_server_create(4, 4, 0, 10, 1, 100)[0] == pg.PG_KV_ERR_ARG
    assert pg.pg_kv_server_create(4, 4, 16, -1, 1, 100)[0] == pg.PG_KV_ERR_ARG
    s = server()
    rid = open_req(s)
    assert step(s, rid, 0) == pg.PG_KV_ERR_ARG
    assert pg.pg_kv_free_pages(s, 2)[0] == pg.PG_KV_ERR_ARG
    assert step(s, rid, 40) == pg.PG_KV_OK
    assert pg.pg_kv_request_pages(s, rid, L, cap=2)[0] == pg.PG_KV_ERR_CAPACITY
    pg.pg_kv_server_destroy(s)


def test_batch_plan_inputs_follow_the_plan_contract():
    ps = 16
    s = server(ps=ps)
    rids = [open_req(s) for _ in range(3)]
    lens = [5, 40, 16]
    for r, n in zip(rids, lens):
        assert step(s, r, n) == pg.PG_KV_OK
    # without a pending step there is nothing to plan
    assert pg.pg_kv_batch_plan_inputs(s, L, rids, [1, 1, 1])[0] == pg.PG_KV_ERR_PENDING
    # a decode step of one token each is admitted (pending), then the local family's inputs
    for r in rids:
        assert pg.pg_kv_admit_step(s, r, 1) == pg.PG_KV_OK
    rc, indptr, pages, last, start = pg.pg_kv_batch_plan_inputs(s, L, rids, [1, 1, 1])
    assert rc == pg.PG_KV_OK
    kv_len = (np.diff(indptr) - 1) * ps + last
    assert (kv_len == np.array(lens) + 1).all()                    # coverage: kv_len = start + qo_len
    assert (start == np.array(lens)).all()                         # start = the committed frontier
    assert ((1 <= last) & (last <= ps)).all()
    assert len(set(pages.tolist())) == len(pages)                  # no page held twice
    for i, r in enumerate(rids):
        assert tuple(pages[indptr[i]:indptr[i + 1]]) == tuple(pg.pg_kv_request_pages(s, r, L)[1])
    # a step count other than the pending one has no plan
    assert pg.pg_kv_batch_plan_inputs(s, L, rids, [1, 1, 100])[0] == pg.PG_KV_ERR_ARG
    pg.pg_kv_server_destroy(s)


@pytest.mark.parametrize("ring", [False, True], ids=["linear", "ring"])
def test_random_traffic_keeps_the_books(ring):
    rng = np.random.default_rng(11)
    total = (48, 24)
    ring_pages = -(-(30 + 19) // 8)  # window 30, steps of at most 19 tokens
    if ring:
        rc, s = pg.pg_kv_server_create_ring(total[0], total[1], 8, 30, 19, 1 << 20)
        assert rc == pg.PG_KV_OK
    else:
        s = server(pages_local=total[0], pages_global=total[1], ps=8, window=1 << 20)
    live = {}
    for _ in range(600):
        op = rng.integers(4)
        if op == 0 or not live:
            live[open_req(s)] = 0
        elif op == 1:
            r = int(rng.choice(list(live)))
            assert pg.pg_kv_request_close(s, r) == pg.PG_KV_OK
            del live[r]
        else:
            r = int(rng.choice(list(live)))
            if rng.random() < 0.1:
                pg.pg_kv_inject_refusal(s, int(rng.integers(2)), 1)
            before = free(s), state(s, r)
            rc = pg.pg_kv_admit_step(s, r, int(rng.integers(1, 20)))
            if rc != pg.PG_KV_OK:
                assert rc == pg.PG_KV_ERR_NO_PAGES
                assert (free(s), state(s, r)) == before
            elif rng.random() < 0.3:       # the step failed after admission
                assert pg.pg_kv_abort_step(s, r) == pg.PG_KV_OK
                assert (free(s), state(s, r)) == before
            else:
                assert pg.pg_kv_commit_step(s, r) == pg.PG_KV_OK
            pg.pg_kv_inject_refusal(s, 0, 0)
            pg.pg_kv_inject_refusal(s, 1, 0)
        # conservation and exclusivity in both pools
        for fam in (L, G):
            held = [p for r in live for p in pg.pg_kv_request_pages(s, r, fam)[1]]
            assert len(held) == len(set(held))
            assert len(held) + pg.pg_kv_free_pages(s, fam)[1] == total[fam]
            assert all(0 <= p < total[fam] for p in held)
        for r in live:
            f, nl, ng, _, _ = state(s, r)
            assert ng == -(-f // 8)
            assert nl == (min(ng, ring_pages) if ring else ng)
    pg.pg_kv_server_destroy(s)


def test_ring_server_caps_the_local_family_at_its_ring():
    ps, window, max_step = 16, 100, 64
    ring = -(-(window + max_step) // ps)                 # 11 pages
    rc, s = pg.pg_kv_server_create_ring(40, 64, ps, window, max_step, 1 << 20)
    assert rc == pg.PG_KV_OK
    rid = open_req(s)
    frontier = 0
    for n in [37, 20, 64, 1, 50, 64, 1, 64, 3, 64, 64]:
        assert step(s, rid, n) == pg.PG_KV_OK
        frontier += n
        f, nl, ng, local, _ = state(s, rid)
        assert f == frontier
        assert nl == min(-(-frontier // ps), ring)      # grows, then stays at the ring
        assert ng == -(-frontier // ps)                  # the global family keeps growing
        assert free(s) == (40 - nl, 64 - ng)
    assert frontier > 2 * ring * ps                      # wrapped more than once
    # a step longer than the ring allows beside the window is refused, nothing changed
    before = free(s), state(s, rid)
    assert step(s, rid, max_step + 1) == pg.PG_KV_ERR_WINDOW
    assert (free(s), state(s, rid)) == before
    # plan inputs of a pending 3-token step: the ring's pages in ring order, start = frontier
    assert pg.pg_kv_admit_step(s, rid, 3) == pg.PG_KV_OK
    rc, indptr, pages, last, start = pg.pg_kv_batch_plan_inputs(s, L, [rid], [3])
    assert rc == pg.PG_KV_OK
    assert tuple(pages) == state(s, rid)[3] and len(pages) == ring
    assert start[0] == frontier and last[0] == (frontier + 3 - 1) % ps + 1
    assert pg.pg_kv_request_close(s, rid) == pg.PG_KV_OK
    assert free(s) == (40, 64)
    pg.pg_kv_server_destroy(s)


def test_ring_server_rejects_bad_arguments():
    assert pg.pg_kv_server_create_ring(8, 8, 16, 100, 0, 1 << 20)[0] == pg.PG_KV_ERR_ARG
    assert pg.pg_kv_server_create_ring(8, 8, 0, 100, 8, 1 << 20)[0] == pg.PG_KV_ERR_ARG
    assert pg.pg_kv_server_create_ring(8, 8, 16, -1, 8, 1 << 20)[0] == pg.PG_KV_ERR_ARG


def test_frontier_moves_only_on_commit():
    ps = 16
    s = server(ps=ps)
    rid = open_req(s)
    assert step(s, rid, 20) == pg.PG_KV_OK
    assert pg.pg_kv_admit_step(s, rid, 30) == pg.PG_KV_OK
    f, nl, ng, _, _ = state(s, rid)
    assert f == 20 and nl == ng == -(-50 // ps)          # pages held, frontier not moved
    assert pg.pg_kv_request_pending(s, rid) == (pg.PG_KV_OK, 30)
    # one pending step at a time
    before = free(s), state(s, rid)
    assert pg.pg_kv_admit_step(s, rid, 1) == pg.PG_KV_ERR_PENDING
    assert (free(s), state(s, rid)) == before
    assert pg.pg_kv_commit_step(s, rid) == pg.PG_KV_OK
    assert state(s, rid)[0] == 50
    assert pg.pg_kv_request_pending(s, rid) == (pg.PG_KV_OK, 0)
    # nothing pending: commit and abort are refused and change nothing
    before = free(s), state(s, rid)
    assert pg.pg_kv_commit_step(s, rid) == pg.PG_KV_ERR_PENDING
    assert pg.pg_kv_abort_step(s, rid) == pg.PG_KV_ERR_PENDING
    assert (free(s), state(s, rid)) == before
    assert pg.pg_kv_commit_step(s, rid + 99) == pg.PG_KV_ERR_FOREIGN
    assert pg.pg_kv_abort_step(s, rid + 99) == pg.PG_KV_ERR_FOREIGN
    pg.pg_kv_server_destroy(s)


@pytest.mark.parametrize("ring", [False, True], ids=["linear", "ring"])
def test_aborted_step_restores_both_pools_and_the_frontier(ring):
    # the review finding: a step that fails after admission (plan, copy, launch or tail) must not
    # leave the frontier claiming its tokens, else a retry's start_pos skips them
    ps = 16
    if ring:
        rc, s = pg.pg_kv_server_create_ring(40, 64, ps, 100, 64, 1 << 20)
        assert rc == pg.PG_KV_OK
        steps = [64, 64, 64, 40]                          # past the 11-page ring
    else:
        s = server(ps=ps)
        steps = [37, 20]
    rid = open_req(s)
    for n in steps:
        assert step(s, rid, n) == pg.PG_KV_OK
    frontier = sum(steps)
    before = free(s), state(s, rid)
    rc0, ind0, pages0, last0, start0 = (None,) * 5
    for attempt in range(3):
        assert pg.pg_kv_admit_step(s, rid, 33) == pg.PG_KV_OK
        rc, ind, pages, last, start = pg.pg_kv_batch_plan_inputs(s, L, [rid], [33])
        assert rc == pg.PG_KV_OK and start[0] == frontier
        if attempt == 0:
            ind0, pages0, last0 = ind, pages, last
        else:                                             # a retry plans the very same span
            assert (ind == ind0).all() and (pages == pages0).all() and (last == last0).all()
        if attempt < 2:
            assert pg.pg_kv_abort_step(s, rid) == pg.PG_KV_OK
            assert (free(s), state(s, rid)) == before
    assert pg.pg_kv_commit_step(s, rid) == pg.PG_KV_OK
    assert state(s, rid)[0] == frontier + 33
    # closing a request with a pending step returns every page
    assert pg.pg_kv_admit_step(s, rid, 5) == pg.PG_KV_OK
    assert pg.pg_kv_request_close(s, rid) == pg.PG_KV_OK
    assert free(s) == ((40, 64) if ring else (64, 64))
    pg.pg_kv_server_destroy(s)
