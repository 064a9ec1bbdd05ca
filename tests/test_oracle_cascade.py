"""Pins of the oracle's key segments, log-sum-exp output and state merging (cascade
attention for requests that share a key prefix).

The pages leave this variant open: they define the masked softmax attention over a request's
keys ("Rust wrapper for the hd256 windowed paged prefill", Description). The normaliser of
that softmax, lse = log sum_j exp(s_j), and the exact merge of two disjoint key sets follow
from the definition. These tests pin the oracle to a pure-loop brute force, to closed forms,
and to the identity that attention over a request's keys equals the merge of attention over
its shared prefix and over its own suffix.
"""
import math

import numpy as np
import pytest

import brute
from oracle import oracle as O
from paged_sliding_window_qkv_gb300 import workloads as W


def fill_pool(ci: W.CascadeInputs, full=True, segments=True):
    """Pool bits holding the cascade's three layouts, written slot by slot with the brute
    page walk (position i of a key run is the i-th slot visited)."""
    f, ps = ci.full, ci.full.page_size
    pool = np.full((1, f.num_pages, 2, ci.num_kv_heads, ps, ci.head_dim), W.POOL_SENTINEL,
                   np.uint16)

    def put(pages, rows_k, rows_v):
        for i, (pg, sl) in enumerate(brute.slots_for_request(pages, len(rows_k), ps)):
            pool[0, pg, 0, :, sl, :] = rows_k[i]
            pool[0, pg, 1, :, sl, :] = rows_v[i]

    P = ci.prefix_len
    for r in range(f.num_req):
        if full:
            put(f.page_ids[f.kv_page_indptr[r]:f.kv_page_indptr[r + 1]], ci.hist_k[r], ci.hist_v[r])
        if segments:
            s = ci.suffix
            put(s.page_ids[s.kv_page_indptr[r]:s.kv_page_indptr[r + 1]], ci.hist_k[r][P:],
                ci.hist_v[r][P:])
    if segments:
        p = ci.prefix
        put(p.page_ids[p.kv_page_indptr[0]:p.kv_page_indptr[1]], ci.hist_k[0][:P], ci.hist_v[0][:P])
    return pool


def run(ci, pool, b, kv_start, hkv, window, scale):
    return O.attention(ci.q, pool, 0, b.qo_indptr, b.kv_page_indptr, b.page_ids,
                       b.last_page_len, b.start_pos, hkv, window, scale, kv_start=kv_start,
                       return_lse=True)


@pytest.mark.parametrize("prefix_len,suffix_lens,steps,window,ps", [
    (37, [5, 20, 1], [5, 3, 1], -1, 4),
    (16, [9, 33], [9, 17], 11, 8),      # the window reaches back across the prefix boundary
    (50, [7, 2], [1, 1], 3, 4),         # decode rows whose window misses the whole prefix
])
def test_prefix_and_suffix_merge_to_the_single_pass(prefix_len, suffix_lens, steps, window, ps):
    rng = np.random.Generator(np.random.PCG64(prefix_len + ps))
    hq, hkv, D = 4, 2, 8
    ci = W.make_cascade(rng, prefix_len, suffix_lens, steps, ps, hq, hkv, D)
    pool = fill_pool(ci)
    R = ci.full.num_req
    o_full, l_full = run(ci, pool, ci.full, None, hkv, window, 0.7)
    o_pre, l_pre = run(ci, pool, ci.prefix, np.zeros(R, np.int64), hkv, window, 0.7)
    o_suf, l_suf = run(ci, pool, ci.suffix, np.full(R, prefix_len, np.int64), hkv, window, 0.7)
    o_m, l_m = O.merge_states(o_pre, l_pre, o_suf, l_suf)
    assert np.allclose(o_m, o_full, atol=1e-12, rtol=0)
    assert np.allclose(l_m, l_full, atol=1e-12, rtol=0)
    if window >= 0 and min(steps) == 1:
        assert np.isneginf(l_pre).any()        # the neutral state did occur


def test_lse_matches_brute_force():
    rng = np.random.Generator(np.random.PCG64(99))
    hq, hkv, D, ps, P = 4, 2, 6, 4, 9
    ci = W.make_cascade(rng, P, [6, 11], [6, 4], ps, hq, hkv, D)
    pool = fill_pool(ci)
    _, pos = O.token_request_and_position(ci.full.qo_indptr, ci.full.start_pos)
    req, _ = O.token_request_and_position(ci.full.qo_indptr, ci.full.start_pos)
    for window in (-1, 5):
        _, l_full = run(ci, pool, ci.full, None, hkv, window, 0.8)
        _, l_suf = run(ci, pool, ci.suffix, np.full(2, P, np.int64), hkv, window, 0.8)
        for t in range(len(pos)):
            r = int(req[t])
            qq = [[list(O.bf16_to_f64(ci.q[t, h])) for h in range(hq)]]
            kk = [[list(O.bf16_to_f64(ci.hist_k[r][j, g])) for g in range(hkv)]
                  for j in range(len(ci.hist_k[r]))]
            ref = brute.lse_contiguous(qq, kk, [int(pos[t])], list(range(len(kk))), window, 0.8,
                                       hq // hkv)[0]
            assert np.allclose(l_full[t], ref, atol=1e-12, rtol=0)
            ref_s = brute.lse_contiguous(qq, kk[P:], [int(pos[t])], list(range(P, len(kk))),
                                         window, 0.8, hq // hkv)[0]
            assert np.allclose(l_suf[t], ref_s, atol=1e-12, rtol=0)


def test_lse_closed_forms():
    rng = np.random.Generator(np.random.PCG64(5))
    hq, hkv, D, ps = 2, 1, 8, 4
    ci = W.make_cascade(rng, 8, [12], [3], ps, hq, hkv, D)
    # equal keys: every visible score is the same s, so lse = s + log(visible count)
    for r in range(1):
        ci.hist_k[r][:] = ci.hist_k[r][0]
    pool = fill_pool(ci)
    _, pos = O.token_request_and_position(ci.full.qo_indptr, ci.full.start_pos)
    for window in (-1, 0, 6):
        _, lse = run(ci, pool, ci.full, None, hkv, window, 0.5)
        for t in range(3):
            n = pos[t] + 1 if window < 0 else min(pos[t] + 1, window + 1)
            for h in range(hq):
                s = 0.5 * float(O.bf16_to_f64(ci.q[t, h]) @ O.bf16_to_f64(ci.hist_k[0][0, 0]))
                assert math.isclose(lse[t, h], s + math.log(n), abs_tol=1e-12)
    # a segment wholly after the queries: nothing visible, the neutral state (0, -inf)
    o, lse = run(ci, pool, ci.suffix, np.array([10 ** 6], np.int64), hkv, -1, 0.5)
    assert (o == 0).all() and np.isneginf(lse).all()


def test_merge_states_algebra():
    rng = np.random.default_rng(3)
    st = [(rng.standard_normal((5, 3)), rng.standard_normal(5) * 4) for _ in range(3)]
    (oa, la), (ob, lb), (oc, lc) = st
    zero = (np.zeros((5, 3)), np.full(5, -np.inf))
    o, l = O.merge_states(oa, la, *zero)
    assert np.allclose(o, oa, atol=1e-15) and np.allclose(l, la, atol=1e-15)
    o1, l1 = O.merge_states(oa, la, ob, lb)
    o2, l2 = O.merge_states(ob, lb, oa, la)
    assert np.allclose(o1, o2, atol=1e-14) and np.allclose(l1, l2, atol=1e-14)
    o3, l3 = O.merge_states(*O.merge_states(oa, la, ob, lb), oc, lc)
    o4, l4 = O.merge_states(oa, la, *O.merge_states(ob, lb, oc, lc))
    assert np.allclose(o3, o4, atol=1e-13) and np.allclose(l3, l4, atol=1e-13)
    # the weights are softmax(lse): lse of the merge is log(e^la + e^lb)
    assert np.allclose(l1, np.logaddexp(la, lb), atol=1e-14)
    o, l = O.merge_states(*zero, *zero)
    assert (o == 0).all() and np.isneginf(l).all()


def test_segment_slots_follow_the_page_walk_from_the_segment_start():
    # position kv_start + i lives in the i-th slot of the request's pages
    rng = np.random.Generator(np.random.PCG64(23))
    ps = 4
    ci = W.make_cascade(rng, 13, [9, 22], [9, 5], ps, 2, 1, 8)
    s = ci.suffix
    req, pos = O.token_request_and_position(s.qo_indptr, s.start_pos)
    page, slot = O.slot_of(req, pos, s.kv_page_indptr, s.page_ids, ps, kv_start=np.full(2, 13))
    for t in range(len(pos)):
        r = int(req[t])
        pages = s.page_ids[s.kv_page_indptr[r]:s.kv_page_indptr[r + 1]]
        walk = brute.slots_for_request(pages, int(pos[t]) - 13 + 1, ps)
        assert (int(page[t]), int(slot[t])) == walk[-1]
    # a segment starting at 0 is the linear mapping
    f = ci.full
    req, pos = O.token_request_and_position(f.qo_indptr, f.start_pos)
    a = O.slot_of(req, pos, f.kv_page_indptr, f.page_ids, ps, kv_start=np.zeros(2, np.int64))
    b = O.slot_of(req, pos, f.kv_page_indptr, f.page_ids, ps)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
