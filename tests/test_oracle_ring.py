"""Pins of the oracle's ring slot mapping (window-crossing callers).

"serving prep needs pool-write forms", Proposed Plan: slots equal positions only below the
sliding window; "window-crossing callers need a separate slot mapping". The ring mapping puts
logical page pos // page_size in the request's page (pos // page_size) mod (pages held). These
tests pin it to the linear mapping where no wrap occurs, to its period, and to a dense brute
force over the true K/V history of a request streamed far past its window.
"""
import numpy as np

import brute
from oracle import oracle as O
from paged_sliding_window_qkv_gb300 import workloads as W


def test_ring_without_wrap_equals_linear_mapping():
    rng = np.random.Generator(np.random.PCG64(3))
    b = W.make_batch(rng, [7, 13, 1], [0, 5, 19], 4, spare_pages=4)
    req, pos = O.token_request_and_position(b.qo_indptr, b.start_pos)
    assert all(np.array_equal(x, y) for x, y in zip(
        O.slot_of(req, pos, b.kv_page_indptr, b.page_ids, 4, ring=True),
        O.slot_of(req, pos, b.kv_page_indptr, b.page_ids, 4)))
    q = W.bf16_normal(rng, (b.num_tokens, 4, 8))
    pool = W.bf16_normal(rng, (1, b.num_pages, 2, 2, 4, 8))
    args = (q, pool, 0, b.qo_indptr, b.kv_page_indptr, b.page_ids, b.last_page_len, b.start_pos,
            2, 3, 0.8)
    assert np.array_equal(O.attention(*args, ring=True), O.attention(*args))


def test_ring_slots_repeat_with_the_ring_length_and_never_collide_within_it():
    ps, R = 4, 5
    pages = np.array([9, 2, 7, 0, 4], np.int64)
    indptr = np.array([0, R], np.int64)
    p = np.arange(200, dtype=np.int64)
    pg_, sl = O.slot_of(np.zeros_like(p), p, indptr, pages, ps, ring=True)
    key = pg_ * ps + sl
    assert np.array_equal(key[:-R * ps], key[R * ps:])
    for s in range(0, 200 - R * ps):
        assert len(set(key[s:s + R * ps].tolist())) == R * ps


def test_ring_stream_matches_dense_window_over_the_true_history():
    # one request streamed in steps far past its window through a ring of R pages; every step
    # writes its K/V at ring slots, then attends; the result must equal brute-force attention
    # over the dense history (every position's true K/V) under the same window
    D, hq, hkv, ps, W_ = 8, 2, 1, 4, 9
    steps = [23, 1, 1, 5, 1, 7] + [1] * 100 + [3]
    R = -(-(W_ + max(steps)) // ps)          # the ring holds the window plus a step
    assert R * ps >= W_ + max(steps)
    rng = np.random.Generator(np.random.PCG64(17))
    pages = rng.permutation(R + 6)[:R].astype(np.int32)
    num_pages = R + 6
    pool = np.full((1, num_pages, 2, hkv, ps, D), W.POOL_SENTINEL, np.uint16)
    hist_k, hist_v = [], []
    start = 0
    for n in steps:
        k_new = W.bf16_normal(rng, (n, hkv, D))
        v_new = W.bf16_normal(rng, (n, hkv, D))
        hist_k += [k_new[i] for i in range(n)]
        hist_v += [v_new[i] for i in range(n)]
        qo = np.array([0, n], np.int64)
        indptr = np.array([0, R], np.int64)
        req, pos = O.token_request_and_position(qo, np.array([start]))
        pg_, sl = O.slot_of(req, pos, indptr, pages, ps, ring=True)
        pool[0, pg_, 0, :, sl, :] = k_new
        pool[0, pg_, 1, :, sl, :] = v_new
        q = W.bf16_normal(rng, (n, hq, D))
        got = O.attention(q, pool, 0, qo, indptr, pages, None, np.array([start]), hkv, W_, 0.9,
                          ring=True)
        kk = [[list(O.bf16_to_f64(hist_k[j][h])) for h in range(hkv)] for j in range(start + n)]
        vv = [[list(O.bf16_to_f64(hist_v[j][h])) for h in range(hkv)] for j in range(start + n)]
        qq = [[list(O.bf16_to_f64(q[t, h])) for h in range(hq)] for t in range(n)]
        ref = brute.attention_contiguous(qq, kk, vv, list(range(start, start + n)), W_, 0.9,
                                         hq // hkv)
        assert np.allclose(got, np.array(ref), atol=1e-12, rtol=0), f"step at {start}"
        start += n
    assert start > 4 * R * ps                 # the ring wrapped several times
