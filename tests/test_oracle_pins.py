"""Pins for the fp64 oracle: closed forms, invariants and brute force (CPU only).

Each test fixes something the pages or plain mathematics determine, chosen so
that a plausible slip in the oracle (a dropped term, a wrong sign or index, the
wrong rotary pairing, a transposed operand, an off-by-one window) fails one of
them.
"""
import math

import numpy as np
import pytest
import torch

import brute
from oracle import oracle as O
from paged_sliding_window_qkv_gb300 import workloads as W


def rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


# ---------------------------------------------------------------------------- bf16
def test_bf16_rounding_known_patterns():
    cases = {
        1.0: 0x3F80,
        -2.0: 0xC000,
        1.0 + 2 ** -8: 0x3F80,          # halfway, ties to even (down)
        1.0 + 3 * 2 ** -8: 0x3F82,      # halfway, ties to even (up)
        1.0 + 2 ** -8 + 2 ** -30: 0x3F81,  # just above halfway
        0.0: 0x0000,
        2.0 ** -133: 0x0001,            # smallest subnormal
        3.0e38: 0x7F62,
        1e39: 0x7F80,                   # overflow to inf
    }
    for x, bits in cases.items():
        assert int(O.f64_to_bf16(np.array([x]))[0]) == bits, x


def test_bf16_rounding_matches_library_on_float32_values():
    x = rng(1).standard_normal(100000).astype(np.float32) * np.float32(3.0)
    x[:1000] *= np.float32(1e-38)   # subnormal range
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = O.f64_to_bf16(x.astype(np.float64))
    assert np.array_equal(ref, got)
    back = O.bf16_to_f64(got)
    assert np.array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


# ---------------------------------------------------------------------------- RMSNorm
def test_inv_rms_closed_form_d4():
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    assert O.inv_rms(x, 0.0)[0, 0] == pytest.approx(1.0 / math.sqrt(7.5), rel=1e-15)
    assert O.inv_rms(x, 0.5)[0, 0] == pytest.approx(1.0 / math.sqrt(8.0), rel=1e-15)


def test_weightless_norm_has_unit_rms_and_is_scale_invariant():
    x = rng(2).standard_normal((50, 256))
    y = x * O.inv_rms(x, 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-14)
    y2 = (7.25 * x) * O.inv_rms(7.25 * x, 0.0)
    assert np.allclose(y, y2, atol=1e-14)


# ---------------------------------------------------------------------------- RoPE
def test_rope_d2_is_textbook_rotation():
    # D=2: theta^0 = 1, so position p rotates (x0, x1) by p radians.
    for p in [0, 1, 2, 5, 100]:
        c, s = O.rope_cos_sin(np.array([p]), 2, 10000.0)
        y = O.rope_half_split(np.array([[0.3, -1.7]]), c, s)[0]
        rot = np.array([[math.cos(p), -math.sin(p)], [math.sin(p), math.cos(p)]])
        assert np.allclose(y, rot @ np.array([0.3, -1.7]), atol=1e-15)


def test_rope_half_split_pairing_sign_and_frequency_d4():
    # D=4, theta=100: pair (0,2) turns at 1 rad/position, pair (1,3) at 100^-0.5 = 0.1.
    p = 3
    c, s = O.rope_cos_sin(np.array([p]), 4, 100.0)
    e0 = O.rope_half_split(np.array([[1.0, 0, 0, 0]]), c, s)[0]
    assert np.allclose(e0, [math.cos(3), 0, math.sin(3), 0], atol=1e-15)
    e1 = O.rope_half_split(np.array([[0, 1.0, 0, 0]]), c, s)[0]
    assert np.allclose(e1, [0, math.cos(0.3), 0, math.sin(0.3)], atol=1e-15)
    e2 = O.rope_half_split(np.array([[0, 0, 1.0, 0]]), c, s)[0]
    assert np.allclose(e2, [-math.sin(3), 0, math.cos(3), 0], atol=1e-15)


def test_rope_identity_at_zero_norm_preserving_and_relative():
    r = rng(3)
    D = 256
    x = r.standard_normal((1, D))
    c0, s0 = O.rope_cos_sin(np.array([0]), D, 1e4)
    assert np.array_equal(O.rope_half_split(x, c0, s0), x)
    c, s = O.rope_cos_sin(np.array([777]), D, 1e4)
    y = O.rope_half_split(x, c, s)
    h = D // 2
    assert np.allclose(x[0, :h] ** 2 + x[0, h:] ** 2, y[0, :h] ** 2 + y[0, h:] ** 2, atol=1e-12)
    q, k = r.standard_normal((1, D)), r.standard_normal((1, D))
    dots = []
    for m, n in [(10, 3), (107, 100), (5007, 5000)]:
        cm, sm = O.rope_cos_sin(np.array([m]), D, 1e4)
        cn, sn = O.rope_cos_sin(np.array([n]), D, 1e4)
        dots.append(float((O.rope_half_split(q, cm, sm) @ O.rope_half_split(k, cn, sn).T)[0, 0]))
    assert np.allclose(dots, dots[0], rtol=1e-9, atol=1e-9)


# ---------------------------------------------------------------------------- prep
def _tiny_prep_case(D, hq, hkv, T, seed):
    r = rng(seed)
    q = r.standard_normal((T, hq, D))
    k = r.standard_normal((T, hkv, D))
    v = r.standard_normal((T, hkv, D))
    wq = 1 + 0.1 * r.standard_normal(D)
    wk = 1 + 0.1 * r.standard_normal(D)
    pos = np.arange(5, 5 + T)
    return q, k, v, wq, wk, pos


@pytest.mark.parametrize("D", [4, 8])
def test_prep_hd256_form_matches_brute(D):
    q, k, v, wq, wk, pos = _tiny_prep_case(D, 4, 2, 6, 10 + D)
    eps, theta = 1e-6, 50.0
    qo, ko, vo = O.prep_hd256(q, k, v, wq, wk, eps, pos, theta)
    for t in range(6):
        for h in range(4):
            yb = brute.rope_row(brute.rmsnorm_row(list(q[t, h]), list(wq), eps)[0], pos[t], theta)
            assert np.allclose(qo[t, h], yb, atol=1e-13)
        for h in range(2):
            kb = brute.rope_row(brute.rmsnorm_row(list(k[t, h]), list(wk), eps)[0], pos[t], theta)
            assert np.allclose(ko[t, h], kb, atol=1e-13)
            vb = brute.rmsnorm_row(list(v[t, h]), None, eps)[0]
            assert np.allclose(vo[t, h], vb, atol=1e-13)


def test_prep_hd512_form_v_is_weightless_norm_of_raw_k():
    q, k, _, wq, wk, pos = _tiny_prep_case(8, 4, 1, 5, 21)
    eps, theta = 1e-6, 1e6
    qo, ko, vo = O.prep_hd512(q, k, wq, wk, eps, pos, theta)
    for t in range(5):
        vb, r = brute.rmsnorm_row(list(k[t, 0]), None, eps)
        assert np.allclose(vo[t, 0], vb, atol=1e-14)
        kb = brute.rope_row([k[t, 0, i] * r * wk[i] for i in range(8)], pos[t], theta)
        assert np.allclose(ko[t, 0], kb, atol=1e-13)
    # K = V bit for bit at position 0 with unit weight (rotation is the identity there).
    _, k0, v0 = O.prep_hd512(q[:1], k[:1], wq, np.ones(8), eps, np.array([0]), theta)
    assert np.array_equal(k0, v0)


def test_prep_v_is_never_rotated():
    q, k, v, wq, wk, _ = _tiny_prep_case(8, 2, 2, 1, 31)
    a = O.prep_hd256(q, k, v, wq, wk, 1e-6, np.array([0]), 1e4)[2]
    b = O.prep_hd256(q, k, v, wq, wk, 1e-6, np.array([12345]), 1e4)[2]
    assert np.array_equal(a, b)


def test_slot_contract_matches_brute_walk():
    wl = W.custom_family(W.HD256, [5, 17, 33, 1], [0, 16, 3, 40], seed=77, page_size=4)
    b = wl.batch
    req, pos = O.token_request_and_position(b.qo_indptr, b.start_pos)
    page, slot = O.slot_of(req, pos, b.kv_page_indptr, b.page_ids, b.page_size)
    for r in range(b.num_req):
        kv_len = int(b.start_pos[r] + b.qo_lens[r])
        walk = brute.slots_for_request(b.page_ids[b.kv_page_indptr[r]:b.kv_page_indptr[r + 1]],
                                       kv_len, b.page_size)
        for t in range(int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])):
            p = int(b.start_pos[r]) + t - int(b.qo_indptr[r])
            assert pos[t] == p
            assert (int(page[t]), int(slot[t])) == walk[p]


def test_pool_writes_hit_each_row_once_and_stay_in_the_layer():
    wl = W.custom_family(W.HD256, [9, 20], [0, 7], seed=5, num_layers=3, layer=1, spare_pages=3)
    b, f = wl.batch, wl.family
    req, pos = O.token_request_and_position(b.qo_indptr, b.start_pos)
    offs = O.prep_pool_writes(req, pos, b.kv_page_indptr, b.page_ids, b.page_size, wl.layer,
                              b.num_pages, f.num_kv_heads, f.head_dim)
    flat = offs.ravel()
    assert len(np.unique(flat)) == len(flat)
    layer_elems = b.num_pages * 2 * f.num_kv_heads * b.page_size * f.head_dim
    assert np.all(flat // layer_elems == 1)
    # the layout's own multi-index, flattened by numpy
    shape = (wl.num_layers, b.num_pages, 2, f.num_kv_heads, b.page_size, f.head_dim)
    for t in range(b.num_tokens):
        pg, sl = O.slot_of(req[t:t + 1], pos[t:t + 1], b.kv_page_indptr, b.page_ids, b.page_size)
        for kv in range(2):
            for h in range(f.num_kv_heads):
                idx = np.ravel_multi_index((wl.layer, int(pg[0]), kv, h, int(sl[0]), 0), shape)
                assert offs[t, kv, h] == idx


# ---------------------------------------------------------------------------- attention
def _paged_case(D, hq, hkv, qo_lens, start_pos, ps, seed, num_pages=None):
    """Random q and a random pool; returns oracle inputs plus contiguous K/V per request."""
    r = rng(seed)
    b = W.make_batch(r, qo_lens, start_pos, ps, num_pages=num_pages, spare_pages=2)
    T = b.num_tokens
    q = W.bf16_normal(r, (T, hq, D))
    pool = W.bf16_normal(r, (1, b.num_pages, 2, hkv, ps, D))
    return b, q, pool


def _contiguous_kv(b, pool, r):
    kv_len = int(b.start_pos[r] + b.qo_lens[r])
    pages = b.page_ids[b.kv_page_indptr[r]:b.kv_page_indptr[r + 1]]
    k = [[list(O.bf16_to_f64(pool[0, pages[j // b.page_size], 0, h, j % b.page_size]))
          for h in range(pool.shape[3])] for j in range(kv_len)]
    v = [[list(O.bf16_to_f64(pool[0, pages[j // b.page_size], 1, h, j % b.page_size]))
          for h in range(pool.shape[3])] for j in range(kv_len)]
    return k, v


@pytest.mark.parametrize("ps", [1, 4, 16])
@pytest.mark.parametrize("window_left", [-1, 0, 2, 100])
def test_attention_matches_brute(ps, window_left):
    D, hq, hkv = 8, 4, 2
    b, q, pool = _paged_case(D, hq, hkv, [7, 13, 1], [0, 5, 19], ps, seed=100 + ps)
    got = O.attention(q, pool, 0, b.qo_indptr, b.kv_page_indptr, b.page_ids, b.last_page_len,
                      b.start_pos, hkv, window_left, 0.7)
    for r in range(b.num_req):
        k, v = _contiguous_kv(b, pool, r)
        t0, t1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        qq = [[list(O.bf16_to_f64(q[t, h])) for h in range(hq)] for t in range(t0, t1)]
        pos = [int(b.start_pos[r]) + i for i in range(t1 - t0)]
        ref = brute.attention_contiguous(qq, k, v, pos, window_left, 0.7, hq // hkv)
        assert np.allclose(got[t0:t1], np.array(ref), atol=1e-12, rtol=0)


def _run(b, q, pool, hkv, w, scale=1.0, rows=None):
    return O.attention(q, pool, 0, b.qo_indptr, b.kv_page_indptr, b.page_ids, b.last_page_len,
                       b.start_pos, hkv, w, scale, rows=rows)


def test_window_zero_returns_own_value():
    b, q, pool = _paged_case(16, 4, 2, [11, 6], [0, 9], 4, seed=7)
    out = _run(b, q, pool, 2, 0)
    req, pos = O.token_request_and_position(b.qo_indptr, b.start_pos)
    page, slot = O.slot_of(req, pos, b.kv_page_indptr, b.page_ids, 4)
    for t in range(b.num_tokens):
        for h in range(4):
            assert np.array_equal(out[t, h], O.bf16_to_f64(pool[0, page[t], 1, h // 2, slot[t]]))


def test_wide_window_equals_plain_causal():
    b, q, pool = _paged_case(16, 4, 1, [20, 3], [0, 30], 4, seed=8)
    full = _run(b, q, pool, 1, -1)
    for w in [32, 33, 1000]:
        assert np.allclose(_run(b, q, pool, 1, w), full, atol=1e-13, rtol=0)
    assert not np.allclose(_run(b, q, pool, 1, 5), full)


def test_zero_scale_is_mean_of_visible_values():
    b, q, pool = _paged_case(8, 2, 1, [10], [4], 2, seed=9)
    out = _run(b, q, pool, 1, 3, scale=0.0)
    k, v = _contiguous_kv(b, pool, 0)
    for t in range(10):
        p = 4 + t
        vis = [j for j in range(p + 1) if p - j <= 3]
        mean = np.mean([v[j][0] for j in vis], axis=0)
        assert np.allclose(out[t, 0], mean, atol=1e-14)


def test_two_keys_closed_form():
    b, q, pool = _paged_case(8, 1, 1, [2], [0], 16, seed=10)
    out = _run(b, q, pool, 1, -1, scale=0.5)
    k, v = _contiguous_kv(b, pool, 0)
    qq = O.bf16_to_f64(q[1, 0])
    s0, s1 = 0.5 * qq @ np.array(k[0][0]), 0.5 * qq @ np.array(k[1][0])
    a = 1.0 / (1.0 + math.exp(s1 - s0))
    assert np.allclose(out[1, 0], a * np.array(v[0][0]) + (1 - a) * np.array(v[1][0]), atol=1e-14)
    assert np.array_equal(out[0, 0], np.array(v[0][0]))


def test_page_permutation_invariance():
    b, q, pool = _paged_case(16, 4, 2, [30, 12], [0, 21], 4, seed=11, num_pages=40)
    ref = _run(b, q, pool, 2, 9)
    perm = rng(12).permutation(b.num_pages)
    pool2 = np.empty_like(pool)
    pool2[:, perm] = pool
    b2 = W.Batch(b.qo_indptr, b.kv_page_indptr, perm[b.page_ids].astype(np.int32),
                 b.last_page_len, b.start_pos, b.page_size, b.num_pages)
    assert np.allclose(_run(b2, q, pool2, 2, 9), ref, atol=1e-13, rtol=0)


def test_batch_independence():
    b, q, pool = _paged_case(16, 4, 2, [9, 14, 5], [3, 0, 40], 4, seed=13)
    ref = _run(b, q, pool, 2, 7)
    for r in range(3):
        t0, t1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        p0, p1 = int(b.kv_page_indptr[r]), int(b.kv_page_indptr[r + 1])
        br = W.Batch(np.array([0, t1 - t0]), np.array([0, p1 - p0]), b.page_ids[p0:p1],
                     b.last_page_len[r:r + 1], b.start_pos[r:r + 1], 4, b.num_pages)
        assert np.allclose(_run(br, q[t0:t1], pool, 2, 7), ref[t0:t1], atol=1e-13, rtol=0)


def test_gqa_equals_mha_with_repeated_kv_heads():
    b, q, pool = _paged_case(16, 4, 2, [12], [3], 4, seed=14)
    ref = _run(b, q, pool, 2, -1)
    pool_mha = np.repeat(pool, 2, axis=3)   # kv head g -> heads 2g, 2g+1
    assert np.allclose(_run(b, q, pool_mha, 4, -1), ref, atol=1e-13, rtol=0)


def test_decode_equals_last_prefill_row():
    b, q, pool = _paged_case(16, 2, 1, [25], [0], 4, seed=15)
    full = _run(b, q, pool, 1, 6)
    bd = W.Batch(np.array([0, 1]), b.kv_page_indptr, b.page_ids, b.last_page_len,
                 np.array([24]), 4, b.num_pages)
    dec = _run(bd, q[24:25], pool, 1, 6)
    assert np.allclose(dec[0], full[24], atol=1e-13, rtol=0)


def test_sampled_rows_equal_full_evaluation():
    b, q, pool = _paged_case(16, 4, 2, [10, 7], [0, 3], 4, seed=16)
    full = _run(b, q, pool, 2, 4)
    rows = np.array([[0, 3], [12, 0], [16, 2], [5, 1]])
    got = _run(b, q, pool, 2, 4, rows=rows)
    for i, (t, h) in enumerate(rows):
        assert np.allclose(got[i], full[t, h], atol=1e-13, rtol=0)


def test_visible_pairs_counts():
    assert O.visible_pairs(np.array([0, 9]), np.array([0]), 3) == 30
    assert O.visible_pairs(np.array([0, 512]), np.array([0]), -1) == 131328
    assert O.visible_pairs(np.array([0, 16384]), np.array([0]), 1023) == 16253440
