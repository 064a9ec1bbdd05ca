"""Plain fp64 CPU oracle for paged two-family QKV prep and paged attention.

TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
benchmark's CPU-baseline leg may import this module. The product path (the
CUDA library and its Python binding) never calls it, and this module imports
nothing from the product package.

Everything is evaluated in float64 from the bf16 inputs; results are rounded to
bf16 only by ``f64_to_bf16`` when a caller compares them with bf16 outputs.
Each function states the passage it follows. The pages are three web pages of
one inference-engine project:

* "feat(kernels): Rust wrapper for the hd256 windowed paged prefill"
  (Description): attention reads a paged pool, ``sm_scale`` is explicit and
  unscaled attention uses 1.0, ``window_left`` has an inclusive-distance
  contract, GQA maps query heads to KV heads by integer division.
* "gemma4: serving prep needs pool-write forms" (Description, Proposed Plan):
  Q is RMS-normed and rotated into a contiguous buffer; K is normed and rotated
  and V weightless-normed, never rotated, straight into the layer's pool blocks;
  for head_dim 512, V is the weightless norm of the same raw K sharing its
  inverse RMS; the slot of token t is ``start_pos + t``.
* "feat(gemma4): paged KV serving across both attention families"
  (Description): local layers hd256 with 8 KV heads under a sliding window,
  global layers hd512 with 1 KV head under full attention; decode runs the
  prefill entry with one token.

Readings where the pages are silent (each listed in the design notes):
RMSNorm is ``x / sqrt(mean(x^2) + eps) * w`` with ``w`` a direct multiplier;
norm, then weight, then rotary; rotary pairs element ``i`` with ``i + D/2``
(half-split) over the full head dim with frequency ``theta^(-2i/D)``; the pool
is ``[layer][page][K=0,V=1][kv_head][slot][D]``; key ``j`` is visible from
query position ``p`` iff ``j <= p`` and (``window_left < 0`` or
``p - j <= window_left``).

Cascade attention for requests sharing a key prefix is a variant the pages
leave open; the oracle takes its plainest reading. A key segment is a request's
run of key positions [kv_start, kv_start + n) held from slot 0 of its pages;
``lse`` is the natural-log normaliser log sum_j exp(s_j) of the same masked
softmax; ``merge_states`` combines the states of two disjoint key sets exactly.

Row chunking in ``attention`` only bounds memory: every output row is the
plain definition evaluated on its own.
"""
from __future__ import annotations

import numpy as np

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


# --------------------------------------------------------------------------------------
# bf16 <-> fp64
# --------------------------------------------------------------------------------------
def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (uint16) as float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def f64_to_bf16(x) -> np.ndarray:
    """Round float64 values directly to bfloat16, nearest with ties to even.

    bf16 keeps 8 significant bits: for ``|x| = m * 2^e`` with ``0.5 <= m < 1``
    the spacing of representable values is ``2^(e-8)``, floored at the
    smallest subnormal ``2^-133``. ``np.rint`` rounds halves to even.
    """
    x = np.asarray(x, dtype=np.float64)
    finite = np.isfinite(x)
    xf = np.where(finite, x, 0.0)
    _, e = np.frexp(xf)
    sp = np.maximum(e - 8, -133)
    q = np.ldexp(np.rint(np.ldexp(xf, -sp)), sp)
    over = np.abs(q) > BF16_MAX
    q = np.where(over, np.copysign(np.inf, xf), q)
    q = np.where(finite, q, x)
    with np.errstate(over="ignore"):
        f = q.astype(np.float32)
    bits = (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    bits = np.where(np.isnan(x), np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


# --------------------------------------------------------------------------------------
# RMSNorm and rotary embedding
# --------------------------------------------------------------------------------------
def inv_rms(x: np.ndarray, eps: float) -> np.ndarray:
    """1 / sqrt(mean(x^2) + eps) over the last axis (per token, per head).

    "serving prep needs pool-write forms", Description: the hd512 V block
    shares this denominator with K.
    """
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def rope_cos_sin(positions, head_dim: int, theta: float):
    """cos and sin of ``pos * theta^(-2i/D)`` for i in [0, D/2), in fp64."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = float(theta) ** (-2.0 * i / head_dim)
    ang = np.asarray(positions, dtype=np.float64)[..., None] * inv_freq
    return np.cos(ang), np.sin(ang)


def rope_half_split(y: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate pairs (y[i], y[i + D/2]) by the angle whose cos/sin are given."""
    h = y.shape[-1] // 2
    a, b = y[..., :h], y[..., h:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1)


# --------------------------------------------------------------------------------------
# Positions and the slot contract
# --------------------------------------------------------------------------------------
def token_request_and_position(qo_indptr, start_pos):
    """Request index and absolute position of every token of a ragged batch.

    "serving prep needs pool-write forms", Proposed Plan: slot positions
    derive from ``start_pos + token``.
    """
    qo_indptr = np.asarray(qo_indptr, dtype=np.int64)
    start_pos = np.asarray(start_pos, dtype=np.int64)
    lens = np.diff(qo_indptr)
    req = np.repeat(np.arange(len(lens), dtype=np.int64), lens)
    local = np.arange(int(qo_indptr[-1]), dtype=np.int64) - qo_indptr[req]
    return req, start_pos[req] + local


def slot_of(req, pos, kv_page_indptr, page_ids, page_size: int, ring: bool = False,
            kv_start=None):
    """(physical page id, in-page slot) holding KV position ``pos`` of ``req``.

    With ``ring`` the request's pages form a ring ("serving prep needs pool-write forms",
    Proposed Plan: window-crossing callers need a separate slot mapping): logical page
    pos // page_size lives in the request's page (pos // page_size) mod (pages held), so a
    position reuses the slot of the position one ring length (pages x page_size) earlier.
    With ``kv_start`` (key segments) position kv_start_r + i lives in slot i of the request's
    pages: the index counts from the segment's first position.
    """
    kv_page_indptr = np.asarray(kv_page_indptr, dtype=np.int64)
    page_ids = np.asarray(page_ids, dtype=np.int64)
    req = np.asarray(req, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64)
    if kv_start is not None:
        pos = pos - np.asarray(kv_start, dtype=np.int64)[req]
    logical = pos // page_size
    if ring:
        logical = logical % (kv_page_indptr[req + 1] - kv_page_indptr[req])
    return page_ids[kv_page_indptr[req] + logical], pos % page_size


def pool_row_offset(layer, page, kv, head, slot, num_pages: int, num_kv_heads: int,
                    page_size: int, head_dim: int):
    """Element offset of one head row in a dense [L][P][2][Hkv][ps][D] pool."""
    return ((((np.asarray(layer, np.int64) * num_pages + page) * 2 + kv) * num_kv_heads
             + head) * page_size + slot) * head_dim


# --------------------------------------------------------------------------------------
# Prep: norm + rotary, K/V into the pool
# --------------------------------------------------------------------------------------
def prep_hd256(q_raw, k_raw, v_raw, w_q, w_k, eps, positions, theta):
    """hd256 serving prep ("serving prep needs pool-write forms", Proposed Plan,
    first item): q = rope(norm_wq(q)), k = rope(norm_wk(k)), v = norm(v) unrotated.

    Arrays are fp64: q_raw [T, Hq, D], k_raw/v_raw [T, Hkv, D], w [D].
    Returns (q_out, k, v) in fp64.
    """
    D = q_raw.shape[-1]
    c, s = rope_cos_sin(positions, D, theta)
    c, s = c[:, None, :], s[:, None, :]
    q = rope_half_split(q_raw * inv_rms(q_raw, eps) * w_q, c, s)
    k = rope_half_split(k_raw * inv_rms(k_raw, eps) * w_k, c, s)
    v = v_raw * inv_rms(v_raw, eps)
    return q, k, v


def prep_hd512(q_raw, k_raw, w_q, w_k, eps, positions, theta):
    """hd512 serving prep ("serving prep needs pool-write forms", Proposed Plan,
    second item): k = rope(norm_wk(k_raw)); v = k_raw * inv_rms(k_raw), the
    weightless norm of the same raw K with the same denominator, unrotated.
    Q is normed and rotated like the hd256 form.
    """
    D = q_raw.shape[-1]
    c, s = rope_cos_sin(positions, D, theta)
    c, s = c[:, None, :], s[:, None, :]
    q = rope_half_split(q_raw * inv_rms(q_raw, eps) * w_q, c, s)
    r_k = inv_rms(k_raw, eps)
    k = rope_half_split(k_raw * r_k * w_k, c, s)
    v = k_raw * r_k
    return q, k, v


def prep_pool_writes(req, pos, kv_page_indptr, page_ids, page_size, layer, num_pages,
                     num_kv_heads, head_dim, ring: bool = False, kv_start=None):
    """Element offsets [T, 2, Hkv] of the K and V rows each token writes."""
    page, slot = slot_of(req, pos, kv_page_indptr, page_ids, page_size, ring, kv_start)
    kv = np.arange(2, dtype=np.int64)[None, :, None]
    head = np.arange(num_kv_heads, dtype=np.int64)[None, None, :]
    return pool_row_offset(layer, page[:, None, None], kv, head, slot[:, None, None],
                           num_pages, num_kv_heads, page_size, head_dim)


# --------------------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------------------
def visible(p, j, window_left: int):
    """Causal mask with the inclusive-distance window ("Rust wrapper for the
    hd256 windowed paged prefill", Description): key j is visible from query
    position p iff j <= p and (window_left < 0 or p - j <= window_left)."""
    p = np.asarray(p)
    j = np.asarray(j)
    m = j <= p
    if window_left >= 0:
        m = m & (p - j <= window_left)
    return m


def gather_kv(pool_bits: np.ndarray, layer: int, pages_of_req, kv_len: int, page_size: int,
              ring: bool = False):
    """K and V of positions [0, kv_len) of one request, fp64 [kv_len, Hkv, D] each. With
    ``ring`` (see slot_of) a position older than one ring length reads whatever newer position
    now holds its slot; the window mask keeps such keys out of every softmax."""
    j = np.arange(kv_len, dtype=np.int64)
    pages_of_req = np.asarray(pages_of_req, dtype=np.int64)
    logical = j // page_size
    if ring:
        logical = logical % len(pages_of_req)
    pages = pages_of_req[logical]
    slots = j % page_size
    k = bf16_to_f64(pool_bits[layer, pages, 0, :, slots, :])
    v = bf16_to_f64(pool_bits[layer, pages, 1, :, slots, :])
    return k, v


def attend_rows(q_rows, p_rows, k, v, window_left: int, sm_scale: float, key_pos=None,
                with_lse: bool = False):
    """Masked softmax attention of query rows q_rows [n, D] at positions p_rows
    over keys k [kv, D] and values v [kv, D]: o = sum_j softmax_j(s) v_j with
    s_j = sm_scale * <q, k_j> over the visible j. ``key_pos`` gives the keys'
    positions (default 0 .. kv-1).

    With ``with_lse`` also returns lse = log(sum_j exp(s_j)) over the visible j, the
    normaliser of the same softmax (natural log). A row that sees no key has o = 0 and
    lse = -inf: the neutral state of merge_states.
    """
    key_pos = np.arange(k.shape[0]) if key_pos is None else np.asarray(key_pos)
    s = sm_scale * (q_rows @ k.T)
    mask = visible(np.asarray(p_rows)[:, None], key_pos[None, :], window_left)
    s = np.where(mask, s, -np.inf)
    seen = mask.any(axis=1)
    m = np.where(seen, np.max(s, axis=1), 0.0)[:, None]
    e = np.where(mask, np.exp(s - m), 0.0)
    den = np.sum(e, axis=1, keepdims=True)
    o = np.where(seen[:, None], (e @ v) / np.where(den > 0, den, 1.0), 0.0)
    if not with_lse:
        return o
    lse = np.where(seen, m[:, 0] + np.log(np.where(seen, den[:, 0], 1.0)), -np.inf)
    return o, lse


def merge_states(o_a, lse_a, o_b, lse_b):
    """Attention state of the union of two disjoint key sets from the states of each:
    with w_x = exp(lse_x - M), M = max(lse_a, lse_b), o = (w_a o_a + w_b o_b) / (w_a + w_b)
    and lse = M + log(w_a + w_b). The softmax over the union is the two softmaxes reweighted
    by their normalisers, so merging is exact; (0, -inf) is the neutral state.
    """
    o_a, o_b = np.asarray(o_a, np.float64), np.asarray(o_b, np.float64)
    lse_a, lse_b = np.asarray(lse_a, np.float64), np.asarray(lse_b, np.float64)
    M = np.maximum(lse_a, lse_b)
    fin = np.isfinite(M)
    Mz = np.where(fin, M, 0.0)
    wa = np.where(np.isfinite(lse_a), np.exp(lse_a - Mz), 0.0)
    wb = np.where(np.isfinite(lse_b), np.exp(lse_b - Mz), 0.0)
    den = wa + wb
    o = np.where(fin[..., None], (wa[..., None] * o_a + wb[..., None] * o_b)
                 / np.where(den > 0, den, 1.0)[..., None], 0.0)
    lse = np.where(fin, Mz + np.log(np.where(den > 0, den, 1.0)), -np.inf)
    return o, lse


def attention(q_bits, pool_bits, layer: int, qo_indptr, kv_page_indptr, page_ids,
              last_page_len, start_pos, num_kv_heads: int, window_left: int,
              sm_scale: float, rows=None, row_chunk: int = 512, ring: bool = False,
              kv_start=None, return_lse: bool = False):
    """Paged prefill attention over a page table (fp64).

    q_bits: bf16 bits [T, Hq, D]; pool_bits: bf16 bits [L, P, 2, Hkv, ps, D].
    The kv length of request r is (pages_r - 1) * ps + last_page_len_r (with ``ring``:
    start_pos_r + qo_len_r, the pages forming a ring, see slot_of), and its
    queries sit at positions start_pos_r + t. Query head h reads KV head
    h // (Hq / Hkv). ``rows``: optional int array [n, 2] of (token, head) to
    evaluate; returns fp64 [n, D]. Without it returns fp64 [T, Hq, D].

    ``kv_start`` (a key segment, for cascade attention): request r's pages hold key
    positions [kv_start_r, kv_start_r + n_r), n_r = (pages_r - 1) * ps + last_page_len_r,
    position kv_start_r + i in slot i (page i // ps, offset i % ps); keys outside the
    segment are not seen. ``return_lse`` also returns the natural-log normaliser of every
    row (see attend_rows), shaped like the output without its last axis.
    """
    qo_indptr = np.asarray(qo_indptr, dtype=np.int64)
    kv_page_indptr = np.asarray(kv_page_indptr, dtype=np.int64)
    page_ids = np.asarray(page_ids, dtype=np.int64)
    if not ring:
        last_page_len = np.asarray(last_page_len, dtype=np.int64)
    T, Hq, D = q_bits.shape
    ps = pool_bits.shape[4]
    group = Hq // num_kv_heads
    req_of, pos_of = token_request_and_position(qo_indptr, start_pos)
    if rows is None:
        tt, hh = np.meshgrid(np.arange(T), np.arange(Hq), indexing="ij")
        sel = np.stack([tt.ravel(), hh.ravel()], axis=1)
    else:
        sel = np.asarray(rows, dtype=np.int64).reshape(-1, 2)
    out = np.zeros((len(sel), D), dtype=np.float64)
    lse = np.full(len(sel), -np.inf, dtype=np.float64)
    sel_req = req_of[sel[:, 0]] if len(sel) else np.zeros(0, np.int64)
    for r in np.unique(sel_req):
        npages = kv_page_indptr[r + 1] - kv_page_indptr[r]
        if ring:
            kv_len = int(np.asarray(start_pos, np.int64)[r] + qo_indptr[r + 1] - qo_indptr[r])
        else:
            kv_len = int((npages - 1) * ps + last_page_len[r])
        # kv_len keys from slot 0 on: positions 0 .. kv_len-1, or the segment's
        k, v = gather_kv(pool_bits, layer, page_ids[kv_page_indptr[r]:kv_page_indptr[r + 1]],
                         kv_len, ps, ring)
        key_pos = np.arange(kv_len, dtype=np.int64)
        if kv_start is not None:
            key_pos = key_pos + int(np.asarray(kv_start, np.int64)[r])
        idx_r = np.nonzero(sel_req == r)[0]
        for g in range(num_kv_heads):
            idx = idx_r[(sel[idx_r, 1] // group) == g]
            for c in range(0, len(idx), row_chunk):
                ii = idx[c:c + row_chunk]
                qr = bf16_to_f64(q_bits[sel[ii, 0], sel[ii, 1], :])
                out[ii], lse[ii] = attend_rows(qr, pos_of[sel[ii, 0]], k[:, g, :], v[:, g, :],
                                               window_left, sm_scale, key_pos, with_lse=True)
    if rows is None:
        out, lse = out.reshape(T, Hq, D), lse.reshape(T, Hq)
    return (out, lse) if return_lse else out


def visible_pairs(qo_indptr, start_pos, window_left: int) -> int:
    """Number of (query, key) pairs the mask keeps, per query head."""
    _, pos = token_request_and_position(qo_indptr, start_pos)
    n = pos + 1
    if window_left >= 0:
        n = np.minimum(n, window_left + 1)
    return int(n.sum())
