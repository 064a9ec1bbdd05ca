"""Brute-force restatement of the method on tiny inputs, in pure-Python loops.

Independent of ``oracle/`` (imports nothing from it): it builds dense mask
matrices, contiguous (unpaged) K/V and evaluates every sum with ``math``. It
exists only to pin the oracle on inputs small enough for loops.
"""
from __future__ import annotations

import math


def rmsnorm_row(x, w, eps):
    """x * w / sqrt(mean(x^2) + eps) for one head row (w=None: weightless)."""
    d = len(x)
    ss = 0.0
    for a in x:
        ss += a * a
    r = 1.0 / math.sqrt(ss / d + eps)
    if w is None:
        return [a * r for a in x], r
    return [x[i] * r * w[i] for i in range(d)], r


def rope_row(y, pos, theta):
    """Half-split rotary: pair (i, i + D/2) rotated by pos * theta^(-2i/D)."""
    d = len(y)
    h = d // 2
    out = [0.0] * d
    for i in range(h):
        ang = pos * theta ** (-2.0 * i / d)
        c, s = math.cos(ang), math.sin(ang)
        out[i] = y[i] * c - y[i + h] * s
        out[i + h] = y[i + h] * c + y[i] * s
    return out


def dense_mask(q_positions, kv_len, window_left):
    """M[i][j] = 1 iff key j is visible from query i (inclusive-distance window)."""
    m = []
    for p in q_positions:
        row = []
        for j in range(kv_len):
            ok = j <= p
            if window_left >= 0 and p - j > window_left:
                ok = False
            row.append(1 if ok else 0)
        m.append(row)
    return m


def attention_contiguous(q, k, v, q_positions, window_left, sm_scale, group):
    """q [n][Hq][D], k/v [kv][Hkv][D] (contiguous positions 0..kv-1).

    Returns o [n][Hq][D] with query head h reading KV head h // group.
    """
    n, hq, d = len(q), len(q[0]), len(q[0][0])
    kv = len(k)
    mask = dense_mask(q_positions, kv, window_left)
    out = []
    for i in range(n):
        orow = []
        for h in range(hq):
            g = h // group
            s = []
            for j in range(kv):
                if mask[i][j]:
                    acc = 0.0
                    for e in range(d):
                        acc += q[i][h][e] * k[j][g][e]
                    s.append(sm_scale * acc)
                else:
                    s.append(None)
            mx = max(x for x in s if x is not None)
            num = [0.0] * d
            den = 0.0
            for j in range(kv):
                if s[j] is None:
                    continue
                wgt = math.exp(s[j] - mx)
                den += wgt
                for e in range(d):
                    num[e] += wgt * v[j][g][e]
            orow.append([x / den for x in num])
        out.append(orow)
    return out


def slots_for_request(page_ids, kv_len, page_size):
    """[(page_id, slot)] for positions 0..kv_len-1, by walking pages one slot at a time."""
    out = []
    pi, slot = 0, 0
    for _ in range(kv_len):
        out.append((int(page_ids[pi]), slot))
        slot += 1
        if slot == page_size:
            slot = 0
            pi += 1
    return out


def lse_contiguous(q, k, q_positions, key_positions, window_left, sm_scale, group):
    """log(sum_j exp(sm_scale <q, k_j>)) over the keys visible from each query, by loops.

    q [n][Hq][D]; k [kv][Hkv][D] with key j at position key_positions[j]. Returns
    lse [n][Hq]; -inf where a query sees no key.
    """
    out = []
    for i, p in enumerate(q_positions):
        row = []
        for h in range(len(q[i])):
            g = h // group
            s = []
            for j, kp in enumerate(key_positions):
                if kp > p or (window_left >= 0 and p - kp > window_left):
                    continue
                acc = 0.0
                for e in range(len(q[i][h])):
                    acc += q[i][h][e] * k[j][g][e]
                s.append(sm_scale * acc)
            if not s:
                row.append(-math.inf)
                continue
            mx = max(s)
            row.append(mx + math.log(sum(math.exp(x - mx) for x in s)))
        out.append(row)
    return out
