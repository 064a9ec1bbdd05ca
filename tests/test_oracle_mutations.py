"""Plant plausible mistakes in the oracle (CPU only) and check that a pin fails.

Each case monkeypatches one oracle function with a wrong variant and runs the
pin that should catch it; the test passes only if that pin now fails.
"""
import numpy as np
import pytest

import test_oracle_cascade as CA
import test_oracle_pins as P
from oracle import oracle as O


def _interleaved_rope(y, cos, sin):
    out = np.empty_like(y)
    out[..., 0::2] = y[..., 0::2] * cos - y[..., 1::2] * sin
    out[..., 1::2] = y[..., 1::2] * cos + y[..., 0::2] * sin
    return out


def _sign_flipped_rope(y, cos, sin):
    h = y.shape[-1] // 2
    a, b = y[..., :h], y[..., h:]
    return np.concatenate([a * cos + b * sin, b * cos - a * sin], axis=-1)


def _wrong_frequency(positions, head_dim, theta):
    i = np.arange(head_dim // 2, dtype=np.float64)
    ang = np.asarray(positions, dtype=np.float64)[..., None] * float(theta) ** (-i / head_dim)
    return np.cos(ang), np.sin(ang)


def _sum_not_mean_rms(x, eps):
    return 1.0 / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def _window_off_by_one(p, j, window_left):
    p, j = np.asarray(p), np.asarray(j)
    m = j <= p
    if window_left >= 0:
        m = m & (p - j < window_left)
    return m


def _non_causal(p, j, window_left):
    p, j = np.asarray(p), np.asarray(j)
    m = np.ones(np.broadcast(p, j).shape, bool)
    if window_left >= 0:
        m = m & (np.abs(p - j) <= window_left)
    return m


def _slot_off_by_one(req, pos, kv_page_indptr, page_ids, page_size):
    kv_page_indptr = np.asarray(kv_page_indptr, dtype=np.int64)
    page_ids = np.asarray(page_ids, dtype=np.int64)
    pos = np.asarray(pos, dtype=np.int64) + 1
    return page_ids[kv_page_indptr[np.asarray(req)] + pos // page_size], pos % page_size


def _rotated_v_hd512(q_raw, k_raw, w_q, w_k, eps, positions, theta):
    D = q_raw.shape[-1]
    c, s = O.rope_cos_sin(positions, D, theta)
    c, s = c[:, None, :], s[:, None, :]
    q = O.rope_half_split(q_raw * O.inv_rms(q_raw, eps) * w_q, c, s)
    r_k = O.inv_rms(k_raw, eps)
    k = O.rope_half_split(k_raw * r_k * w_k, c, s)
    return q, k, O.rope_half_split(k_raw * r_k, c, s)


def _merge_without_normalisers(o_a, lse_a, o_b, lse_b):
    # averages the two states as if both had the same normaliser
    return (np.asarray(o_a) + np.asarray(o_b)) / 2, np.maximum(lse_a, lse_b)


_attend = O.attend_rows


def _lse_is_the_max(q_rows, p_rows, k, v, window_left, sm_scale, key_pos=None, with_lse=False):
    # returns the row maximum where the log-sum-exp belongs
    res = _attend(q_rows, p_rows, k, v, window_left, sm_scale, key_pos, with_lse)
    if not with_lse:
        return res
    kp = np.arange(k.shape[0]) if key_pos is None else np.asarray(key_pos)
    s = sm_scale * (q_rows @ k.T)
    mask = O.visible(np.asarray(p_rows)[:, None], kp[None, :], window_left)
    return res[0], np.where(mask.any(1), np.max(np.where(mask, s, -np.inf), axis=1), -np.inf)


def _segment_ignored(q_rows, p_rows, k, v, window_left, sm_scale, key_pos=None, with_lse=False):
    # reads a key segment as if it started at position 0
    return _attend(q_rows, p_rows, k, v, window_left, sm_scale, None, with_lse)


MUTATIONS = [
    ("rope_half_split", _interleaved_rope, lambda: P.test_rope_half_split_pairing_sign_and_frequency_d4()),
    ("rope_half_split", _sign_flipped_rope, lambda: P.test_rope_d2_is_textbook_rotation()),
    ("rope_cos_sin", _wrong_frequency, lambda: P.test_rope_half_split_pairing_sign_and_frequency_d4()),
    ("inv_rms", _sum_not_mean_rms, lambda: P.test_inv_rms_closed_form_d4()),
    ("visible", _window_off_by_one, lambda: P.test_attention_matches_brute(4, 2)),
    ("visible", _non_causal, lambda: P.test_attention_matches_brute(4, -1)),
    ("slot_of", _slot_off_by_one, lambda: P.test_slot_contract_matches_brute_walk()),
    ("prep_hd512", _rotated_v_hd512, lambda: P.test_prep_hd512_form_v_is_weightless_norm_of_raw_k()),
    ("merge_states", _merge_without_normalisers,
     lambda: CA.test_prefix_and_suffix_merge_to_the_single_pass(37, [5, 20, 1], [5, 3, 1], -1, 4)),
    ("attend_rows", _lse_is_the_max, lambda: CA.test_lse_matches_brute_force()),
    ("attend_rows", _segment_ignored,
     lambda: CA.test_prefix_and_suffix_merge_to_the_single_pass(16, [9, 33], [9, 17], 11, 8)),
]


@pytest.mark.parametrize("name,bad,pin", MUTATIONS,
                         ids=[f"{m[0]}:{m[1].__name__}" for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, bad, pin):
    monkeypatch.setattr(O, name, bad)
    with pytest.raises(AssertionError):
        pin()
