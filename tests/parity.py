"""Parity helpers: oracle expectations for a workload family and the comparison gates.

Gates:
* prep: |gpu - bf16(oracle)| <= ulp_bf16(max(|oracle|, 2^-8)) element by element (one
  bf16 ulp; below 2^-8 the floor 2^-15 absorbs fp32 cancellation in the rotation),
  untouched pool rows byte-exact;
* attention: max |gpu - oracle| <= 3e-2 and mean |gpu - oracle| <= 3e-3 against the
  unrounded fp64 oracle.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as O
from paged_sliding_window_qkv_gb300.runner import device_to_bits
from paged_sliding_window_qkv_gb300 import workloads as W

ATTN_MAX = 3e-2
ATTN_MEAN = 3e-3


def ulp_bf16(x):
    x = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -8)
    _, e = np.frexp(x)
    return np.ldexp(1.0, e - 8)


def prep_gate(gpu_bits, ref64, what=""):
    gpu = O.bf16_to_f64(gpu_bits)
    refr = O.bf16_to_f64(O.f64_to_bf16(ref64))
    err = np.abs(gpu - refr)
    tol = ulp_bf16(ref64)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements beyond 1 bf16 ulp; "
                           f"worst {float(np.max(err - tol)):.3e}")
    return float(np.mean(err == 0))


def attn_gate(gpu, ref, what=""):
    err = np.abs(np.asarray(gpu, np.float64) - ref)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= ATTN_MAX and mean <= ATTN_MEAN, f"{what}: max {mx:.3e} mean {mean:.3e}"
    return mx, mean


def prep_reference(fi: W.FamilyInputs, ring: bool = False):
    """Oracle prep outputs (fp64) and the pool row offsets each token writes."""
    f, b = fi.family, fi.batch
    req, pos = O.token_request_and_position(b.qo_indptr, b.start_pos)
    q = O.bf16_to_f64(fi.q_raw)
    k = O.bf16_to_f64(fi.k_raw)
    wq, wk = O.bf16_to_f64(fi.w_q), O.bf16_to_f64(fi.w_k)
    if f.head_dim == 256:
        qo, ko, vo = O.prep_hd256(q, k, O.bf16_to_f64(fi.v_raw), wq, wk, fi.eps, pos, f.rope_theta)
    else:
        qo, ko, vo = O.prep_hd512(q, k, wq, wk, fi.eps, pos, f.rope_theta)
    offs = O.prep_pool_writes(req, pos, b.kv_page_indptr, b.page_ids, b.page_size, fi.layer,
                              b.num_pages, f.num_kv_heads, f.head_dim, ring=ring)
    return qo, ko, vo, offs


def check_prep(run, fi: W.FamilyInputs, initial_pool_bits=None, ring: bool = False):
    """Compare q_out and the pool after prep with the oracle; untouched rows byte-exact."""
    torch.cuda.synchronize()
    f = fi.family
    D = f.head_dim
    qo, ko, vo, offs = prep_reference(fi, ring)
    frac_q = prep_gate(device_to_bits(run.q_out), qo, "q_out")
    rows_dev = run.pool.view(-1, D)
    row_idx = torch.from_numpy((offs // D).reshape(-1)).to(rows_dev.device)
    got = device_to_bits(rows_dev.index_select(0, row_idx)).reshape(offs.shape + (D,))
    frac_k = prep_gate(got[:, 0], ko, "K rows")
    frac_v = prep_gate(got[:, 1], vo, "V rows")
    # untouched sweep: every other row keeps its initial bytes
    written = torch.zeros(rows_dev.shape[0], dtype=torch.bool, device=rows_dev.device)
    written[row_idx] = True
    if initial_pool_bits is None:
        sentinel = torch.tensor(np.array([W.POOL_SENTINEL], np.uint16).view(np.int16)[0],
                                dtype=torch.int16, device=rows_dev.device)
        changed = (rows_dev.view(torch.int16) != sentinel).any(dim=1)
    else:
        init = torch.from_numpy(np.ascontiguousarray(initial_pool_bits).view(np.int16).reshape(-1, D))
        changed = (rows_dev.view(torch.int16) != init.to(rows_dev.device)).any(dim=1)
    stray = changed & ~written
    assert not bool(stray.any()), f"{int(stray.sum())} pool rows outside the written slots changed"
    return frac_q, frac_k, frac_v


def attn_reference(fi: W.FamilyInputs, q_bits, pool_bits, window_left=None, rows=None,
                   ring: bool = False):
    b = fi.batch
    w = fi.family.window_left if window_left is None else window_left
    return O.attention(q_bits, pool_bits, fi.layer, b.qo_indptr, b.kv_page_indptr, b.page_ids,
                       b.last_page_len, b.start_pos, fi.family.num_kv_heads, w, fi.sm_scale,
                       rows=rows, ring=ring)


def bf16_out(run):
    torch.cuda.synchronize()
    return O.bf16_to_f64(device_to_bits(run.out))
