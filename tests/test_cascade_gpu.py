"""Cascade attention on the GPU: log-sum-exp outputs, key-segment plans and state merging.

Requests share a key prefix; attention over each request's keys equals the merge of attention
over the shared prefix (one segment plan that lists the same pages for every request) and over
the request's own keys (a second segment plan). Checked against the oracle, whose segment,
lse and merge functions the CPU tests pin to brute force and closed forms:

* out: the attention gate (max 3e-2, mean 3e-3 against fp64);
* lse: |gpu - oracle| <= 1e-2. The kernels normalise by the sum of the bf16-rounded softmax
  weights they multiply V by; each weight carries a relative rounding error below 2^-8, so the
  sum (and exp(lse)) is within 2^-8 relative and lse within about 4e-3 of the exact value;
  fp32 scores add far less. The gate keeps a factor of about 2.5 above that.
"""
import numpy as np
import pytest
import torch

import brute
import parity as PT
from oracle import oracle as O
from paged_sliding_window_qkv_gb300 import pg
from paged_sliding_window_qkv_gb300 import workloads as W
from paged_sliding_window_qkv_gb300.runner import bits_to_device, device_to_bits
from test_oracle_cascade import fill_pool

pytestmark = pytest.mark.gpu

LSE_TOL = 1e-2
FAMS = {256: (16, 8), 512: (16, 1)}


def plan_of(b: W.Batch, hq, hkv, D, kv_start=None):
    if kv_start is None:
        rc, plan = pg.pg_plan_paged_prefill(None, b.num_req, b.qo_indptr, b.kv_page_indptr,
                                            b.page_ids, b.last_page_len, b.start_pos, hq, hkv,
                                            D, b.page_size)
    else:
        rc, plan = pg.pg_plan_paged_segment(None, b.num_req, b.qo_indptr, b.kv_page_indptr,
                                            b.page_ids, b.last_page_len, kv_start, b.start_pos,
                                            hq, hkv, D, b.page_size)
    pg.check(rc, "plan")
    return plan


def attn_lse(plan, pool_desc, q, D, window, scale):
    T, hq = q.shape[0], q.shape[1]
    out = torch.empty(T, hq, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, hq, dtype=torch.float32, device="cuda")
    ws_bytes = pg.pg_workspace_bytes(plan)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda") if ws_bytes else None
    fn = pg.pg_attn_paged_prefill_lse if D == 256 else pg.pg_attn_paged_prefill_hd512_lse
    pg.check(fn(plan, pool_desc, 0, q, out, lse, window, scale, ws, ws_bytes), "attention+lse")
    return out, lse


def lse_gate(gpu, ref, what):
    gpu = np.asarray(gpu, np.float64)
    both_inf = np.isneginf(gpu) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):  # -inf - -inf where both are the neutral state
        err = np.where(both_inf, 0.0, np.abs(gpu - ref))
    assert np.all(np.isfinite(err)), f"{what}: -inf rows disagree"
    assert err.max() <= LSE_TOL, f"{what}: lse max err {err.max():.3e}"


CASES = [
    # D, prefix, suffix lens, step lens, window, page size
    (256, 300, [40, 130, 64], [40, 17, 64], -1, 16),     # prefill steps (tcgen05 path)
    (256, 300, [90, 250, 33], [90, 1, 9], 100, 16),      # window inside the suffix for late rows
    (256, 700, [600, 300, 5], [1, 1, 1], 500, 16),       # decode steps, several key chunks
    (512, 257, [100, 63], [100, 40], -1, 16),
    (512, 1100, [700, 20], [1, 1], -1, 16),              # decode, chunked prefix
    (512, 150, [80, 31], [80, 31], 60, 16),
    (256, 90, [30, 17], [30, 5], -1, 4),                  # page size 4: the general kernel
    (256, 333, [70, 140], [70, 33], 200, 32),             # tcgen05 path, one K box per page
    (512, 205, [90, 45], [90, 45], -1, 8),                # tcgen05 path, four K boxes per part
]


@pytest.mark.parametrize("D,prefix,suffix,steps,window,ps", CASES)
def test_cascade_matches_single_pass_and_oracle(D, prefix, suffix, steps, window, ps):
    hq, hkv = FAMS[D]
    rng = np.random.Generator(np.random.PCG64(D + prefix + window))
    ci = W.make_cascade(rng, prefix, suffix, steps, ps, hq, hkv, D)
    pool_bits = fill_pool(ci)
    pool = bits_to_device(pool_bits)
    desc = pg.pool_descriptor(pool)
    q = bits_to_device(ci.q)
    R = ci.full.num_req
    scale = 0.06
    plans = [plan_of(ci.full, hq, hkv, D), plan_of(ci.prefix, hq, hkv, D, np.zeros(R, np.int64)),
             plan_of(ci.suffix, hq, hkv, D, np.full(R, prefix, np.int64))]
    (o_full, l_full), (o_pre, l_pre), (o_suf, l_suf) = [attn_lse(p, desc, q, D, window, scale)
                                                        for p in plans]
    o_m = torch.empty_like(o_full)
    l_m = torch.empty_like(l_full)
    rows = o_full.shape[0] * hq
    pg.check(pg.pg_merge_attn_states(o_pre, l_pre, o_suf, l_suf, o_m, l_m, rows, D), "merge")
    torch.cuda.synchronize()
    assert pg.pg_device_status() == pg.PG_OK
    ref_o, ref_l = O.attention(ci.q, pool_bits, 0, ci.full.qo_indptr, ci.full.kv_page_indptr,
                               ci.full.page_ids, ci.full.last_page_len, ci.full.start_pos, hkv,
                               window, scale, return_lse=True)
    ref_po, ref_pl = O.attention(ci.q, pool_bits, 0, ci.prefix.qo_indptr,
                                 ci.prefix.kv_page_indptr, ci.prefix.page_ids,
                                 ci.prefix.last_page_len, ci.prefix.start_pos, hkv, window, scale,
                                 kv_start=np.zeros(R, np.int64), return_lse=True)
    bits = lambda t: O.bf16_to_f64(device_to_bits(t))
    PT.attn_gate(bits(o_full), ref_o, "single pass")
    lse_gate(l_full.cpu().numpy(), ref_l, "single pass")
    PT.attn_gate(bits(o_pre), ref_po, "prefix segment")
    lse_gate(l_pre.cpu().numpy(), ref_pl, "prefix segment")
    PT.attn_gate(bits(o_m), ref_o, "merged cascade")
    lse_gate(l_m.cpu().numpy(), ref_l, "merged cascade")
    if window >= 0:
        # rows whose window misses the whole prefix: the neutral state, exactly
        none = np.isneginf(ref_pl)
        assert np.isneginf(l_pre.cpu().numpy()[none]).all()
        assert (device_to_bits(o_pre)[none] == 0).all()
    for p in plans:
        p.close()


def test_merge_kernel_matches_oracle_and_may_write_in_place():
    rng = np.random.Generator(np.random.PCG64(31))
    rows, D = 1000, 512
    oa, ob = W.bf16_normal(rng, (rows, D)), W.bf16_normal(rng, (rows, D))
    la = (rng.standard_normal(rows) * 6).astype(np.float32)
    lb = (rng.standard_normal(rows) * 6).astype(np.float32)
    la[::7] = -np.inf
    lb[::11] = -np.inf
    ref_o, ref_l = O.merge_states(O.bf16_to_f64(oa), la, O.bf16_to_f64(ob), lb)
    ta, tb = bits_to_device(oa), bits_to_device(ob)
    tla, tlb = torch.from_numpy(la).cuda(), torch.from_numpy(lb).cuda()
    pg.check(pg.pg_merge_attn_states(ta, tla, tb, tlb, ta, tla, rows, D), "merge in place")
    torch.cuda.synchronize()
    got = O.bf16_to_f64(device_to_bits(ta))
    # fp32 weights, one bf16 rounding of the result
    assert np.all(np.abs(got - ref_o) <= PT.ulp_bf16(ref_o) + 1e-5 * np.abs(ref_o).max())
    gl = tla.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref_l)
    assert np.array_equal(np.isneginf(gl), ~fin)
    assert np.abs(gl[fin] - ref_l[fin]).max() <= 1e-5 * max(1.0, np.abs(ref_l[fin]).max())


def test_prep_on_a_suffix_segment_writes_its_slots_and_the_prefix_plan_refuses_prep():
    hq, hkv, D, ps = 16, 8, 256, 16
    rng = np.random.Generator(np.random.PCG64(77))
    ci = W.make_cascade(rng, 45, [30, 9], [30, 9], ps, hq, hkv, D)
    R = ci.full.num_req
    suf = plan_of(ci.suffix, hq, hkv, D, np.full(R, 45, np.int64))
    pre = plan_of(ci.prefix, hq, hkv, D, np.zeros(R, np.int64))
    fi = W.family_inputs(rng, W.HD256, ci.suffix, 1, 0, "sentinel", 5)
    pool = torch.full(fi.pool_shape, -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    desc = pg.pool_descriptor(pool)
    rope_rows = 256
    cos = torch.empty(rope_rows, D // 2, dtype=torch.float32, device="cuda")
    sin = torch.empty_like(cos)
    pg.check(pg.pg_rope_table(cos, sin, rope_rows, D, W.HD256.rope_theta), "rope")
    dev = {k: bits_to_device(getattr(fi, k)) for k in ("q_raw", "k_raw", "v_raw", "w_q", "w_k")}
    q_out = torch.empty(ci.full.num_tokens, hq, D, dtype=torch.bfloat16, device="cuda")
    args = (desc, 0, dev["q_raw"], hq * D, dev["k_raw"], hkv * D, dev["v_raw"], hkv * D,
            dev["w_q"], dev["w_k"], fi.eps, cos, sin, rope_rows, q_out)
    before = pg.pg_launch_count()
    assert pg.pg_prep_paged_hd256(pre, *args) == pg.PG_ERR_COVERAGE
    assert pg.pg_launch_count() == before
    pg.check(pg.pg_prep_paged_hd256(suf, *args), "prep on the suffix segment")
    torch.cuda.synchronize()
    # expected: token at position p writes index p - 45 of the request's suffix pages
    req, pos = O.token_request_and_position(ci.suffix.qo_indptr, ci.suffix.start_pos)
    qo, ko, vo = O.prep_hd256(O.bf16_to_f64(fi.q_raw), O.bf16_to_f64(fi.k_raw),
                              O.bf16_to_f64(fi.v_raw), O.bf16_to_f64(fi.w_q),
                              O.bf16_to_f64(fi.w_k), fi.eps, pos, W.HD256.rope_theta)
    pb = device_to_bits(pool)
    for t in range(len(pos)):
        r = int(req[t])
        pages = ci.suffix.page_ids[ci.suffix.kv_page_indptr[r]:ci.suffix.kv_page_indptr[r + 1]]
        walk = brute.slots_for_request(pages, int(pos[t]) - 45 + 1, ps)
        pgid, sl = walk[-1]
        PT.prep_gate(pb[0, pgid, 0, :, sl, :], ko[t], f"K row of token {t}")
        PT.prep_gate(pb[0, pgid, 1, :, sl, :], vo[t], f"V row of token {t}")
    PT.prep_gate(device_to_bits(q_out), qo, "q_out")
    suf.close()
    pre.close()


def test_segment_decode_without_allocation_matches_the_workspace_path():
    hq, hkv = FAMS[512]
    D = 512
    rng = np.random.Generator(np.random.PCG64(5150))
    ci = W.make_cascade(rng, 1100, [700, 20, 3], [1, 1, 1], 16, hq, hkv, D)
    pool = bits_to_device(fill_pool(ci, full=False))
    desc = pg.pool_descriptor(pool)
    q = bits_to_device(ci.q)
    R = ci.full.num_req
    for b, ks in ((ci.prefix, np.zeros(R, np.int64)), (ci.suffix, np.full(R, 1100, np.int64))):
        plan = plan_of(b, hq, hkv, D, ks)
        ref, _ = attn_lse(plan, desc, q, D, -1, 0.06)
        out = torch.empty_like(ref)
        pg.check(pg.pg_attn_paged_decode_noalloc(plan, desc, 0, q, out, -1, 0.06), "noalloc decode")
        torch.cuda.synchronize()
        assert np.array_equal(device_to_bits(out), device_to_bits(ref))
        plan.close()
