"""Window-crossing requests streamed through ring-addressed pages on the GPU.

"gemma4: serving prep needs pool-write forms", Proposed Plan: slots equal positions only
below the sliding window, and callers that cross it need a separate slot mapping. With
pg_plan_paged_prefill_ring a request holds a fixed ring of pages; position p lives in
page (p / page_size) mod (pages held). Three requests are streamed in mixed prefill and
decode steps until their rings have wrapped; every step's prep (pool writes, q_out) and
attention are compared with the oracle's ring mapping, which the CPU tests pin to a dense
brute force over the true history.
"""
import numpy as np
import pytest
import torch

import parity as PT
from oracle import oracle as O
from paged_sliding_window_qkv_gb300 import pg
from paged_sliding_window_qkv_gb300 import workloads as W
from paged_sliding_window_qkv_gb300.runner import FamilyRun, device_to_bits

pytestmark = pytest.mark.gpu

PS = 16
WIN = 100
# per batch step, the new tokens of each request; all-ones rows are decode steps
SCHEDULE = [[300, 37, 16], [1, 1, 1], [250, 1, 64], [7, 1, 1], [1, 300, 1], [400, 1, 64],
            [1, 1, 1], [129, 200, 33], [1, 1, 1], [2, 3, 1]]


def ring_pages(rng, num_pages):
    steps = np.array(SCHEDULE)
    rings = [-(-(WIN + int(steps[:, i].max())) // PS) for i in range(steps.shape[1])]
    rings[1] += 1                                    # one ring larger than it must be
    perm = rng.permutation(num_pages).astype(np.int32)
    indptr = np.zeros(len(rings) + 1, np.int64)
    indptr[1:] = np.cumsum(rings)
    return indptr, perm[:indptr[-1]]


@pytest.mark.parametrize("fam", [W.HD256, W.HD512], ids=["hd256", "hd512"])
def test_ring_stream_matches_oracle(fam):
    rng = np.random.Generator(np.random.PCG64(777))
    num_pages = 96
    indptr, page_ids = ring_pages(rng, num_pages)
    start = np.zeros(3, np.int64)
    pool = None
    for k, steps in enumerate(SCHEDULE):
        qo = np.zeros(4, np.int64)
        qo[1:] = np.cumsum(steps)
        b = W.Batch(qo, indptr, page_ids, np.ones(3, np.int32), start.copy(), PS, num_pages)
        fi = W.family_inputs(rng, fam, b, 1, 0, "sentinel", 7)
        run = FamilyRun(fi, pool_bits=pool, rope_rows=4096, ring_window=WIN)
        run.prep()
        run.attn(window_left=WIN)
        assert pg.pg_device_status() == pg.PG_OK
        PT.check_prep(run, fi, initial_pool_bits=pool, ring=True)
        pool = device_to_bits(run.pool)
        q_bits = device_to_bits(run.q_out)
        ref = PT.attn_reference(fi, q_bits, pool, window_left=WIN, ring=True)
        PT.attn_gate(PT.bf16_out(run), ref, f"step {k} {steps}")
        if k == 5:  # a narrower window than the plan's runs on the same plan
            run.attn(window_left=37)
            ref = PT.attn_reference(fi, q_bits, pool, window_left=37, ring=True)
            PT.attn_gate(PT.bf16_out(run), ref, f"step {k}, window 37")
        run.close()
        start += np.array(steps)
    caps = np.diff(indptr) * PS
    assert (start > caps).all()                      # every ring wrapped
    assert start[0] > 2 * caps[0]


def test_ring_plan_bounds_the_attention_window():
    rng = np.random.Generator(np.random.PCG64(5))
    indptr = np.array([0, 8], np.int64)
    b = W.Batch(np.array([0, 20], np.int64), indptr, np.arange(8, dtype=np.int32),
                np.ones(1, np.int32), np.array([500], np.int64), PS, 8)
    fi = W.family_inputs(rng, W.HD256, b, 1, 0, "sentinel", 7)
    run = FamilyRun(fi, rope_rows=4096, ring_window=WIN)
    before = pg.pg_launch_count()
    assert run.attn_status(window_left=WIN + 1) == pg.PG_ERR_WINDOW
    assert run.attn_status(window_left=-1) == pg.PG_ERR_WINDOW
    assert pg.pg_launch_count() == before
    run.close()


def test_ring_plan_lse_matches_oracle():
    # one prefill step past the window through a wrapped ring, with the log-sum-exp output
    D, hq, hkv = 256, 16, 8
    rng = np.random.Generator(np.random.PCG64(91))
    R = -(-(WIN + 40) // PS)
    num_pages = R + 3
    pages = rng.permutation(num_pages)[:R].astype(np.int32)
    pool_bits = W.bf16_normal(rng, (1, num_pages, 2, hkv, PS, D))
    qo, start = np.array([0, 40], np.int64), np.array([700], np.int64)
    indptr = np.array([0, R], np.int64)
    rc, plan = pg.pg_plan_paged_prefill_ring(None, 1, qo, indptr, pages, start, hq, hkv, D, PS, WIN)
    pg.check(rc, "ring plan")
    pool = torch.from_numpy(pool_bits.view(np.int16)).cuda().view(torch.bfloat16)
    q_bits = W.bf16_normal(rng, (40, hq, D))
    q = torch.from_numpy(q_bits.view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.empty_like(q)
    lse = torch.empty(40, hq, dtype=torch.float32, device="cuda")
    pg.check(pg.pg_attn_paged_prefill_lse(plan, pg.pool_descriptor(pool), 0, q, out, lse, WIN, 0.06),
             "attention+lse")
    torch.cuda.synchronize()
    ref_o, ref_l = O.attention(q_bits, pool_bits, 0, qo, indptr, pages, None, start, hkv, WIN, 0.06,
                               ring=True, return_lse=True)
    PT.attn_gate(O.bf16_to_f64(device_to_bits(out)), ref_o, "ring + lse")
    assert np.abs(lse.cpu().numpy() - ref_l).max() <= 1e-2
    plan.close()
