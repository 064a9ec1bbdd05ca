"""Serving two attention families from allocator-issued pages (include/pg_kv.h) on the GPU.

Requests are admitted step by step in both families' pools; each step's plan inputs come from
the allocator, prep writes K/V into the pages it issued, and attention reads them back. Prep and
attention are checked against the oracle after a prefill step and a decode step, so the
page lists, last-page lengths and start positions the allocator produces are exactly what the
kernels and the oracle agree on. A step is committed only after both families' calls succeeded
("feat(gemma4): paged KV serving across both attention families", review finding "Commit KV
frontiers only after a successful step"); a step refused after admission is aborted and its
retry writes the same span.
"""
import numpy as np
import pytest

import parity as PT
from paged_sliding_window_qkv_gb300 import pg
from paged_sliding_window_qkv_gb300 import workloads as W
from paged_sliding_window_qkv_gb300.runner import FamilyRun, device_to_bits

pytestmark = pytest.mark.gpu

PS = 16
FAMS = {pg.PG_KV_LOCAL: W.HD256, pg.PG_KV_GLOBAL: W.HD512}


def step_inputs(srv, fam_id, rids, steps, num_pages, rng, pool_seed):
    rc, indptr, pages, last, start = pg.pg_kv_batch_plan_inputs(srv, fam_id, rids, steps)
    assert rc == pg.PG_KV_OK
    qo = np.zeros(len(rids) + 1, np.int64)
    qo[1:] = np.cumsum(steps)
    b = W.Batch(qo, indptr, pages, last, start, PS, num_pages)
    return W.family_inputs(rng, FAMS[fam_id], b, 1, 0, "sentinel", pool_seed)


def test_allocator_pages_drive_prep_and_attention():
    num_pages = 24
    rc, srv = pg.pg_kv_server_create(num_pages, num_pages, PS, 1023, 1, 4096)
    assert rc == pg.PG_KV_OK
    rids = [pg.pg_kv_request_open(srv)[1] for _ in range(3)]
    rng = np.random.Generator(np.random.PCG64(2024))
    pools = {}
    for steps in ([37, 20, 16], [1, 1, 1]):            # a prefill step, then a decode step
        for r, n in zip(rids, steps):
            assert pg.pg_kv_admit_step(srv, r, n) == pg.PG_KV_OK
        for fam_id in (pg.PG_KV_LOCAL, pg.PG_KV_GLOBAL):
            fi = step_inputs(srv, fam_id, rids, steps, num_pages, rng, 7)
            before = pools.get(fam_id)
            run = FamilyRun(fi, pool_bits=before, rope_rows=4096)
            run.prep()
            run.attn()
            pools[fam_id] = device_to_bits(run.pool)
            assert pg.pg_device_status() == pg.PG_OK
            PT.check_prep(run, fi, initial_pool_bits=before)
            ref = PT.attn_reference(fi, device_to_bits(run.q_out), pools[fam_id])
            PT.attn_gate(PT.bf16_out(run), ref, f"family {fam_id} steps {steps}")
            run.close()
        for r in rids:
            assert pg.pg_kv_commit_step(srv, r) == pg.PG_KV_OK
    for r in rids:
        assert pg.pg_kv_request_close(srv, r) == pg.PG_KV_OK
    assert pg.pg_kv_free_pages(srv, pg.PG_KV_LOCAL)[1] == num_pages
    pg.pg_kv_server_destroy(srv)


def test_step_refused_after_admission_is_aborted_and_retried():
    # a step whose prep is refused before launch (the rotary tables one row short of its last
    # position) is aborted: the pools' occupancy and the frontier return to their state before
    # admission, the pool bytes are untouched, and the retried step plans the same span and
    # passes the oracle gates in both families
    num_pages = 24
    rope_ok = 4096
    rc, srv = pg.pg_kv_server_create(num_pages, num_pages, PS, 1023, 1, rope_ok)
    assert rc == pg.PG_KV_OK
    rids = [pg.pg_kv_request_open(srv)[1] for _ in range(3)]
    rng = np.random.Generator(np.random.PCG64(2025))
    pools = {}
    for steps in ([37, 20, 16], [1, 1, 1], [5, 9, 2]):
        last_pos = max(pg.pg_kv_request_info(srv, r)[1] + n for r, n in zip(rids, steps)) - 1
        for attempt in ("refused", "retry"):
            free_before = [pg.pg_kv_free_pages(srv, f)[1] for f in (pg.PG_KV_LOCAL, pg.PG_KV_GLOBAL)]
            front_before = [pg.pg_kv_request_info(srv, r)[1] for r in rids]
            for r, n in zip(rids, steps):
                assert pg.pg_kv_admit_step(srv, r, n) == pg.PG_KV_OK
            ok = True
            for fam_id in (pg.PG_KV_LOCAL, pg.PG_KV_GLOBAL):
                fi = step_inputs(srv, fam_id, rids, steps, num_pages, rng, 7)
                before = pools.get(fam_id)
                rope_rows = last_pos if attempt == "refused" else rope_ok
                run = FamilyRun(fi, pool_bits=before, rope_rows=rope_rows)
                launches = pg.pg_launch_count()
                rc = run.prep_status()
                if attempt == "refused":
                    assert rc == pg.PG_ERR_ROPE_RANGE
                    assert pg.pg_launch_count() == launches
                    if before is not None:        # nothing was written into the pool
                        assert np.array_equal(device_to_bits(run.pool), before)
                    ok = False
                    run.close()
                    break
                pg.check(rc, "prep")
                run.attn()
                pools[fam_id] = device_to_bits(run.pool)
                assert pg.pg_device_status() == pg.PG_OK
                PT.check_prep(run, fi, initial_pool_bits=before)
                ref = PT.attn_reference(fi, device_to_bits(run.q_out), pools[fam_id])
                PT.attn_gate(PT.bf16_out(run), ref, f"family {fam_id} steps {steps} retried")
                run.close()
            for r in rids:
                assert (pg.pg_kv_commit_step if ok else pg.pg_kv_abort_step)(srv, r) == pg.PG_KV_OK
            if not ok:
                assert [pg.pg_kv_free_pages(srv, f)[1]
                        for f in (pg.PG_KV_LOCAL, pg.PG_KV_GLOBAL)] == free_before
                assert [pg.pg_kv_request_info(srv, r)[1] for r in rids] == front_before
    for r in rids:
        assert pg.pg_kv_request_close(srv, r) == pg.PG_KV_OK
    pg.pg_kv_server_destroy(srv)


def test_ring_server_pages_carry_the_local_family_past_its_window():
    # the local family on a ring server (window 100, steps of up to 64 tokens: 11-page rings)
    # and the global family growing linearly, stepped until every ring has wrapped
    win, max_step = 100, 64
    pages = {pg.PG_KV_LOCAL: 36, pg.PG_KV_GLOBAL: 64}
    rc, srv = pg.pg_kv_server_create_ring(pages[pg.PG_KV_LOCAL], pages[pg.PG_KV_GLOBAL], PS, win,
                                          max_step, 4096)
    assert rc == pg.PG_KV_OK
    rids = [pg.pg_kv_request_open(srv)[1] for _ in range(3)]
    rng = np.random.Generator(np.random.PCG64(4242))
    pools = {}
    schedule = [[37, 20, 16], [1, 1, 1], [64, 50, 64], [1, 1, 1], [64, 64, 30], [1, 1, 1],
                [64, 1, 64], [1, 1, 1], [64, 64, 64], [64, 64, 64], [1, 1, 1]]
    for steps in schedule:
        for r, n in zip(rids, steps):
            assert pg.pg_kv_admit_step(srv, r, n) == pg.PG_KV_OK
        for fam_id in (pg.PG_KV_LOCAL, pg.PG_KV_GLOBAL):
            ring = fam_id == pg.PG_KV_LOCAL
            fi = step_inputs(srv, fam_id, rids, steps, pages[fam_id], rng, 7)
            before = pools.get(fam_id)
            run = FamilyRun(fi, pool_bits=before, rope_rows=4096, ring_window=win if ring else None)
            run.prep()
            run.attn(window_left=win if ring else None)
            pools[fam_id] = device_to_bits(run.pool)
            assert pg.pg_device_status() == pg.PG_OK
            PT.check_prep(run, fi, initial_pool_bits=before, ring=ring)
            ref = PT.attn_reference(fi, device_to_bits(run.q_out), pools[fam_id],
                                    window_left=win if ring else None, ring=ring)
            PT.attn_gate(PT.bf16_out(run), ref, f"family {fam_id} steps {steps}")
            run.close()
        for r in rids:
            assert pg.pg_kv_commit_step(srv, r) == pg.PG_KV_OK
    f = pg.pg_kv_request_info(srv, rids[0])[1]
    assert f > 2 * 11 * PS                                  # the first request's ring wrapped twice
    for r in rids:
        assert pg.pg_kv_request_close(srv, r) == pg.PG_KV_OK
    pg.pg_kv_server_destroy(srv)
