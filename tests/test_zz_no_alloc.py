"""Decode attention without allocation, through the C ABI (GPU).

pg_attn_paged_decode_noalloc serves callers that may not allocate device memory at call
time (for example under an allocator that forbids cudaMalloc once serving has started);
it keeps its split-KV partials in a static scratch buffer inside the library. These
tests compare it with the fp64 oracle and with the workspace entry points on the same
decode plans, twice in a row with different windows so the second call runs over the
first call's leftovers, and check its size limit. This file is named to be collected
last."""
import numpy as np
import pytest
import torch

import parity
from oracle import oracle as O
from paged_sliding_window_qkv_gb300 import pg
from paged_sliding_window_qkv_gb300 import workloads as W
from paged_sliding_window_qkv_gb300.runner import FamilyRun, device_to_bits

pytestmark = pytest.mark.gpu


def _bits64(t):
    torch.cuda.synchronize()
    return O.bf16_to_f64(device_to_bits(t))


@pytest.mark.parametrize("fam", [W.HD256, W.HD512], ids=["hd256", "hd512"])
def test_noalloc_decode_matches_workspace_entry_on_two_calls(fam):
    rng = np.random.Generator(np.random.PCG64(77))
    hi = 1024 if fam.head_dim == 256 else 6000
    starts = rng.integers(1, hi, size=24, endpoint=True)
    starts[:3] = [1, 600, hi]
    fi = W.custom_family(fam, np.ones(24, np.int64), starts, seed=78, pool_fill="normal")
    run = FamilyRun(fi)
    assert 0 < run.ws_bytes <= pg.PG_NOALLOC_SCRATCH_BYTES
    windows = [fam.window_left, 300]
    for w in windows:
        run.attn(q=run.q_raw, window_left=w)
        ref = _bits64(run.out)
        got = torch.full_like(run.out, float("nan"))
        rc = pg.pg_attn_paged_decode_noalloc(run.plan, run.pool_desc, fi.layer, run.q_raw, got,
                                             w, fi.sm_scale)
        assert rc == pg.PG_OK, pg.pg_status_string(rc)
        oracle = parity.attn_reference(fi, fi.q_raw, device_to_bits(run.pool), window_left=w)
        parity.attn_gate(_bits64(got), oracle, f"{fam.name} no-alloc decode vs oracle, window {w}")
        parity.attn_gate(_bits64(got), ref, f"{fam.name} no-alloc decode, window {w}")
    assert pg.pg_device_status() == pg.PG_OK
    run.close()


def test_noalloc_rejects_oversized_and_prefill_plans():
    # a decode plan whose partials need more than the static scratch holds: at page size 12 the
    # decode runs in fixed key chunks with one partial per (request, head, chunk)
    R, kv = 64, 16384
    rng = np.random.Generator(np.random.PCG64(79))
    b = W.make_batch(rng, np.ones(R, np.int64), np.full(R, kv - 1), 12)
    rc, plan = pg.pg_plan_paged_prefill(None, R, b.qo_indptr, b.kv_page_indptr, b.page_ids,
                                        b.last_page_len, b.start_pos, 16, 1, 512, 12)
    assert rc == pg.PG_OK
    assert pg.pg_workspace_bytes(plan) > pg.PG_NOALLOC_SCRATCH_BYTES
    small = torch.zeros(1, 4, 2, 1, 16, 512, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(R, 16, 512, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    before = pg.pg_launch_count()
    assert pg.pg_attn_paged_decode_noalloc(plan, pg.pool_descriptor(small), 0, q, out, -1,
                                           1.0) == pg.PG_ERR_WORKSPACE
    assert pg.pg_launch_count() == before
    plan.close()
    # a prefill plan is not this entry's form
    fi = W.custom_family(W.HD256, [5, 9], [0, 3], seed=80)
    run = FamilyRun(fi)
    torch.cuda.synchronize()
    before = pg.pg_launch_count()
    assert pg.pg_attn_paged_decode_noalloc(run.plan, run.pool_desc, 0, run.q_raw, run.out, -1,
                                           1.0) == pg.PG_ERR_PLAN_MISMATCH
    assert pg.pg_launch_count() == before
    run.close()
