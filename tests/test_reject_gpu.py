"""Launch-stage reject contract and the device-side second layer (GPU).

Each reject returns its status with no kernel launched (library launch counter) and
no caller byte written (pool, q_out and out compared before and after). The device
second layer is exercised by corrupting the plan's device copy of a page id: the
host check (which uses the bounds recorded from the host inputs) passes, the kernel
sees the bad id, skips the access and raises the status word; nothing traps."""
import ctypes as C
import math

import numpy as np
import pytest
import torch

import rejects
from paged_sliding_window_qkv_gb300 import pg
from paged_sliding_window_qkv_gb300 import workloads as W
from paged_sliding_window_qkv_gb300.runner import FamilyRun

pytestmark = pytest.mark.gpu


def _base_run(fam=W.HD256):
    a = rejects.base_plan_args()
    rng = np.random.Generator(np.random.PCG64(4242))
    b = W.make_batch(rng, [20, 9], [0, 5], 16, num_pages=16)
    assert np.array_equal(b.page_ids, a["page_ids"])
    fi = W.family_inputs(rng, fam, b, 1, 0, "sentinel", 1)
    run = FamilyRun(fi)
    run.q_out.fill_(float("nan"))
    run.out.fill_(float("nan"))
    return run


def _snapshot(run):
    torch.cuda.synchronize()
    return [t.view(torch.int16).clone() for t in (run.pool, run.q_out, run.out)]


def _unchanged(run, snap):
    torch.cuda.synchronize()
    return all(torch.equal(t.view(torch.int16), s) for t, s in zip((run.pool, run.q_out, run.out), snap))


def _launch_case(name, run):
    """Returns a list of zero-arg callables giving the statuses for this case."""
    fi = run.fi
    pd = run.pool_desc
    calls = []
    if name == "in_range_control":
        calls = [run.prep_status, run.attn_status]
    elif name in ("page_id_past_pool", "plan_pages_past_pool"):
        # a pool with fewer pages than the plan's largest id
        n = int(fi.batch.page_ids.max()) if name == "page_id_past_pool" else 1
        small = torch.full((1, n, 2, 8, 16, 256), -1, dtype=torch.int16, device="cuda").view(torch.bfloat16)
        run._small = small
        sd = pg.pool_descriptor(small)
        calls = [lambda: _with_pool(run, sd, "prep"), lambda: _with_pool(run, sd, "attn")]
    elif name == "contradictory_layout":
        bad = pg.pool_descriptor(run.pool, stride_head=pd.stride_head + 8)
        calls = [lambda: _with_pool(run, bad, "prep"), lambda: _with_pool(run, bad, "attn")]
    elif name == "partial_page_pool":
        bad = pg.pool_descriptor(run.pool, capacity=pd.capacity - 256)
        calls = [lambda: _with_pool(run, bad, "prep"), lambda: _with_pool(run, bad, "attn")]
    elif name == "layer_out_of_range":
        calls = [lambda: _with_layer(run, 1, "prep"), lambda: _with_layer(run, -1, "attn")]
    elif name == "non_finite_scale":
        calls = [lambda: run.fi.__setattr__("sm_scale", math.inf) or run.attn_status(),
                 lambda: run.fi.__setattr__("sm_scale", math.nan) or run.attn_status(),
                 lambda: run.fi.__setattr__("eps", math.nan) or run.prep_status(),
                 lambda: run.fi.__setattr__("eps", 0.0) or run.prep_status()]
    elif name == "position_past_rope_tables":
        calls = [lambda: pg.pg_prep_paged_hd256(
            run.plan, pd, 0, run.q_raw, 4096, run.k_raw, 2048, run.v_raw, 2048, run.w_q, run.w_k,
            1e-6, run.rope_cos, run.rope_sin, run.rope_rows - 1, run.q_out)]
    elif name == "other_stream":
        s = torch.cuda.Stream()
        run._s = s
        calls = [lambda: _on_stream(run, s, "prep"), lambda: _on_stream(run, s, "attn")]
    else:
        raise KeyError(name)
    return calls


def _with_pool(run, desc, which):
    old = run.pool_desc
    run.pool_desc = desc
    try:
        return run.prep_status() if which == "prep" else run.attn_status()
    finally:
        run.pool_desc = old


def _with_layer(run, layer, which):
    old = run.fi.layer
    run.fi.layer = layer
    try:
        return run.prep_status() if which == "prep" else run.attn_status()
    finally:
        run.fi.layer = old


def _on_stream(run, s, which):
    old = run.stream
    run.stream = s
    try:
        return run.prep_status() if which == "prep" else run.attn_status()
    finally:
        run.stream = old


LAUNCH_CASES = [c for c in rejects.load_cases() if c[1] == "launch"]


@pytest.mark.parametrize("name,stage,expected,source", LAUNCH_CASES,
                         ids=[c[0] for c in LAUNCH_CASES])
def test_launch_rejects(name, stage, expected, source):
    run = _base_run()
    snap = _snapshot(run)
    calls = _launch_case(name, run)
    want = getattr(pg, expected)
    before = pg.pg_launch_count()
    for call in calls:
        rc = call()
        assert rc == want, (name, pg.pg_status_string(rc))
    if want == pg.PG_OK:
        assert pg.pg_launch_count() > before
        assert not _unchanged(run, snap)
        assert pg.pg_device_status() == pg.PG_OK
    else:
        assert pg.pg_launch_count() == before
        assert _unchanged(run, snap)
    run.close()


def test_attention_rejects_bad_window_and_small_workspace():
    run = _base_run()
    # a decode plan needs workspace
    fi = W.custom_family(W.HD512, np.ones(3, np.int64), [600, 3000, 9], seed=3, pool_fill="normal")
    dec = FamilyRun(fi)
    assert dec.ws_bytes > 0
    torch.cuda.synchronize()
    before = pg.pg_launch_count()
    assert run.attn_status(window_left=-2) == pg.PG_ERR_WINDOW
    assert pg.pg_attn_paged_prefill_hd512(dec.plan, dec.pool_desc, 0, dec.q_raw, dec.out, -1, 1.0,
                                          dec.ws, dec.ws_bytes - 4) == pg.PG_ERR_WORKSPACE
    assert pg.pg_attn_paged_prefill_hd512(dec.plan, dec.pool_desc, 0, dec.q_raw, dec.out, -1, 1.0,
                                          None, 0) == pg.PG_ERR_WORKSPACE
    # an hd512 plan on the hd256 entry
    assert pg.pg_attn_paged_prefill(dec.plan, run.pool_desc, 0, dec.q_raw, dec.out, -1, 1.0,
                                    dec.ws, dec.ws_bytes) == pg.PG_ERR_PLAN_MISMATCH
    # misaligned output
    assert pg.pg_attn_paged_prefill(run.plan, run.pool_desc, 0, run.q_out, run.out.data_ptr() + 2,
                                    -1, 1.0) == pg.PG_ERR_ALIGN
    assert pg.pg_launch_count() == before
    run.close()
    dec.close()


def test_failed_plan_update_leaves_plan_intact():
    run = _base_run()
    info0 = run.plan.info()
    a = rejects.plan_case("last_page_len_past_ps")
    rc, _ = pg.pg_plan_paged_prefill(run.plan, a["num_req"], a["qo_indptr"], a["kv_page_indptr"],
                                     a["page_ids"], a["last_page_len"], a["start_pos"], 16, 8,
                                     256, 16)
    assert rc == pg.PG_ERR_LAST_PAGE_LEN
    info1 = run.plan.info()
    for f, _ in pg.pg_plan_info_t._fields_:
        assert getattr(info0, f) == getattr(info1, f), f
    run.prep()
    run.attn()
    assert pg.pg_device_status() == pg.PG_OK
    run.close()


def test_plan_update_in_place_takes_effect():
    run = _base_run()
    rng = np.random.Generator(np.random.PCG64(5))
    b = W.make_batch(rng, [3], [40], 16, num_pages=16)
    rc, _ = pg.pg_plan_paged_prefill(run.plan, b.num_req, b.qo_indptr, b.kv_page_indptr, b.page_ids,
                                     b.last_page_len, b.start_pos, 16, 8, 256, 16)
    assert rc == pg.PG_OK
    i = run.plan.info()
    assert (i.num_req, i.num_tokens, i.max_pos_end) == (1, 3, 43)
    run.close()


def _cudart():
    for name in ("libcudart.so.13", "libcudart.so"):
        try:
            return C.CDLL(name)
        except OSError:
            continue
    pytest.skip("libcudart not loadable by name")


def test_device_second_layer_flags_and_skips_bad_page_ids():
    run = _base_run()
    torch.cuda.synchronize()
    assert pg.pg_device_status() == pg.PG_OK
    # The pool the calls see is the first 16 pages of an allocation of 16 + 8 pages, so the bad
    # id planted below (a spare page) addresses memory this test owns even if a kernel's bounds
    # check ever failed to hold; the spare pages must stay untouched.
    n_pages, spare = run.pool.shape[1], 8
    big = torch.full((1, n_pages + spare) + tuple(run.pool.shape[2:]), -1, dtype=torch.int16,
                     device="cuda").view(torch.bfloat16)
    run.pool = big[:, :n_pages]
    assert run.pool.is_contiguous()
    # one layer: its stride is the dense one, whatever the allocation behind it holds
    run.pool_desc = pg.pool_descriptor(run.pool, stride_layer=run.pool.stride(1) * n_pages)
    assert run.pool_desc.num_pages == n_pages
    info = run.plan.info()
    # corrupt the device copy of the first page id of request 1 (host bounds stay valid)
    first = int(run.fi.batch.kv_page_indptr[1])
    bad = np.array([n_pages + 3], np.int32)
    rt = _cudart()
    rt.cudaMemcpy.argtypes = [C.c_void_p, C.c_void_p, C.c_size_t, C.c_int]
    assert rt.cudaMemcpy(info.d_page_ids + 4 * first, bad.ctypes.data, 4, 1) == 0
    assert run.prep_status() == pg.PG_OK
    assert pg.pg_device_status() == pg.PG_ERR_DEVICE_BOUNDS
    assert pg.pg_device_status() == pg.PG_OK   # read-and-clear
    torch.cuda.synchronize()
    assert run.attn_status() == pg.PG_OK
    assert pg.pg_device_status() == pg.PG_ERR_DEVICE_BOUNDS
    assert torch.isfinite(run.out[:20].float()).all()   # request 0 unaffected
    torch.cuda.synchronize()
    assert bool((big[:, n_pages:].view(torch.int16) == -1).all())   # spare pages untouched
    run.close()


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    # Failure detection without a GPU fault: the test hook makes the leading CTA of each pair
    # withhold its first key-tile arrival (no copy is issued for it), so the QK issuer's wait
    # on that slot can never complete; with a 50 ms limit every role of both CTAs gives up,
    # the pair drains, frees its tensor memory and returns, and the status word reports the
    # timeout. A later call with the hook off is checked against the oracle.
    import parity as PT
    from oracle import oracle as O
    from paged_sliding_window_qkv_gb300.runner import device_to_bits
    for fam, n in ((W.HD256, 512), (W.HD512, 256)):
        fi = W.custom_family(fam, [n], [0], seed=31, pool_fill="normal")
        run = FamilyRun(fi)
        torch.cuda.synchronize()
        assert pg.pg_device_status() == pg.PG_OK
        try:
            assert pg.pg_test_bounded_wait(1, 50_000_000) == pg.PG_OK
            assert run.attn_status(q=run.q_raw) == pg.PG_OK
            assert pg.pg_device_status() == pg.PG_ERR_DEVICE_TIMEOUT
        finally:
            assert pg.pg_test_bounded_wait(0) == pg.PG_OK
        assert pg.pg_device_status() == pg.PG_OK
        run.attn(q=run.q_raw)
        torch.cuda.synchronize()
        assert pg.pg_device_status() == pg.PG_OK
        ref = PT.attn_reference(fi, fi.q_raw, device_to_bits(run.pool),
                                rows=np.array([[t, h] for t in (0, n // 2, n - 1) for h in range(16)]))
        got = PT.bf16_out(run)
        rows = [(t, h) for t in (0, n // 2, n - 1) for h in range(16)]
        PT.attn_gate(np.stack([got[t, h] for t, h in rows]), ref, f"{fam.name} after a timeout")
        run.close()
    assert pg.pg_test_bounded_wait(2, 50_000_000) == pg.PG_ERR_ARG
    assert pg.pg_test_bounded_wait(1, 10) == pg.PG_ERR_ARG


def test_ring_and_segment_plans_update_in_place_and_survive_a_failed_update():
    pages = np.arange(9, dtype=np.int32)
    geo = (16, 8, 256, 16)
    rc, plan = pg.pg_plan_paged_prefill_ring(None, 1, [0, 10], [0, 9], pages, [0], *geo, 100)
    assert rc == pg.PG_OK
    rc, _ = pg.pg_plan_paged_prefill_ring(plan, 1, [0, 40], [0, 9], pages, [700], *geo, 100)
    assert rc == pg.PG_OK
    i = plan.info()
    assert (i.num_tokens, i.max_pos_end) == (40, 740)
    # 9 x 16 = 144 slots < window 100 + 60 tokens, and positions wrap: refused, plan unchanged
    rc, _ = pg.pg_plan_paged_prefill_ring(plan, 1, [0, 60], [0, 9], pages, [700], *geo, 100)
    assert rc == pg.PG_ERR_COVERAGE
    assert (plan.info().num_tokens, plan.info().max_pos_end) == (40, 740)
    plan.close()
    rc, seg = pg.pg_plan_paged_segment(None, 1, [0, 4], [0, 2], [3, 5], [16], [100], [128], *geo)
    assert rc == pg.PG_OK
    rc, _ = pg.pg_plan_paged_segment(seg, 1, [0, 4], [0, 2], [3, 5], [16], [172], [200], *geo)
    assert rc == pg.PG_OK and seg.info().max_pos_end == 204
    # keys [200, 232) would run past the step's last position 203: refused, plan unchanged
    rc, _ = pg.pg_plan_paged_segment(seg, 1, [0, 4], [0, 2], [3, 5], [16], [200], [200], *geo)
    assert rc == pg.PG_ERR_COVERAGE
    assert seg.info().max_pos_end == 204
    seg.close()
