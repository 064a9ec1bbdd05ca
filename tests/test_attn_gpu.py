"""Paged attention vs the fp64 oracle, through the C ABI (GPU).

Attention alone: q and a randomly filled pool come from the seeded generator and go
to both sides. End to end: prep then attention on the GPU against the oracle's
prep (rounded to bf16, as the path stores it) followed by the oracle's attention.
Gate: max |err| <= 3e-2, mean |err| <= 3e-3."""
import numpy as np
import pytest
import torch

import parity
from oracle import oracle as O
from paged_sliding_window_qkv_gb300 import workloads as W
from paged_sliding_window_qkv_gb300.runner import FamilyRun, bits_to_device, device_to_bits

pytestmark = pytest.mark.gpu


def _attn_only(fi, window_left=None, rows=None):
    pool = fi.make_pool() if fi.pool_fill == "normal" else W.bf16_normal(
        np.random.Generator(np.random.PCG64(fi.pool_seed)), fi.pool_shape)
    run = FamilyRun(fi, pool_bits=pool)
    run.attn(q=run.q_raw, window_left=window_left)
    gpu = parity.bf16_out(run)
    ref = parity.attn_reference(fi, fi.q_raw, pool, window_left, rows=rows)
    run.close()
    if rows is not None:
        gpu = gpu[rows[:, 0], rows[:, 1]]
    return gpu, ref


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_attention_matches_oracle_on_config(cfg):
    for fi in W.make_workload(cfg).families:
        gpu, ref = _attn_only(fi)
        parity.attn_gate(gpu, ref, f"cfg{cfg} {fi.family.name}")


def test_decode_step_matches_oracle_config4():
    for fi in W.make_workload(4).families:
        gpu, ref = _attn_only(fi)
        parity.attn_gate(gpu, ref, f"cfg4 {fi.family.name}")


@pytest.mark.parametrize("fam", [W.HD256, W.HD512], ids=["hd256", "hd512"])
@pytest.mark.parametrize("window_left", [-1, 0, 1, 15, 16, 63, 100, 5000])
def test_windows_and_ragged_tiles(fam, window_left):
    fi = W.custom_family(fam, [1, 7, 64, 65, 130], [0, 40, 3, 200, 17], seed=31, spare_pages=3,
                         pool_fill="normal", window_left=window_left)
    gpu, ref = _attn_only(fi)
    parity.attn_gate(gpu, ref, f"{fam.name} W={window_left}")


@pytest.mark.parametrize("fam", [W.HD256, W.HD512], ids=["hd256", "hd512"])
@pytest.mark.parametrize("ps", [8, 32, 64])
def test_tensor_core_path_at_other_page_sizes(fam, ps):
    # the tcgen05 path copies one box of min(ps, 32) K rows / min(ps, 64) V rows per page, so
    # page sizes 8, 32 and 64 give 4, 1 and 1 K boxes per lane batch (16 gives 2)
    fi = W.custom_family(fam, [1, 9, 64, 130, 257], [0, 40, 3, 200, 17], seed=41 + ps,
                         page_size=ps, spare_pages=3, pool_fill="normal",
                         window_left=100 if fam is W.HD256 else -1)
    gpu, ref = _attn_only(fi)
    parity.attn_gate(gpu, ref, f"{fam.name} page size {ps}")


def test_window_zero_returns_own_value_on_gpu():
    fi = W.custom_family(W.HD256, [37], [5], seed=37, pool_fill="normal", window_left=0)
    pool = fi.make_pool()
    run = FamilyRun(fi, pool_bits=pool)
    run.attn(q=run.q_raw)
    gpu = parity.bf16_out(run)
    b = fi.batch
    req, pos = O.token_request_and_position(b.qo_indptr, b.start_pos)
    page, slot = O.slot_of(req, pos, b.kv_page_indptr, b.page_ids, b.page_size)
    for t in range(b.num_tokens):
        for h in range(16):
            assert np.array_equal(gpu[t, h], O.bf16_to_f64(pool[0, page[t], 1, h // 2, slot[t]]))
    run.close()


@pytest.mark.parametrize("fam", [W.HD256, W.HD512], ids=["hd256", "hd512"])
def test_decode_chunk_boundaries(fam):
    # kv lengths around the split-KV chunk sizes, windowed and not
    chunk = 256 if fam.head_dim == 256 else 512
    starts = [0, 1, chunk - 1, chunk, chunk + 1, 2 * chunk, 3 * chunk + 5, 5000]
    for w in [-1, 300, 1023]:
        fi = W.custom_family(fam, np.ones(len(starts), np.int64), starts, seed=41,
                             pool_fill="normal", window_left=w)
        gpu, ref = _attn_only(fi)
        parity.attn_gate(gpu, ref, f"{fam.name} decode W={w}")


def test_other_head_groupings():
    for hq, hkv, d in [(8, 8, 256), (16, 4, 256), (16, 16, 512), (8, 1, 512)]:
        fam = W.Family("x", hq, hkv, d, 1e4, 50)
        fi = W.custom_family(fam, [3, 70], [0, 9], seed=43, pool_fill="normal")
        gpu, ref = _attn_only(fi)
        parity.attn_gate(gpu, ref, f"Hq={hq} Hkv={hkv} D={d}")


def test_page_permutation_invariance_on_gpu():
    fi = W.custom_family(W.HD256, [90, 20], [0, 33], seed=47, pool_fill="normal", spare_pages=7)
    pool = fi.make_pool()
    run = FamilyRun(fi, pool_bits=pool)
    run.attn(q=run.q_raw)
    a = run.out.clone()
    perm = np.random.Generator(np.random.PCG64(48)).permutation(fi.batch.num_pages)
    pool2 = np.empty_like(pool)
    pool2[:, perm] = pool
    b = fi.batch
    fi2 = W.FamilyInputs(fi.family, W.Batch(b.qo_indptr, b.kv_page_indptr,
                                            perm[b.page_ids].astype(np.int32), b.last_page_len,
                                            b.start_pos, b.page_size, b.num_pages),
                         fi.num_layers, fi.layer, fi.q_raw, fi.k_raw, fi.v_raw, fi.w_q, fi.w_k,
                         "normal", fi.pool_seed)
    run2 = FamilyRun(fi2, pool_bits=pool2)
    run2.attn(q=run2.q_raw)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), run2.out.view(torch.int16))
    run.close()
    run2.close()


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_end_to_end_prep_then_attention(cfg):
    for fi in W.make_workload(cfg).families:
        run = FamilyRun(fi)
        run.prep()
        run.attn()
        gpu = parity.bf16_out(run)
        qo, ko, vo, offs = parity.prep_reference(fi)
        pool = fi.make_pool()
        flat = pool.reshape(-1, fi.family.head_dim)
        flat[(offs[:, 0] // fi.family.head_dim).ravel()] = O.f64_to_bf16(ko).reshape(-1, fi.family.head_dim)
        flat[(offs[:, 1] // fi.family.head_dim).ravel()] = O.f64_to_bf16(vo).reshape(-1, fi.family.head_dim)
        ref = parity.attn_reference(fi, O.f64_to_bf16(qo), pool)
        parity.attn_gate(gpu, ref, f"cfg{cfg} {fi.family.name} end to end")
        run.close()


def test_full_size_config5_rows():
    # The long 16384-token prefill of both families in the launch the benchmark times, after
    # the prep it times. Prep is gated on every element (one bf16 ulp, untouched pool rows
    # byte-exact). Attention is gated on the oracle's attention over the GPU's own q_out and
    # pool bytes, so its error is not mixed with prep rounding (sm_scale 1.0 leaves the logits
    # unscaled, so a one-ulp prep difference moves a logit by about 0.06): every row of two
    # seeded heads plus every head of 512 seeded tokens (first, last and window-edge tokens
    # among them). The end-to-end error against the oracle's own prep is reported as well.
    wl = W.make_workload(5)
    rng = np.random.Generator(np.random.PCG64(55))
    for fi in wl.families:
        run = FamilyRun(fi)
        run.prep()
        run.attn()
        gpu = parity.bf16_out(run)
        parity.check_prep(run, fi)
        T, Hq = fi.batch.num_tokens, fi.family.num_qo_heads
        heads = rng.choice(Hq, 2, replace=False)
        toks = np.unique(np.concatenate([[0, 1, 63, 64, 127, 128, 1023, 1024, 1025, T - 2, T - 1],
                                         rng.choice(T, 512 - 11, replace=False)]))
        rows = np.concatenate([
            np.stack(np.meshgrid(np.arange(T), heads, indexing="ij"), axis=-1).reshape(-1, 2),
            np.stack(np.meshgrid(toks, np.arange(Hq), indexing="ij"), axis=-1).reshape(-1, 2)])
        rows = np.unique(rows, axis=0)
        ref = parity.attn_reference(fi, device_to_bits(run.q_out), device_to_bits(run.pool),
                                    rows=rows)
        got = gpu[rows[:, 0], rows[:, 1]]
        parity.attn_gate(got, ref, f"cfg5 {fi.family.name}: {len(rows)} rows")
        # end to end from the raw inputs (the oracle's prep feeding the oracle's attention)
        qo, ko, vo, offs = parity.prep_reference(fi)
        pool = fi.make_pool()
        D = fi.family.head_dim
        flat = pool.reshape(-1, D)
        flat[(offs[:, 0] // D).ravel()] = O.f64_to_bf16(ko).reshape(-1, D)
        flat[(offs[:, 1] // D).ravel()] = O.f64_to_bf16(vo).reshape(-1, D)
        sel = rows[rng.choice(len(rows), 4096, replace=False)]
        e2e = np.abs(gpu[sel[:, 0], sel[:, 1]] -
                     parity.attn_reference(fi, O.f64_to_bf16(qo), pool, rows=sel))
        print(f"cfg5 {fi.family.name} end to end (4096 rows): max {e2e.max():.3e} "
              f"mean {e2e.mean():.3e}")
        assert e2e.mean() <= parity.ATTN_MEAN
        run.close()


def test_empty_plan_launches_nothing():
    from paged_sliding_window_qkv_gb300 import pg
    rc, plan = pg.pg_plan_paged_prefill(None, 0, [0], [0], [], [], [], 16, 8, 256, 16)
    assert rc == pg.PG_OK
    pool = torch.zeros(1, 2, 2, 8, 16, 256, dtype=torch.bfloat16, device="cuda")
    before = pg.pg_launch_count()
    assert pg.pg_attn_paged_prefill(plan, pg.pool_descriptor(pool), 0, None, None, -1, 1.0) == pg.PG_OK
    assert pg.pg_launch_count() == before
    plan.close()
