"""Prep kernels vs the fp64 oracle, through the C ABI (GPU).

q_out and every written K/V row within one bf16 ulp; every other pool row keeps
its initial bytes (sentinel or random fill)."""
import numpy as np
import pytest
import torch

import parity
from paged_sliding_window_qkv_gb300 import workloads as W
from paged_sliding_window_qkv_gb300.runner import FamilyRun

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_prep_matches_oracle_on_config(cfg):
    wl = W.make_workload(cfg)
    for fi in wl.families:
        run = FamilyRun(fi)
        run.prep()
        parity.check_prep(run, fi)
        run.close()


def test_prep_decode_step_on_random_pool():
    # config 4's shape with fewer requests: one new token per request onto existing KV
    for fam, lens in [(W.HD256, (1, 1024)), (W.HD512, (1, 16384))]:
        rng = np.random.Generator(np.random.PCG64(9))
        start = rng.integers(lens[0], lens[1], size=12, endpoint=True)
        fi = W.custom_family(fam, np.ones(12, np.int64), start, seed=91, spare_pages=5,
                             pool_fill="normal")
        init = fi.make_pool()
        run = FamilyRun(fi, pool_bits=init)
        run.prep()
        parity.check_prep(run, fi, initial_pool_bits=init)
        run.close()


@pytest.mark.parametrize("fam", [W.HD256, W.HD512], ids=["hd256", "hd512"])
def test_prep_ragged_with_start_offsets_and_layers(fam):
    # requests continuing from earlier positions, pages split mid-request, 3 layers
    fi = W.custom_family(fam, [1, 15, 16, 17, 40], [0, 3, 16, 31, 100], seed=7, num_layers=3,
                         layer=2, spare_pages=6)
    run = FamilyRun(fi)
    run.prep()
    parity.check_prep(run, fi)
    run.close()


@pytest.mark.parametrize("ps", [1, 8, 32])
def test_prep_other_page_sizes(ps):
    fi = W.custom_family(W.HD256, [5, 33], [2, 0], seed=17, page_size=ps, spare_pages=4)
    run = FamilyRun(fi)
    run.prep()
    parity.check_prep(run, fi)
    run.close()


def test_prep_strided_inputs():
    # raw q/k/v rows taken out of one fused projection buffer: token strides > heads * D
    fi = W.custom_family(W.HD256, [7, 12], [0, 4], seed=23)
    run = FamilyRun(fi)
    T = fi.batch.num_tokens
    fused = torch.empty(T, 16 * 256 + 2 * 8 * 256 + 64, dtype=torch.bfloat16, device="cuda")
    fused[:, :4096] = run.q_raw.view(T, -1)
    fused[:, 4096:6144] = run.k_raw.view(T, -1)
    fused[:, 6144:8192] = run.v_raw.view(T, -1)
    stride = fused.shape[1]
    from paged_sliding_window_qkv_gb300 import pg
    rc = pg.pg_prep_paged_hd256(run.plan, run.pool_desc, 0, fused, stride, fused[:, 4096:],
                                stride, fused[:, 6144:], stride, run.w_q, run.w_k, fi.eps,
                                run.rope_cos, run.rope_sin, run.rope_rows, run.q_out)
    assert rc == pg.PG_OK
    parity.check_prep(run, fi)
    run.close()


def test_prep_is_idempotent_and_deterministic():
    fi = W.custom_family(W.HD512, [30], [0], seed=29)
    run = FamilyRun(fi)
    run.prep()
    torch.cuda.synchronize()
    a, pa = run.q_out.clone(), run.pool.clone()
    run.prep()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), run.q_out.view(torch.int16))
    assert torch.equal(pa.view(torch.int16), run.pool.view(torch.int16))
    run.close()


def test_rope_table_matches_oracle_angles():
    from oracle import oracle as O
    from paged_sliding_window_qkv_gb300 import pg
    rows, D = 20000, 512
    c = torch.empty(rows, D // 2, dtype=torch.float32, device="cuda")
    s = torch.empty_like(c)
    assert pg.pg_rope_table(c, s, rows, D, 1e6) == pg.PG_OK
    rc, rs = O.rope_cos_sin(np.arange(rows), D, 1e6)
    assert np.max(np.abs(c.cpu().numpy() - rc)) < 1e-7
    assert np.max(np.abs(s.cpu().numpy() - rs)) < 1e-7
