"""C-ABI checks that need no GPU: the library loads, exports every declared symbol,
and rejects bad plans before touching CUDA."""
import glob
import os
import re

import numpy as np
import pytest

import rejects
from paged_sliding_window_qkv_gb300 import pg

INCLUDE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")


def declared_functions():
    names = set()
    for h in sorted(glob.glob(os.path.join(INCLUDE, "*.h"))):
        text = open(h).read()
        names |= set(re.findall(r"^[A-Za-z_][\w \*]*?\b(pg_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ["pg_plan_paged_prefill", "pg_prep_paged_hd256", "pg_prep_paged_hd512",
                     "pg_attn_paged_prefill", "pg_attn_paged_prefill_hd512", "pg_kv_admit_step"]:
        assert required in names


def test_every_declared_symbol_is_exported():
    for name in declared_functions():
        assert hasattr(pg._lib, name), name


def test_status_strings_are_distinct():
    codes = [v for k, v in vars(pg).items() if k.startswith("PG_ERR_") or k == "PG_OK"]
    texts = {pg.pg_status_string(c) for c in codes}
    assert len(texts) == len(codes)
    assert pg.pg_status_string(12345) == "unknown status"


def _plan(a):
    return pg.pg_plan_paged_prefill(None, a["num_req"], a["qo_indptr"], a["kv_page_indptr"],
                                    a["page_ids"], a["last_page_len"], a["start_pos"],
                                    a["num_qo_heads"], a["num_kv_heads"], a["head_dim"],
                                    a["page_size"], stream=0)


PLAN_CASES = [c for c in rejects.load_cases() if c[1] == "plan"]


@pytest.mark.parametrize("name,stage,expected,source", PLAN_CASES, ids=[c[0] for c in PLAN_CASES])
def test_pages_plan_rejects(name, stage, expected, source):
    before = pg.pg_launch_count()
    rc, plan = _plan(rejects.plan_case(name))
    assert rc == getattr(pg, expected), (name, pg.pg_status_string(rc))
    assert plan is None
    assert pg.pg_launch_count() == before


@pytest.mark.parametrize("name", sorted(rejects.PLAN_ONLY_EXTRA))
def test_more_plan_rejects(name):
    a, expected = rejects.plan_extra_case(name)
    rc, plan = _plan(a)
    assert rc == getattr(pg, expected), (name, pg.pg_status_string(rc))
    assert plan is None


def test_decode_plan_past_the_chunked_grid_is_rejected():
    # head_dim 512 decode runs in 512-key chunks, one grid z index each: a request that sees more
    # than 65535 chunks (33,553,921 keys and up) cannot be launched and is refused at plan time
    ps, kv = 12, 65535 * 512 + 1
    npages = -(-kv // ps)
    rc, plan = pg.pg_plan_paged_prefill(None, 1, [0, 1], [0, npages], np.arange(npages, dtype=np.int32),
                                        [kv - (npages - 1) * ps], [kv - 1], 16, 1, 512, ps, stream=0)
    assert rc == pg.PG_ERR_I32_OVERFLOW and plan is None


def test_zero_kv_heads_wins_over_other_faults():
    # the head relation is settled first, before anything could divide by it
    a = rejects.plan_case("zero_kv_heads")
    a["last_page_len"][0] = 999
    a["num_qo_heads"] = 7
    rc, _ = _plan(a)
    assert rc == pg.PG_ERR_ZERO_KV_HEADS


def test_null_plan_is_rejected_everywhere():
    d = pg.pg_pool_t()
    assert pg.pg_prep_paged_hd256(None, d, 0, 0, 0, 0, 0, 0, 0, 0, 0, 1e-6, 0, 0, 1, 0, 0) == pg.PG_ERR_ARG
    assert pg.pg_prep_paged_hd512(None, d, 0, 0, 0, 0, 0, 0, 0, 1e-6, 0, 0, 1, 0, 0) == pg.PG_ERR_ARG
    assert pg.pg_attn_paged_prefill(None, d, 0, 0, 0, -1, 1.0, None, 0, 0) == pg.PG_ERR_ARG
    assert pg.pg_attn_paged_prefill_hd512(None, d, 0, 0, 0, -1, 1.0, None, 0, 0) == pg.PG_ERR_ARG
    assert pg.pg_workspace_bytes(None) == 0
    assert pg.pg_rope_table(0, 0, 4, 256, 1e4, 0) == pg.PG_ERR_ARG


def _ring_plan(pages, qo_len, start, window_left, ps=16):
    return pg.pg_plan_paged_prefill_ring(
        None, 1, np.array([0, qo_len], np.int64), np.array([0, pages], np.int64),
        np.arange(pages, dtype=np.int32), np.array([start], np.int64), 16, 8, 256, ps,
        window_left, stream=0)


def test_ring_plan_rejects_before_touching_cuda():
    # the ring must hold the window plus the step: 8 pages x 16 = 128 >= 100 + 28, not + 29
    before = pg.pg_launch_count()
    assert _ring_plan(8, 29, 5000, 100)[0] == pg.PG_ERR_COVERAGE
    assert _ring_plan(8, 29, 5000, 100)[1] is None
    assert _ring_plan(8, 1, 0, -1)[0] == pg.PG_ERR_WINDOW
    assert _ring_plan(0, 1, 0, 0)[0] == pg.PG_ERR_ARG          # a request with no pages
    assert pg.pg_launch_count() == before


def _segment_plan(kv_start, qo_len=4, start=100, pages=2, last=16):
    return pg.pg_plan_paged_segment(
        None, 1, np.array([0, qo_len], np.int64), np.array([0, pages], np.int64),
        np.arange(pages, dtype=np.int32), np.array([last], np.int32),
        np.array([kv_start], np.int64), np.array([start], np.int64), 16, 8, 256, 16, stream=0)


def test_segment_plan_rejects_before_touching_cuda():
    before = pg.pg_launch_count()
    assert _segment_plan(-1)[0] == pg.PG_ERR_ARG                  # negative segment start
    assert _segment_plan(100, qo_len=4, start=100)[0] == pg.PG_ERR_COVERAGE  # keys past the step
    assert _segment_plan(0, last=17)[0] == pg.PG_ERR_LAST_PAGE_LEN
    assert pg.pg_plan_paged_segment(None, 1, np.array([0, 1], np.int64), np.array([0, 1], np.int64),
                                    np.zeros(1, np.int32), np.ones(1, np.int32), None,
                                    np.array([5], np.int64), 16, 8, 256, 16, stream=0)[0] == pg.PG_ERR_ARG
    assert pg.pg_launch_count() == before


def test_merge_and_lse_entries_reject_bad_arguments():
    before = pg.pg_launch_count()
    assert pg.pg_merge_attn_states(0, 0, 0, 0, 0, 0, 0, 256, stream=0) == pg.PG_OK      # nothing to merge
    assert pg.pg_merge_attn_states(0, 0, 0, 0, 0, 0, -1, 256, stream=0) == pg.PG_ERR_ARG
    assert pg.pg_merge_attn_states(0, 0, 0, 0, 0, 0, 4, 12, stream=0) == pg.PG_ERR_ARG  # head_dim % 8
    assert pg.pg_merge_attn_states(0, 0, 0, 0, 0, 0, 4, 256, stream=0) == pg.PG_ERR_ARG  # null inputs
    assert pg.pg_merge_attn_states(16, 4, 16, 4, 16, 4, 1 << 31, 256, stream=0) == pg.PG_ERR_I32_OVERFLOW
    assert pg.pg_merge_attn_states(16, 4, 24, 4, 16, 4, 4, 256, stream=0) == pg.PG_ERR_ALIGN
    d = pg.pg_pool_t()
    assert pg.pg_attn_paged_prefill_lse(None, d, 0, 0, 0, 0, -1, 1.0, stream=0) == pg.PG_ERR_ARG
    assert pg.pg_attn_paged_prefill_hd512_lse(None, d, 0, 0, 0, 0, -1, 1.0, stream=0) == pg.PG_ERR_ARG
    assert pg.pg_launch_count() == before


def test_ring_plan_accepts_a_ring_that_has_not_wrapped_yet():
    # 2 pages x 16 = 32 slots < window 100 + 20 tokens, but positions 0..19 never wrap: the
    # coverage check passes (the build then needs a GPU for its upload)
    rc = _ring_plan(2, 20, 0, 100)[0]
    assert rc != pg.PG_ERR_COVERAGE
    assert _ring_plan(2, 20, 13, 100)[0] == pg.PG_ERR_COVERAGE   # positions 13..32 wrap


def test_headers_are_plain_c():
    # the boundary is a C ABI: each header compiles as strict C99 on its own
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    for h in sorted(glob.glob(os.path.join(INCLUDE, "*.h"))):
        r = subprocess.run([cc, "-x", "c", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                            "-fsyntax-only", "-"], input=f'#include "{h}"\n', text=True,
                           capture_output=True)
        assert r.returncode == 0, (h, r.stderr)


def test_the_boundary_links_and_runs_from_plain_c(tmp_path):
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    here = os.path.dirname(os.path.abspath(__file__))
    libdir = os.path.dirname(os.path.abspath(pg._lib._name))
    exe = str(tmp_path / "abi_smoke")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", f"-I{INCLUDE}",
                        os.path.join(here, "abi_smoke.c"), "-o", exe, f"-L{libdir}", "-lpg",
                        f"-Wl,-rpath,{libdir}"], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and "c abi ok" in r.stdout, (r.returncode, r.stdout, r.stderr)
