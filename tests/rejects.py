"""The reject contract of ``tests/golden/reject_cases.txt`` as runnable cases.

``plan_case(name)`` returns keyword arguments for ``pg_plan_paged_prefill``;
``launch_case(name, run)`` mutates the arguments of one prep or attention call of
a ``FamilyRun`` and returns (callable, which-entry). Both are plain host logic.
"""
from __future__ import annotations

import os

import numpy as np

from paged_sliding_window_qkv_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "reject_cases.txt")


def load_cases():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, stage, expected, source = [c.strip() for c in line.split("|")]
        rows.append((name, stage, expected, source))
    return rows


def base_plan_args(page_size=16):
    """A valid 2-request hd256 plan over a 16-page pool."""
    rng = np.random.Generator(np.random.PCG64(4242))
    b = W.make_batch(rng, [20, 9], [0, 5], page_size, num_pages=16)
    return dict(num_req=b.num_req, qo_indptr=b.qo_indptr.copy(),
                kv_page_indptr=b.kv_page_indptr.copy(), page_ids=b.page_ids.copy(),
                last_page_len=b.last_page_len.copy(), start_pos=b.start_pos.copy(),
                num_qo_heads=16, num_kv_heads=8, head_dim=256, page_size=page_size)


def plan_case(name):
    a = base_plan_args()
    if name == "last_page_len_past_ps":
        a["last_page_len"][0] = a["page_size"] + 1
    elif name == "batch_length_past_i32":
        # qo_len of 2^32 + 20 would truncate to the legal-looking 20 in int32
        a["qo_indptr"] = a["qo_indptr"] + np.array([0, 1 << 32, 1 << 32])
        a["start_pos"][0] = 0
    elif name == "zero_kv_heads":
        a["num_kv_heads"] = 0
    elif name == "page_coverage_short":
        a["start_pos"][1] += 16  # positions run past the pages held
    else:
        raise KeyError(name)
    return a


PLAN_ONLY_EXTRA = {
    # further plan-time rejects not listed on the pages but implied by the same checks
    "heads_not_multiple": (dict(num_qo_heads=12, num_kv_heads=8), "PG_ERR_HEADS"),
    "last_page_len_zero": (dict(last_page_len=np.array([0, 14], np.int32)), "PG_ERR_LAST_PAGE_LEN"),
    "negative_page_id": (dict(page_ids=None), "PG_ERR_PAGE_OOB"),
    "empty_request": (dict(qo_indptr=np.array([0, 0, 9])), "PG_ERR_ARG"),
    "negative_start": (dict(start_pos=np.array([-1, 5])), "PG_ERR_ARG"),
    "start_past_i32": (dict(start_pos=np.array([0, (1 << 31) - 5])), "PG_ERR_I32_OVERFLOW"),
}


def plan_extra_case(name):
    a = base_plan_args()
    over, expected = PLAN_ONLY_EXTRA[name]
    for k, v in over.items():
        if k == "page_ids":
            a["page_ids"] = a["page_ids"].copy()
            a["page_ids"][1] = -3
        else:
            a[k] = v
    return a, expected
