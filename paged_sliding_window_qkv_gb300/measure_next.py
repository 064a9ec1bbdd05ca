"""Throughput of the calls beyond the single prefill/decode step, on seeded synthetic inputs.

    python -m paged_sliding_window_qkv_gb300.measure_next [--case NAME] [--iters 20]

Prints one JSON line per case: CUDA-event time per call (inputs resident, L2 flushed between
calls by a 512 MiB write), the algorithmic bytes or FLOP of the call and the fraction of the
measured peak. Attention here only reads the pool, so the pools hold N(0,1) bf16 written
directly (no prep), and the queries are N(0,1) bf16. Cases:

* ``merge``: merging two attention states of 16384 tokens x 16 heads at head_dim 512
  (pg_merge_attn_states); bytes = rows x (3 x 512 x 2 + 12).
* ``cascade-decode-hd512``: one decode step of 64 requests that share an 8192-token prefix and
  hold U[1, 1024] tokens of their own, full causal: the single pass over each request's own copy
  of all its keys, against the cascade (the shared prefix as one key segment listed for every
  request, the own keys as another, and the merge). Bytes are the single pass's K/V reads.
* ``ring-decode-hd256``: one decode step of 64 requests at positions U[4096, 32768) holding only
  a ring of ceil((window + 1) / 16) + 1 pages, window_left 1023, against the same window on
  linear pages; bytes = visible keys x 8 heads x 256 x 2 x 2.
* ``ring-prefill-hd256``: a 4096-token chunk at position 65536 of one request on a ring of
  ceil((window + 4096) / 16) + 1 pages, window_left 1023, against the same chunk on linear pages; FLOP = 4 x 256 x 16 x visible pairs.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np
import torch

from . import pg

CASES = ("merge", "cascade-decode-hd512", "ring-decode-hd256", "ring-prefill-hd256")
FLUSH_BYTES = 512 << 20


def peaks():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    try:
        d = json.load(open(os.path.join(root, "MEASURED_PEAKS.json")))
        hbm = float(d.get("hbm_gbs") or d.get("hbm", {}).get("gbs"))
        bf16 = float(d.get("bf16_tflops") or d.get("bf16", {}).get("tflops"))
        return hbm, bf16, "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def timed(fn, iters, flush):
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(iters)]
    for a, b in ev:
        flush.zero_()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return float(np.median([a.elapsed_time(b) for a, b in ev]))


def randn_bf16(shape, gen):
    return torch.randn(shape, generator=gen, device="cuda", dtype=torch.bfloat16)


class Attn:
    """One attention call on a plan over a pool, with its output and workspace."""

    def __init__(self, plan, pool, q, D, window, lse=False):
        self.plan, self.pool, self.q, self.D, self.window = plan, pool, q, D, window
        self.desc = pg.pool_descriptor(pool)
        self.out = torch.empty_like(q)
        self.lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device="cuda") if lse else None
        self.wsb = pg.pg_workspace_bytes(plan)
        self.ws = torch.empty(self.wsb, dtype=torch.uint8, device="cuda") if self.wsb else None

    def __call__(self):
        if self.lse is None:
            fn = pg.pg_attn_paged_prefill if self.D == 256 else pg.pg_attn_paged_prefill_hd512
            rc = fn(self.plan, self.desc, 0, self.q, self.out, self.window, 1.0, self.ws, self.wsb)
        else:
            fn = pg.pg_attn_paged_prefill_lse if self.D == 256 else pg.pg_attn_paged_prefill_hd512_lse
            rc = fn(self.plan, self.desc, 0, self.q, self.out, self.lse, self.window, 1.0, self.ws,
                    self.wsb)
        pg.check(rc, "attention")


def table(lens, ps, first_page):
    """Page table (indptr, ids, last_page_len) for runs of the given lengths on consecutive
    page ids from first_page (the ids are permuted by the caller)."""
    lens = np.asarray(lens, np.int64)
    n = -(-lens // ps)
    indptr = np.zeros(len(lens) + 1, np.int64)
    indptr[1:] = np.cumsum(n)
    ids = np.arange(first_page, first_page + indptr[-1], dtype=np.int64)
    last = (lens - (n - 1) * ps).astype(np.int32)
    return indptr, ids, last


def case_merge(iters, flush, hbm):
    gen = torch.Generator(device="cuda").manual_seed(1)
    rows, D = 16384 * 16, 512
    oa, ob = randn_bf16((rows, D), gen), randn_bf16((rows, D), gen)
    la = torch.randn(rows, generator=gen, device="cuda") * 4
    lb = torch.randn(rows, generator=gen, device="cuda") * 4
    o = torch.empty_like(oa)
    lo = torch.empty_like(la)
    ms = timed(lambda: pg.check(pg.pg_merge_attn_states(oa, la, ob, lb, o, lo, rows, D), "merge"),
               iters, flush)
    nbytes = rows * (3 * D * 2 + 12)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"case": "merge", "rows": rows, "head_dim": D, "ms": ms, "bytes": nbytes,
            "GB/s": gbs, "frac_hbm": gbs / hbm}


def case_cascade(iters, flush, hbm):
    rng = np.random.Generator(np.random.PCG64(11))
    R, P, ps, hq, hkv, D = 64, 8192, 16, 16, 1, 512
    own = rng.integers(1, 1025, R)
    L = P + own
    one = np.arange(R + 1, dtype=np.int64)
    start = (L - 1).astype(np.int64)
    # page ids: full copies, then the shared prefix, then the own runs; permuted over the pool
    f_ip, f_ids, f_last = table(L, ps, 0)
    n_pre = -(-P // ps)
    p_ids = np.arange(f_ids.size, f_ids.size + n_pre)
    s_ip, s_ids, s_last = table(own, ps, f_ids.size + n_pre)
    total = int(s_ids[-1]) + 1
    perm = rng.permutation(total).astype(np.int32)
    gen = torch.Generator(device="cuda").manual_seed(2)
    pool = randn_bf16((1, total, 2, hkv, ps, D), gen)
    q = randn_bf16((R, hq, D), gen)

    def plan(ip, ids, last, kv_start=None):
        if kv_start is None:
            rc, pl = pg.pg_plan_paged_prefill(None, R, one, ip, perm[ids], last, start, hq, hkv, D, ps)
        else:
            rc, pl = pg.pg_plan_paged_segment(None, R, one, ip, perm[ids], last, kv_start, start,
                                              hq, hkv, D, ps)
        pg.check(rc, "plan")
        return pl

    full = Attn(plan(f_ip, f_ids, f_last), pool, q, D, -1)
    pre_ip = np.arange(R + 1, dtype=np.int64) * n_pre
    pre = Attn(plan(pre_ip, np.tile(p_ids, R), np.full(R, P - (n_pre - 1) * ps, np.int32),
                    np.zeros(R, np.int64)), pool, q, D, -1, lse=True)
    suf = Attn(plan(s_ip, s_ids, s_last, np.full(R, P, np.int64)), pool, q, D, -1, lse=True)
    out = torch.empty_like(q)
    lse = torch.empty(R, hq, dtype=torch.float32, device="cuda")

    def cascade():
        pre()
        suf()
        pg.check(pg.pg_merge_attn_states(pre.out, pre.lse, suf.out, suf.lse, out, lse, R * hq, D),
                 "merge")

    t_full = timed(full, iters, flush)
    t_cas = timed(cascade, iters, flush)
    nbytes = int(L.sum()) * hkv * D * 2 * 2 + 2 * R * hq * D * 2
    return {"case": "cascade-decode-hd512", "requests": R, "shared_prefix": P,
            "own_tokens": "U[1,1024]", "single_pass_ms": t_full, "cascade_ms": t_cas,
            "speedup": t_full / t_cas, "single_pass_bytes": nbytes,
            "single_pass_GB/s": nbytes / (t_full * 1e-3) / 1e9,
            "single_pass_frac_hbm": nbytes / (t_full * 1e-3) / 1e9 / hbm,
            "cascade_effective_GB/s": nbytes / (t_cas * 1e-3) / 1e9}


def ring_vs_linear(name, starts, qo_lens, window, hq, hkv, D, ps, iters, flush, work, unit):
    R = len(starts)
    qo = np.zeros(R + 1, np.int64)
    qo[1:] = np.cumsum(qo_lens)
    starts = np.asarray(starts, np.int64)
    ring_pages = -(-(window + np.asarray(qo_lens)) // ps) + 1
    r_ip = np.zeros(R + 1, np.int64)
    r_ip[1:] = np.cumsum(ring_pages)
    L = starts + np.asarray(qo_lens)
    l_ip, l_ids, l_last = table(L, ps, int(r_ip[-1]))
    total = int(l_ids[-1]) + 1
    rng = np.random.Generator(np.random.PCG64(13))
    perm = rng.permutation(total).astype(np.int32)
    gen = torch.Generator(device="cuda").manual_seed(3)
    pool = randn_bf16((1, total, 2, hkv, ps, D), gen)
    q = randn_bf16((int(qo[-1]), hq, D), gen)
    rc, ring = pg.pg_plan_paged_prefill_ring(None, R, qo, r_ip, perm[:r_ip[-1]], starts, hq, hkv,
                                             D, ps, window)
    pg.check(rc, "ring plan")
    rc, lin = pg.pg_plan_paged_prefill(None, R, qo, l_ip, perm[l_ids], l_last, starts, hq, hkv, D, ps)
    pg.check(rc, "linear plan")
    t_ring = timed(Attn(ring, pool, q, D, window), iters, flush)
    t_lin = timed(Attn(lin, pool, q, D, window), iters, flush)
    res = {"case": name, "requests": R, "window_left": window, "ring_ms": t_ring,
           "linear_ms": t_lin, "work": work, "unit": unit,
           "ring_rate": work / (t_ring * 1e-3) / (1e9 if unit == "B" else 1e12),
           "linear_rate": work / (t_lin * 1e-3) / (1e9 if unit == "B" else 1e12)}
    return res


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=CASES + ("all",), default="all")
    ap.add_argument("--iters", type=int, default=20)
    args = ap.parse_args(argv)
    hbm, bf16, src = peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    todo = CASES if args.case == "all" else (args.case,)
    for c in todo:
        if c == "merge":
            res = case_merge(args.iters, flush, hbm)
        elif c == "cascade-decode-hd512":
            res = case_cascade(args.iters, flush, hbm)
        elif c == "ring-decode-hd256":
            rng = np.random.Generator(np.random.PCG64(17))
            starts = rng.integers(4096, 32768, 64)
            work = 64 * 1024 * 8 * 256 * 2 * 2
            res = ring_vs_linear(c, starts, [1] * 64, 1023, 16, 8, 256, 16, args.iters, flush,
                                 work, "B")
            res["frac_hbm_ring"] = res["ring_rate"] / hbm
        else:
            pairs = sum(min(p + 1, 1024) for p in range(65536, 65536 + 4096))
            res = ring_vs_linear(c, [65536], [4096], 1023, 16, 8, 256, 16, args.iters, flush,
                                 4.0 * 256 * 16 * pairs, "FLOP")
            res["frac_bf16_ring"] = res["ring_rate"] / bf16
        res["peaks"] = src
        print(json.dumps(res), flush=True)
    if pg.pg_device_status() != pg.PG_OK:
        print("device status not OK", file=sys.stderr)
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
