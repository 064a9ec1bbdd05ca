"""Run one call of the path on one named workload a few times, for a profiler.

    python -m paged_sliding_window_qkv_gb300.profile --case prefill-hd512-4096 --iters 3

Each case builds its seeded synthetic inputs, runs the call ``--iters`` times on the current
stream and checks the device status word. Cases:

* ``prefill-hd256-16384``: hd256 attention, one 16384-token request, window_left 1023.
* ``prefill-hd512-4096``: hd512 attention, one 4096-token request, causal.
* ``prep-hd256-16384`` / ``prep-hd512-16384``: the prep call of the 16384-token prefill.
* ``decode-hd256`` / ``decode-hd512``: attention of the 64-request decode step.

The attention cases feed the raw q buffer as the query (its values are N(0,1) bf16, which
is enough for timing); prep writes into a pool of N(0,1) values.
"""
from __future__ import annotations

import argparse
import sys

import torch

from . import pg
from . import workloads as W
from .runner import FamilyRun

CASES = ("prefill-hd256-16384", "prefill-hd512-4096", "prep-hd256-16384", "prep-hd512-16384",
         "decode-hd256", "decode-hd512")


def family_for(case: str):
    if case in ("prefill-hd256-16384", "prep-hd256-16384"):
        return W.make_workload(5, pool_fill="normal").families[0]
    if case == "prep-hd512-16384":
        return W.make_workload(5, pool_fill="normal").families[1]
    if case == "prefill-hd512-4096":
        return W.custom_family(W.HD512, [4096], [0], seed=5, pool_fill="normal", spare_pages=0)
    if case == "decode-hd256":
        return W.make_workload(4).families[0]
    if case == "decode-hd512":
        return W.make_workload(4).families[1]
    raise ValueError(case)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=CASES, required=True)
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)
    run = FamilyRun(family_for(args.case))
    for _ in range(args.iters):
        if args.case.startswith("prep"):
            pg.check(run.prep_status(), "prep")
        elif args.case.startswith("prefill"):
            pg.check(run.attn_status(q=run.q_raw), "attention")
        else:
            pg.check(run.attn_status(), "attention")
    torch.cuda.synchronize()
    status = pg.pg_device_status()
    run.close()
    if status != pg.PG_OK:
        print(f"device status {status}", file=sys.stderr)
        return 1
    print("ok", args.case)
    return 0


if __name__ == "__main__":
    sys.exit(main())
