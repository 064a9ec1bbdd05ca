"""The decode step of both families captured in one CUDA graph.

The pages leave the decode form's launch shape open ("measurement-gated"); a serving loop
replays the whole step (prep + attention of both families) as one graph. The entry points make
no allocation, synchronisation or host read on the stream once each kernel has been launched
once, so the step can be captured. The replay is gated against the oracle (prep: q_out and the
pool rows within one bf16 ulp, every other pool row byte-exact; attention: the oracle's
attention over the replayed pool and q_out) and must also reproduce the eager step bit for bit.
"""
import numpy as np
import pytest
import torch

import parity as PT

from paged_sliding_window_qkv_gb300 import pg
from paged_sliding_window_qkv_gb300 import workloads as W
from paged_sliding_window_qkv_gb300.runner import FamilyRun, device_to_bits

pytestmark = pytest.mark.gpu


def test_decode_step_replays_as_one_graph():
    s = torch.cuda.Stream()
    wl = W.make_workload(4)
    with torch.cuda.stream(s):
        runs = [FamilyRun(fi, stream=s) for fi in wl.families]

        def step():
            for r in runs:
                pg.check(r.prep_status(), "prep")
                pg.check(r.attn_status(), "attention")

        step()  # eager: configures every kernel once
        s.synchronize()
        eager_out = [device_to_bits(r.out) for r in runs]
        eager_pool = [device_to_bits(r.pool) for r in runs]
        for r in runs:
            r.out.zero_()
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        before = pg.pg_launch_count()
        with torch.cuda.graph(g, stream=s):
            step()
        launched = pg.pg_launch_count() - before
        g.replay()
        s.synchronize()
    assert launched == 6        # two preps, two split-KV attentions, two merges
    assert pg.pg_device_status() == pg.PG_OK
    for r, fi in zip(runs, wl.families):
        PT.check_prep(r, fi, initial_pool_bits=fi.make_pool())
        ref = PT.attn_reference(fi, device_to_bits(r.q_out), device_to_bits(r.pool))
        PT.attn_gate(PT.bf16_out(r), ref, f"graph replay {fi.family.name}")
    for r, o, p in zip(runs, eager_out, eager_pool):
        assert np.array_equal(device_to_bits(r.out), o)
        assert np.array_equal(device_to_bits(r.pool), p)
    # replays are cheaper than eager steps (printed, not asserted: shared GPUs vary)
    e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    with torch.cuda.stream(s):
        e[0].record(s)
        for _ in range(20):
            step()
        e[1].record(s)
        e[2].record(s)
        for _ in range(20):
            g.replay()
        e[3].record(s)
    s.synchronize()
    print(f"decode step: eager {e[0].elapsed_time(e[1]) / 20 * 1e3:.1f} us, "
          f"graph {e[2].elapsed_time(e[3]) / 20 * 1e3:.1f} us")
    for r in runs:
        r.close()
