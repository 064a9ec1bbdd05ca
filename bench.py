"""Benchmark of the paged two-family prep + attention hot path on GB300.

One step is one mixed serving step over both attention families, one layer each:
  * prefill of one 16384-token request (config 5): hd256 prep + windowed attention
    (window_left 1023) and hd512 prep + full causal attention;
  * a decode step of 64 requests, one new token each, on existing KV of U[1,1024]
    (hd256, window_left 1023) and U[1,16384] (hd512) tokens (config 4): prep +
    split-KV attention + merge.
Inputs are seeded synthetic bf16 N(0,1) (no dataset on the pages), resident in HBM
before the timed region; L2 is flushed (a 512 MiB write) between timed steps.

value: effective attention TFLOP/s of the whole step, 4*D*Hq*(visible query-key
pairs) summed over the step's attention calls / step time. Per-kernel throughput
(prep and decode GB/s, prefill TFLOP/s) is reported under "kernels", each as a fraction of
the measured peaks (frac_measured: MEASURED_PEAKS.json's HBM copy rate and burst bf16 GEMM
rate, since every call runs for milliseconds at most) and of the nominal ones the targets are
stated against (frac_nominal: 8 TB/s HBM, 2.25 PFLOP/s dense bf16). Outside the timed step:
the batched ragged prefill (8 requests of 128-2048 tokens, 4 layers of 8192 pages) and the
decode step replayed as one CUDA graph.

--impl reference times the fp64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attn effective TFLOP/s (% BF16 peak); prep & decode HBM GB/s (% of 8 TB/s)"
WORKLOAD = ("mixed serving step, one layer per family: 16384-token prefill (hd256 window_left "
            "1023 + hd512 full causal) and 64-request decode (existing KV U[1,1024] hd256, "
            "U[1,16384] hd512)")
L2_FLUSH_BYTES = 512 << 20


NOMINAL_HBM_GBS = 8000.0       # HBM3e, nominal
NOMINAL_BF16_TFLOPS = 2250.0   # dense bf16 tensor rate, nominal


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sustained=d["bf16_tflops_sustained"], src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


def rate_entry(ms, work, kind, peaks):
    """Per-call throughput: kind "hbm" (work in bytes) or "tensor" (work in FLOP), as achieved
    rate and as fractions of the measured burst peak and of the nominal peak."""
    if kind == "hbm":
        gbs = work / (ms * 1e-3) / 1e9
        return {"ms": ms, "GB/s": gbs, "bytes": work, "frac_measured": gbs / peaks["hbm"],
                "frac_nominal": gbs / NOMINAL_HBM_GBS}
    tf = work / (ms * 1e-3) / 1e12
    return {"ms": ms, "TFLOP/s": tf, "flops": work, "frac_measured": tf / peaks["bf16"],
            "frac_nominal": tf / NOMINAL_BF16_TFLOPS}


# ---------------------------------------------------------------------------- work model
def visible_pairs(batch, window_left):
    """Query-key pairs the mask keeps, per query head."""
    lens = np.diff(batch.qo_indptr)
    tot = 0
    for r in range(batch.num_req):
        p = batch.start_pos[r] + np.arange(lens[r], dtype=np.int64)
        n = p + 1
        if window_left >= 0:
            n = np.minimum(n, window_left + 1)
        tot += int(n.sum())
    return tot


def attn_flops(fi):
    f = fi.family
    return 4.0 * f.head_dim * f.num_qo_heads * visible_pairs(fi.batch, f.window_left)


def prep_bytes(fi):
    """Algorithmic HBM bytes of one prep call: raw rows in, q_out and K/V rows out,
    one rotary row (cos + sin) and the token's request index per token."""
    f, T = fi.family, fi.batch.num_tokens
    D, Hq, Hkv = f.head_dim, f.num_qo_heads, f.num_kv_heads
    n_in = Hq + (2 * Hkv if D == 256 else Hkv)
    n_out = Hq + 2 * Hkv
    return T * ((n_in + n_out) * D * 2 + D * 4 + 4)


def decode_bytes(fi):
    """Algorithmic HBM bytes of one decode attention call: every visible K and V row
    once, q in, out written, and the page ids of the visible keys."""
    f, b = fi.family, fi.batch
    D, Hq, Hkv = f.head_dim, f.num_qo_heads, f.num_kv_heads
    vis = visible_pairs(b, f.window_left)
    return (vis * Hkv * D * 2 * 2 + b.num_req * Hq * D * 2 * 2
            + (vis // b.page_size + b.num_req) * 4)


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock and throttle samples every 100 ms; only the samples taken inside the
    timed window (mark_start / mark_stop, host time) are summarised. The raw CSV goes to
    $PG_CLOCK_LOG (a directory) when set, else to a temporary file."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        import tempfile
        self.proc = None
        log_dir = os.environ.get("PG_CLOCK_LOG")
        self.keep = bool(log_dir)
        if log_dir:
            self.path = os.path.join(log_dir, f"clocks_rank{device_index}.csv")
        else:
            self.path = os.path.join(tempfile.gettempdir(), f"pg_clocks_{os.getpid()}_{device_index}.csv")
        self.dev = device_index
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", "100"]
            uuid = None
            try:
                import torch
                uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            except Exception:
                pass
            if uuid:
                cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        import datetime
        rows = []
        with open(self.path) as f:
            lines = f.readlines()
        if not self.keep:
            try:
                os.remove(self.path)
            except OSError:
                pass
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t1 is not None
                  and self.t0 <= r[0] <= self.t1]
        window = "timed region"
        if not inside:  # a window shorter than the sampling period: the nearest samples
            inside, window = rows, "around the timed region"
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, _, fl in inside for i, v in enumerate(fl)
                          if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": inside[0][2],
                "reasons": reasons, "samples": len(inside), "window": window}


# ---------------------------------------------------------------------------- oracle leg
_ORACLE_DATA = None


def _oracle_data():
    """Workload families and their (randomly filled) pools for the oracle leg, built once."""
    global _ORACLE_DATA
    if _ORACLE_DATA is None:
        from paged_sliding_window_qkv_gb300 import workloads as W
        fams = W.make_workload(5, pool_fill="normal").families + W.make_workload(4).families
        _ORACLE_DATA = [(fi, fi.make_pool()) for fi in fams]
    return _ORACLE_DATA


def oracle_sample(seconds: float, seed: int = 7):
    """Time the fp64 oracle (as it stands) on sampled rows of the same workload:
    attention rows of the prefill and decode batches of both families plus the prep of
    the sampled tokens. Returns (effective attention FLOPs, seconds, description)."""
    from oracle import oracle as O
    rng = np.random.Generator(np.random.PCG64(seed))
    data = _oracle_data()
    flops, t_used, rows_done, toks_done = 0.0, 0.0, 0, 0
    while t_used < seconds:
        for fi, pool in data:
            b, f = fi.batch, fi.family
            T = b.num_tokens
            n = 8 if T > 64 else 4
            toks = rng.integers(0, T, n)
            heads = rng.integers(0, f.num_qo_heads, n)
            rows = np.stack([toks, heads], axis=1)
            req, pos = O.token_request_and_position(b.qo_indptr, b.start_pos)
            t0 = time.perf_counter()
            tt = np.unique(toks)
            qo = O.bf16_to_f64(fi.q_raw[tt])
            ko = O.bf16_to_f64(fi.k_raw[tt])
            w = (O.bf16_to_f64(fi.w_q), O.bf16_to_f64(fi.w_k))
            if f.head_dim == 256:
                O.prep_hd256(qo, ko, O.bf16_to_f64(fi.v_raw[tt]), *w, fi.eps, pos[tt], f.rope_theta)
            else:
                O.prep_hd512(qo, ko, *w, fi.eps, pos[tt], f.rope_theta)
            O.attention(fi.q_raw, pool, fi.layer, b.qo_indptr, b.kv_page_indptr, b.page_ids,
                        b.last_page_len, b.start_pos, f.num_kv_heads, f.window_left, fi.sm_scale,
                        rows=rows)
            t_used += time.perf_counter() - t0
            p = pos[toks]
            vis = p + 1 if f.window_left < 0 else np.minimum(p + 1, f.window_left + 1)
            flops += float(4.0 * f.head_dim * vis.sum())
            rows_done += n
            toks_done += len(tt)
    desc = (f"{rows_done} sampled attention rows (token, head) and the prep of {toks_done} "
            "sampled tokens over the four calls of the step (both families, prefill and decode)")
    return flops, t_used, desc


def cpu_cores():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = max((i.get("num_threads", 1) for i in info), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------- main arms
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seeds(rank: int):
    """Seeds of this rank's prefill and decode requests: every rank owns its own requests
    (weak scaling, no exchange step on the path)."""
    return 1005 + 7919 * rank, 1004 + 7919 * rank


def max_over_ranks(value: float, world: int, device) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, flops_per_rank: float, ms: float) -> float:
    """Whole-job TFLOP/s: every rank's (equal-sized) work over the slowest rank's time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    per_step = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(per_step / 4)
    tot_f, tot_t, desc = 0.0, 0.0, ""
    for _ in range(args.steps):
        f, t, desc = oracle_sample(per_step)
        tot_f += f
        tot_t += t
    value = tot_f / tot_t / 1e12
    cores = cpu_cores()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "l2": "n/a (host)"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": desc + f"; {per_step:.1f} s of oracle time per step"},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def kernel_traffic(call_name):
    """DRAM bytes per launch of a call from the committed ncu summary (profiles/traffic.json),
    if that capture was taken on the current kernel source; otherwise None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    ent = json.load(open(p)).get("calls", {}).get(call_name)
    if not ent:
        return None
    src = os.path.join(ROOT, "paged_sliding_window_qkv_gb300", "csrc", ent["source"])
    if not os.path.exists(src):
        return None
    if hashlib.sha256(open(src, "rb").read()).hexdigest() != ent["sha256"]:
        return None
    return int(ent["dram_bytes_per_launch"])


def time_calls(calls, stream, flush, reps):
    """Median CUDA-event time (ms) of each zero-argument call, L2 flushed before each rep."""
    import torch
    out = []
    for c in calls:
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            c()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        out.append(statistics.median(ts))
    return out


def run_ours(args):
    import torch
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    from paged_sliding_window_qkv_gb300 import pg
    from paged_sliding_window_qkv_gb300 import workloads as W
    from paged_sliding_window_qkv_gb300.runner import FamilyRun

    peaks = load_peaks()
    # every call runs on one non-default stream (the plans are bound to it, and the decode
    # step's CUDA-graph capture needs a capturable stream); torch's work joins it too
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    # each rank owns its own requests (weak scaling; no exchange step on this path)
    seed5, seed4 = rank_seeds(rank)
    wl5 = W.make_workload(5, seed=seed5)
    wl4 = W.make_workload(4, seed=seed4)
    fams = [("prefill hd256", wl5.families[0]), ("prefill hd512", wl5.families[1]),
            ("decode hd256", wl4.families[0]), ("decode hd512", wl4.families[1])]
    runs = [(name, FamilyRun(fi, stream=stream)) for name, fi in fams]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def step(evs=None):
        i = 0
        for name, r in runs:
            if evs is not None:
                evs[i].record(stream)
            pg.check(r.prep_status(), name + " prep")
            if evs is not None:
                evs[i + 1].record(stream)
            pg.check(r.attn_status(), name + " attention")
            i += 2
        if evs is not None:
            evs[i].record(stream)

    # the clock sampler runs from before the warm-up, so it is sampling when the timed region
    # starts; only samples inside the timed region are summarised
    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    n_ev = 2 * len(runs) + 1
    all_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)]
               for _ in range(args.steps)]
    launches0 = pg.pg_launch_count()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    sampler.mark_start()
    for k in range(args.steps):
        # the flush is queued ahead of the step (no host sync in between), so the step's first
        # event does not also time the host's launch of its first call
        flush.zero_()
        step(all_evs[k])
    torch.cuda.synchronize()
    sampler.mark_stop()
    if world > 1:
        torch.distributed.barrier()
    launches = pg.pg_launch_count() - launches0
    clocks = sampler.stop()
    assert pg.pg_device_status() == pg.PG_OK

    # per-call durations (ms), averaged over steps
    seg = np.array([[all_evs[k][i].elapsed_time(all_evs[k][i + 1]) for i in range(n_ev - 1)]
                    for k in range(args.steps)])
    t_step = max_over_ranks(float(seg.sum(axis=1).mean()), world, "cuda")
    avg = seg.mean(axis=0)
    flops = [attn_flops(fi) for _, fi in fams]
    total_flops = sum(flops)
    value = job_value(world, total_flops, t_step)

    kernels = {}
    for i, (name, fi) in enumerate(fams):
        kernels[name + " prep"] = rate_entry(avg[2 * i], prep_bytes(fi), "hbm", peaks)
        if name.startswith("decode"):
            ent = rate_entry(avg[2 * i + 1], decode_bytes(fi), "hbm", peaks)
            ent["TFLOP/s"] = flops[i] / (avg[2 * i + 1] * 1e-3) / 1e12
        else:
            ent = rate_entry(avg[2 * i + 1], flops[i], "tensor", peaks)
        kernels[name + " attention"] = ent

    # dominant kernel: the call with the largest share of the step. Every call runs for
    # milliseconds at most, so the burst bf16 peak applies.
    dom_i = int(np.argmax(avg))
    dom_name = list(kernels)[dom_i]
    dom = kernels[dom_name]
    if "flops" in dom:
        roof = {"kernel": dom_name, "bound": "tensor", "achieved": dom["TFLOP/s"],
                "peak": peaks["bf16"], "unit": "TFLOP/s", "frac": dom["TFLOP/s"] / peaks["bf16"],
                "frac_nominal": dom["TFLOP/s"] / NOMINAL_BF16_TFLOPS,
                "peak_kind": f"bf16 burst, {peaks['src']}; frac_nominal against 2.25 PFLOP/s"}
    else:
        roof = {"kernel": dom_name, "bound": "hbm", "achieved": dom["GB/s"], "peak": peaks["hbm"],
                "unit": "GB/s", "frac": dom["GB/s"] / peaks["hbm"],
                "frac_nominal": dom["GB/s"] / NOMINAL_HBM_GBS,
                "peak_kind": f"hbm copy, {peaks['src']}; frac_nominal against 8 TB/s"}
    roof["share_of_step"] = float(avg[dom_i] / avg.sum())
    roof["traffic"] = kernel_traffic(dom_name)

    # ---- the decode step replayed as one CUDA graph (prep + attention of both families) ----
    dec = [r for name, r in runs if name.startswith("decode")]

    def decode_step():
        for r in dec:
            pg.check(r.prep_status(), "decode prep")
            pg.check(r.attn_status(), "decode attention")

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        decode_step()
    torch.cuda.synchronize()
    g_ms, e_ms = time_calls([graph.replay, decode_step], stream, flush, max(5, min(20, args.steps)))
    kernels["decode step as one CUDA graph"] = {
        "ms_graph": g_ms, "ms_eager": e_ms, "ms_eager_in_step": float(avg[4:8].sum()),
        "GB/s_graph": (sum(decode_bytes(fi) + prep_bytes(fi) for n, fi in fams
                           if n.startswith("decode")) / (g_ms * 1e-3) / 1e9)}
    del graph

    # ---- batched ragged prefill (8 requests x U[128, 2048] tokens, 4 layers x 8192 pages) ----
    if not args.no_extra:
        fi3 = W.make_workload(3, seed=1003 + 7919 * rank).families[0]
        r3 = FamilyRun(fi3, stream=stream)
        reps = max(5, min(20, args.steps))
        for _ in range(3):
            pg.check(r3.prep_status(), "cfg3 prep")
            pg.check(r3.attn_status(), "cfg3 attention")
        p_ms, a_ms = time_calls([lambda: pg.check(r3.prep_status(), "cfg3 prep"),
                                 lambda: pg.check(r3.attn_status(), "cfg3 attention")],
                                stream, flush, reps)
        kernels["batched prefill hd256 prep (8 requests, 4x8192-page pool)"] = rate_entry(
            p_ms, prep_bytes(fi3), "hbm", peaks)
        kernels["batched prefill hd256 attention (8 requests, 4x8192-page pool)"] = rate_entry(
            a_ms, attn_flops(fi3), "tensor", peaks)
        r3.close()
        del r3
    assert pg.pg_device_status() == pg.PG_OK

    # ---- end to end through the public API with host buffers ----
    # Each step first rebuilds every call's plan in place (small metadata uploads on the plans'
    # stream, ahead of the bulk input copies that would otherwise queue in front of them), then
    # copies each call's inputs in from pinned host memory on a copy stream of its own and its
    # output back on another, so the copies of one call overlap the kernels of its neighbours and
    # use several copy engines (a serving loop pipelines them the same way); the timed region
    # runs from the first upload to the last device-to-host copy. The calls run longest first
    # (prefill hd512, the decode step, prefill hd256): the long kernel hides the other calls'
    # input copies, and the large hd512 output streams back while the shorter calls compute.
    e2e_order = [1, 2, 3, 0]
    inputs, outputs = [], []
    h2d = d2h = 0
    for _, r in runs:
        # every step rebuilds the call's plan in place and uploads its metadata
        h2d += int(r.plan.info().metadata_bytes)
        pairs = []
        for t in [r.q_raw, r.k_raw, r.v_raw]:
            if t is None:
                continue
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            pairs.append((h, t))
            h2d += t.numel() * t.element_size()
        inputs.append(pairs)
        o = torch.empty(r.out.shape, dtype=r.out.dtype, pin_memory=True)
        outputs.append((o, r.out))
        d2h += r.out.numel() * r.out.element_size()
    h2d_streams = [torch.cuda.Stream() for _ in runs]
    d2h_streams = [torch.cuda.Stream() for _ in runs]

    def e2e_step():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in e2e_order:
            name, r = runs[i]
            b = r.fi.batch
            rc, _ = pg.pg_plan_paged_prefill(r.plan, b.num_req, b.qo_indptr, b.kv_page_indptr,
                                             b.page_ids, b.last_page_len, b.start_pos, r.Hq, r.Hkv,
                                             r.D, b.page_size, stream)
            pg.check(rc, name + " plan")
        landed = {}
        for i in e2e_order:
            h2d_streams[i].wait_event(e0)
            with torch.cuda.stream(h2d_streams[i]):
                for h, d in inputs[i]:
                    d.copy_(h, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(h2d_streams[i])
            landed[i] = ev
        back = []
        for i in e2e_order:
            name, r = runs[i]
            stream.wait_event(landed[i])
            pg.check(r.prep_status(), name + " prep")
            pg.check(r.attn_status(), name + " attention")
            done = torch.cuda.Event()
            done.record(stream)
            d2h_streams[i].wait_event(done)
            with torch.cuda.stream(d2h_streams[i]):
                outputs[i][0].copy_(outputs[i][1], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(d2h_streams[i])
            back.append(ev)
        for ev in back:
            stream.wait_event(ev)
        e1.record(stream)
        return e0, e1

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for k in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        e0, e1 = e2e_step()
        torch.cuda.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    t_e2e = max_over_ranks(float(np.mean(e2e_ms)), world, "cuda")
    e2e = {"value": job_value(world, total_flops, t_e2e), "unit": "TFLOP/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e}

    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            f, t, desc = oracle_sample(args.cpu_seconds)
            cpu = {"value": f / t / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(),
                   "kind": "oracle", "sample": desc + f" ({t:.1f} s of oracle time)"}
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic (seeded bf16 N(0,1), page ids shuffled)",
                "config": {"workload": WORKLOAD, "tokens_prefill": 16384, "decode_requests": 64,
                           "e2e": "pinned host inputs in, attention outputs out, and every call's "
                                  "plan rebuilt in place and uploaded, inside the timed region",
                           "l2": f"flushed between steps ({L2_FLUSH_BYTES >> 20} MiB write)",
                           "parallelism": f"replicas x{world} (independent requests per GPU)"},
                "kernels": kernels, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches, "clocks": clocks}
        print(json.dumps(line), flush=True)
    for _, r in runs:
        r.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0



# ---------------------------------------------------------------------------- next rows
NEXT_CASES = ("merge", "cascade-decode-hd512", "ring-decode-hd256", "ring-prefill-hd256")


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


def run_next_rows(args):
    """Calls beyond the single step, one JSON line per case (CUDA events, median of --steps calls
    after 3 warm-up calls, L2 flushed by a 512 MiB write before each call). Attention here only
    reads the pool, so the pools hold N(0,1) bf16 written directly and the queries are N(0,1)
    bf16. Cases:

    * merge: merging two attention states of 16384 tokens x 16 heads at head_dim 512
      (pg_merge_attn_states); bytes = rows x (3 x 512 x 2 + 12).
    * cascade-decode-hd512: a decode step of 64 requests sharing an 8192-token prefix and holding
      U[1, 1024] tokens of their own, full causal: the single pass over each request's own copy of
      all its keys, against the cascade (the prefix as one key segment listed for every request,
      the own keys as another, and the merge). Bytes are the single pass's K/V reads.
    * ring-decode-hd256: a decode step of 64 requests at positions U[4096, 32768) holding a ring
      of ceil((window + 1) / 16) + 1 pages, window_left 1023, against the same window on linear
      pages; bytes = visible keys x 8 heads x 256 x 2 x 2.
    * ring-prefill-hd256: a 4096-token chunk at position 65536 of one request on a ring of
      ceil((window + 4096) / 16) + 1 pages, window_left 1023, against linear pages;
      FLOP = 4 x 256 x 16 x visible pairs.
    """
    # the case helpers above use these two modules as globals
    global pg, torch
    import torch
    from paged_sliding_window_qkv_gb300 import pg
    peaks = load_peaks()
    hbm, bf16 = peaks["hbm"], peaks["bf16"]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    iters = max(5, args.steps)
    for c in NEXT_CASES:
        if c == "merge":
            res = case_merge(iters, flush, hbm)
        elif c == "cascade-decode-hd512":
            res = case_cascade(iters, flush, hbm)
        elif c == "ring-decode-hd256":
            rng = np.random.Generator(np.random.PCG64(17))
            starts = rng.integers(4096, 32768, 64)
            work = 64 * 1024 * 8 * 256 * 2 * 2
            res = ring_vs_linear(c, starts, [1] * 64, 1023, 16, 8, 256, 16, iters, flush,
                                 work, "B")
            res["frac_hbm_ring"] = res["ring_rate"] / hbm
        else:
            pairs = sum(min(p + 1, 1024) for p in range(65536, 65536 + 4096))
            res = ring_vs_linear(c, [65536], [4096], 1023, 16, 8, 256, 16, iters, flush,
                                 4.0 * 256 * 16 * pairs, "FLOP")
            res["frac_bf16_ring"] = res["ring_rate"] / bf16
        res["peaks"] = peaks["src"]
        print(json.dumps(res), flush=True)
    return 0 if pg.pg_device_status() == pg.PG_OK else 1


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the batched-prefill measurement outside the timed step")
    ap.add_argument("--next-rows", action="store_true",
                    help="time the calls beyond the step (merge, cascade, ring) and exit")
    args = ap.parse_args()
    if args.next_rows:
        return run_next_rows(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
