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
(prep and decode GB/s, prefill TFLOP/s) is reported under "kernels".

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


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sustained=d["bf16_tflops_sustained"], src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


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
    """DRAM bytes per launch of a call from the committed ncu summary (profiles/traffic.md),
    if that capture was taken on the current kernel source; otherwise None."""
    p = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(p):
        return None
    for line in open(p):
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) < 4 or cells[0] != call_name:
            continue
        src = os.path.join(ROOT, "paged_sliding_window_qkv_gb300", "csrc", cells[1])
        if not os.path.exists(src):
            return None
        if hashlib.sha256(open(src, "rb").read()).hexdigest() != cells[2]:
            return None
        return int(cells[3])
    return None


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
    stream = torch.cuda.current_stream()
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
        pb = prep_bytes(fi)
        kernels[name + " prep"] = {"ms": avg[2 * i], "GB/s": pb / (avg[2 * i] * 1e-3) / 1e9,
                                   "frac_hbm": pb / (avg[2 * i] * 1e-3) / 1e9 / peaks["hbm"],
                                   "bytes": pb}
        ent = {"ms": avg[2 * i + 1], "TFLOP/s": flops[i] / (avg[2 * i + 1] * 1e-3) / 1e12}
        if name.startswith("decode"):
            db = decode_bytes(fi)
            ent.update({"GB/s": db / (avg[2 * i + 1] * 1e-3) / 1e9,
                        "frac_hbm": db / (avg[2 * i + 1] * 1e-3) / 1e9 / peaks["hbm"],
                        "bytes": db})
        else:
            ent["frac_bf16"] = ent["TFLOP/s"] / peaks["bf16_sustained"]
            ent["flops"] = flops[i]
        kernels[name + " attention"] = ent

    # dominant kernel: the call with the largest share of the step
    dom_i = int(np.argmax(avg))
    dom_name = list(kernels)[dom_i]
    dom = kernels[dom_name]
    if "frac_bf16" in dom:
        roof = {"kernel": dom_name, "bound": "tensor", "achieved": dom["TFLOP/s"],
                "peak": peaks["bf16_sustained"], "unit": "TFLOP/s",
                "frac": dom["TFLOP/s"] / peaks["bf16_sustained"],
                "peak_kind": f"bf16 sustained, {peaks['src']}"}
    else:
        roof = {"kernel": dom_name, "bound": "hbm", "achieved": dom["GB/s"], "peak": peaks["hbm"],
                "unit": "GB/s", "frac": dom["GB/s"] / peaks["hbm"],
                "peak_kind": f"hbm copy, {peaks['src']}"}
    roof["traffic"] = kernel_traffic(dom_name)

    # ---- end to end through the public API with host buffers ----
    # Each call's inputs are copied in from pinned host memory on a copy stream and its output
    # copied back on another, so the copies of one call overlap the kernels of its neighbours
    # (a serving loop pipelines them the same way); the timed region runs from the first
    # host-to-device copy to the last device-to-host copy. The calls run longest first
    # (prefill hd512, the decode step, prefill hd256): the long kernel hides the other calls'
    # input copies, and the large hd512 output streams back while the shorter calls compute.
    e2e_order = [1, 2, 3, 0]
    inputs, outputs = [], []
    h2d = d2h = 0
    for _, r in runs:
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
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_step():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_stream.wait_event(e0)
        landed = {}
        for i in e2e_order:
            with torch.cuda.stream(h2d_stream):
                for h, d in inputs[i]:
                    d.copy_(h, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(h2d_stream)
            landed[i] = ev
        for i in e2e_order:
            name, r = runs[i]
            stream.wait_event(landed[i])
            pg.check(r.prep_status(), name + " prep")
            pg.check(r.attn_status(), name + " attention")
            done = torch.cuda.Event()
            done.record(stream)
            d2h_stream.wait_event(done)
            with torch.cuda.stream(d2h_stream):
                outputs[i][0].copy_(outputs[i][1], non_blocking=True)
        back = torch.cuda.Event()
        back.record(d2h_stream)
        stream.wait_event(back)
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


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
