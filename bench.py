"""Benchmark of the DSpark ancestral draft-block sampler on one GB300.

One step = one whole K=7 draft block (every position kernel, pick and the
proposal writer) over the B=88, V=200064, r=256 workload (float32 drafter
logits, bfloat16 Markov head, T=1, requests 80..87 are CUDA-graph padding
rows), replayed from a CUDA graph -- the configuration the throughput target
is stated on.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (test infrastructure) on the host cores
on a bounded sample of the same workload.  Under torchrun (N > 1) every rank
runs an independent replica (no collective on the path); rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs per K=7 draft block (B×7×200064, r=256) and achieved HBM GB/s vs peak"
PAGES_US_B88 = 841.0  # PR #27 Results, "Drafting alone", B=88 (GB300)
CONFIG_ID = 4


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def workload_desc(w):
    return {
        "workload": ("draft block B=88 K=7 V=200064 r=256: f32 drafter logits "
                     "N(0,4^2)+32 spikes/row, bf16 U,Wb N(0,0.02^2), T=1, "
                     "requests 80-87 CUDA-graph padding rows (NaN logits)"),
        "B": w.B, "K": w.K, "V": w.V, "r": w.r,
        "base_dtype": "f32" if w.base_dtype == 0 else "bf16",
        "head_dtype": "bf16" if w.w_dtype == 1 else "f32",
        "timing": "CUDA-graph replay of dspark_draft_block, CUDA events",
        "l2": "inputs larger than L2 (2.7 GB touched per step; base 493 MB)",
    }


def compulsory_bytes(w):
    """Algorithmic bytes of one block: base read once, Wb read once per
    position, logits written, logits re-read by the proposal writer,
    proposals written (gathers, statistics and tokens are below 0.1%)."""
    elt = 4 if w.base_dtype == 0 else 2
    welt = 2 if w.w_dtype == 1 else 4
    B, K, V, r = w.B, w.K, w.V, w.r
    return B * K * V * elt + K * r * V * welt + 3 * B * K * V * 4


def position_kernel_bytes(w):
    """Algorithmic bytes of one position-kernel launch: base_k read, Wb read,
    logits_k written, the B gathered U rows read."""
    elt = 4 if w.base_dtype == 0 else 2
    welt = 2 if w.w_dtype == 1 else 4
    return w.B * w.V * elt + w.r * w.V * welt + w.B * w.V * 4 + w.B * w.r * welt


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []  # (host monotonic arrival time, csv line)
        self.t_start = None
        self.t_stop = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except OSError:
            self.proc = None
            return self
        # nvidia-smi takes a moment to start: wait (bounded) for its first
        # line so that sampling is live before the timed region opens
        deadline = time.monotonic() + 5.0
        while not self.lines and time.monotonic() < deadline and self.proc.poll() is None:
            time.sleep(0.005)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def start(self):
        """Marks the opening of the timed region (host clock)."""
        self.t_start = time.monotonic()

    def stop(self):
        """Marks the close of the timed region, after its synchronize."""
        self.t_stop = time.monotonic()
        # one more period so the sample taken at the close is read
        time.sleep(2 * self.period_ms / 1000.0)

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        lines = self.lines
        window = "whole sampler lifetime"
        if self.t_start is not None and self.t_stop is not None:
            # keep only the samples read while the timed region ran; a line
            # is read shortly after its query, hence the one-period slack
            slack = self.period_ms / 1000.0
            inside = [(t, ln) for t, ln in lines
                      if self.t_start <= t <= self.t_stop + slack]
            window = "timed region"
            if not inside:
                # region shorter than the sampling period: the first sample
                # read after it opened
                inside = [(t, ln) for t, ln in lines if t >= self.t_start][:1]
                window = "first sample after the timed region opened"
            lines = inside
        rows = []
        for _, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"],
                    "samples": 0, "window": window}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows
                          for i, f in enumerate(flags) if f.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(rows), "period_ms": self.period_ms,
                "window": window}


def source_hash(names):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ancestral_draft_sampling_gb300", "csrc")
    for name in names:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when the kernel's sources changed since the counters were taken."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        ent = d[kernel]
        if ent["source_hash"] != source_hash(ent["sources"]):
            return None
        return ent["dram_bytes_per_launch"]
    except (OSError, ValueError, KeyError):
        return None


def job_timing(ms_total_local, steps, world, dist=None, device="cpu"):
    """Whole-job timing of N independent replicas: the slowest rank's time
    (max over ranks) per step, and whole-job µs per block = that time / N
    (the N replicas each draft one block per step)."""
    ms_total = float(ms_total_local)
    if dist is not None and world > 1:
        import torch
        t = torch.tensor([ms_total], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
        dist.barrier()
    ms_step = ms_total / steps
    return ms_step, ms_step * 1e3 / world


# ------------------------------------------------------------ CPU oracle
def oracle_block_seconds(w, n_requests: int, threads: int):
    """Wall seconds for the oracle to draft `n_requests` requests (all K
    positions each, in order) with `threads` host threads."""
    import numpy as np
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    def one(b):
        prev = int(w.d0[b])
        pad = bool(w.pad_row[b]) if w.pad_row is not None else False
        greedy = bool(w.greedy[b]) if w.greedy is not None else False
        for k in range(w.K):
            res = oracle.draft_position(None if pad else w.base[b, k], w.U, w.Wb,
                                        prev, int(w.seed[b]), int(w.offset[b]),
                                        k, w.T, greedy=greedy, is_pad=pad)
            prev = res.token
        return prev

    reqs = list(range(n_requests))
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, reqs))
    return time.perf_counter() - t0


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, budget_s: float = 20.0):
    threads = cpu_threads()
    n = min(w.B, threads)
    t = oracle_block_seconds(w, n, threads)
    waves_full = -(-w.B // threads)
    per_block_s = t * waves_full  # one wave of n <= threads requests took t
    return {
        "value": per_block_s * 1e6, "unit": "us", "cores": threads,
        "kind": "oracle",
        "sample": (f"{n} of {w.B} requests x {w.K} positions in one parallel "
                   f"wave ({t:.2f} s), scaled by {waves_full} waves to a full "
                   f"block"),
    }


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from ancestral_draft_sampling_gb300 import workloads as wl
    w = wl.make_config(CONFIG_ID)
    threads = cpu_threads()
    n = min(w.B, threads)
    for _ in range(args.warmup):
        oracle_block_seconds(w, n, threads)
    times = [oracle_block_seconds(w, n, threads) for _ in range(args.steps)]
    waves = -(-w.B // threads)
    us = statistics.mean(times) * waves * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "us",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_desc(w),
        "cpu_baseline": {"value": us, "unit": "us", "cores": threads,
                         "kind": "oracle",
                         "sample": (f"each step: {n} of {w.B} requests x {w.K} "
                                    f"positions in one parallel wave, scaled "
                                    f"by {waves} waves")},
        "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- GPU arm
def run_ours(args, rank, world):
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build_library()
    import ancestral_draft_sampling_gb300 as pkg
    from ancestral_draft_sampling_gb300 import workloads as wl
    from tests.parity import to_device

    local = _env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    w = wl.make_config(CONFIG_ID)
    if args.positions != w.K:
        w.K = args.positions
        w.base = np.ascontiguousarray(w.base[:, :w.K])
    dev = to_device(w, f"cuda:{local}")
    B, K, V, r = w.B, w.K, w.V, w.r
    tokens = torch.empty((B, K), dtype=torch.int32, device="cuda")
    logits = torch.empty((B, K, V), dtype=torch.float32, device="cuda")
    probs = torch.empty((B, K, V), dtype=torch.float32, device="cuda")
    ws = pkg.DraftWorkspace(B, K, V, r)

    def call(stream=None):
        pkg.draft_block(dev["base"], dev["U"], dev["Wb"], dev["d0"], dev["seed"],
                        dev["offset"], w.T, greedy=dev["greedy"],
                        pad_row=dev["pad_row"], tokens=tokens, logits=logits,
                        draft_probs=probs, workspace=ws, stream=stream)

    if args.mode == "ncu":
        for _ in range(args.blocks):
            call()
        torch.cuda.synchronize()
        return 0

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        call(side)
    torch.cuda.synchronize()

    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    cur = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        torch.cuda.synchronize()
        clocks.start()
        ev0.record(cur)
        for _ in range(args.steps):
            graph.replay()
        ev1.record(cur)
        torch.cuda.synchronize()
        clocks.stop()
    ms_step, us_per_block = job_timing(ev0.elapsed_time(ev1), args.steps,
                                       world, dist, "cuda")

    # per-kernel durations, CUDA events around every launch on its stream
    prof = {"position": [0.0, 0], "pick": [0.0, 0], "proposal": [0.0, 0]}
    prof_reps = max(3, min(args.steps, 10))
    for _ in range(prof_reps):
        p = pkg.draft_block_profile(dev["base"], dev["U"], dev["Wb"], dev["d0"],
                                    dev["seed"], dev["offset"], w.T,
                                    greedy=dev["greedy"], pad_row=dev["pad_row"],
                                    tokens=tokens, logits=logits,
                                    draft_probs=probs, workspace=ws)
        for key, (ms, n) in p.items():
            prof[key][0] += ms
            prof[key][1] += n
    dominant = max(prof, key=lambda k: prof[k][0])
    avg_ms = {k: (v[0] / v[1] if v[1] else 0.0) for k, v in prof.items()}
    peak, peak_kind = measured_peaks()
    if dominant == "position":
        alg_bytes = position_kernel_bytes(w)
    elif dominant == "proposal":
        alg_bytes = 2 * B * K * V * 4
    else:  # the pick reads one 16-byte statistic per (request, CTA)
        n_ctas = min((V + 127) // 128,
                     torch.cuda.get_device_properties(0).multi_processor_count)
        alg_bytes = B * n_ctas * 16
    achieved = alg_bytes / (avg_ms[dominant] * 1e-3) / 1e9
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": achieved,
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": ncu_traffic(dominant),
                "alg_bytes_per_launch": alg_bytes,
                "avg_launch_ms": avg_ms[dominant],
                "stage_avg_ms": avg_ms,
                "stage_share": {k: v[0] / sum(x[0] for x in prof.values())
                                for k, v in prof.items()}}
    block_gbs = compulsory_bytes(w) / (ms_step * 1e-3) / 1e9

    # end to end through the public API with host buffers
    host_base = torch.from_numpy(
        w.base if w.base.dtype == np.float32 else w.base.view(np.int16)).pin_memory()
    if w.base.dtype != np.float32:
        host_base = host_base.view(torch.bfloat16)
    host_small = {k: dev[k].cpu().pin_memory() for k in ("d0", "seed", "offset")}
    for k2 in ("greedy", "pad_row"):
        if dev[k2] is not None:
            host_small[k2] = dev[k2].cpu().pin_memory()
    host_tokens = torch.empty((B, K), dtype=torch.int32).pin_memory()
    e2e_steps = max(3, min(args.steps, 10))
    cur = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    host_ws = pkg.HostWorkspace(B, K, V, r)

    def e2e_step():
        # dspark_draft_block_host: drafter logits copied position by position
        # on copy_stream while earlier positions compute; tokens copied back
        pkg.draft_block_host(host_base, dev["U"], dev["Wb"], host_small["d0"],
                             host_small["seed"], host_small["offset"], w.T,
                             base_dev=dev["base"], logits=logits,
                             draft_probs=probs, tokens_host=host_tokens,
                             greedy_host=host_small.get("greedy"),
                             pad_row_host=host_small.get("pad_row"),
                             workspace=host_ws, stream=cur,
                             copy_stream=copy_stream)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(cur)
    torch.cuda.synchronize()
    e2e_us = e0.elapsed_time(e1) / e2e_steps * 1e3 / world
    h2d = host_base.numel() * host_base.element_size() + sum(
        t.numel() * t.element_size() for t in host_small.values())
    d2h = host_tokens.numel() * 4
    # the last call's tokens came back through host memory
    assert torch.equal(host_tokens, tokens.cpu()), "host-fed tokens differ"

    # secondary path: standard verification of this block's drafts against
    # target distributions softmax(l + N(0,1)) (timing inputs, made by torch)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(5)
    tl = torch.cat([logits, logits[:, -1:]], dim=1)
    tl = tl + torch.randn(tl.shape, device="cuda", generator=gen)
    target = torch.softmax(tl.nan_to_num(neginf=-1e30), dim=-1)
    # temperature-only target sampling of the same B x (K+1) target rows
    tl_rows = tl.reshape(B * (K + 1), V).contiguous()
    del tl
    seed_rows = dev["seed"].repeat_interleave(K + 1)
    off_rows = dev["offset"].repeat_interleave(K + 1)
    pos_rows = torch.arange(K + 1, dtype=torch.int32, device="cuda").repeat(B)
    smp_tok = torch.empty(B * (K + 1), dtype=torch.int32, device="cuda")
    smp_probs = torch.empty_like(tl_rows)
    smp_ws = torch.empty(pkg._lib.load().dspark_sample_workspace_bytes(B * (K + 1), V),
                         dtype=torch.uint8, device="cuda")

    def sample_call():
        pkg.sample_temperature(tl_rows, seed_rows, off_rows, T=1.0,
                               position=pos_rows, tokens=smp_tok,
                               probs=smp_probs, workspace=smp_ws)

    for _ in range(3):
        sample_call()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record(cur)
    for _ in range(10):
        sample_call()
    g1.record(cur)
    torch.cuda.synchronize()
    sampler = {"us_per_call": g0.elapsed_time(g1) / 10 * 1e3,
               "rows": B * (K + 1), "V": V,
               "bytes": 3 * B * (K + 1) * V * 4,
               "note": "temperature-only sampling of the block's target rows "
                       "(token and probabilities per row)"}
    del tl_rows, smp_probs
    acc_len = torch.empty(B, dtype=torch.int32, device="cuda")
    emitted = torch.empty(B, dtype=torch.int32, device="cuda")

    def time_rule(fn, n_ver=20):
        for _ in range(3):
            fn(probs, target, tokens, dev["seed"], dev["offset"],
               accepted_len=acc_len, emitted_token=emitted)
        torch.cuda.synchronize()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(cur)
        for _ in range(n_ver):
            fn(probs, target, tokens, dev["seed"], dev["offset"],
               accepted_len=acc_len, emitted_token=emitted)
        f1.record(cur)
        torch.cuda.synchronize()
        return f0.elapsed_time(f1) / n_ver * 1e3, float(acc_len.float().mean().item())

    verify_us, mean_std = time_rule(pkg.verify_standard)
    block_us, mean_blk = time_rule(pkg.verify_block)
    verify = {"us_per_call": verify_us, "B": B, "K": K, "V": V,
              "mean_accepted_len": mean_std,
              "upper_bound_bytes": B * V * 8,
              "note": "standard rejection verification of the benchmark "
                      "block's drafts (one thread-block cluster of CTAs per request)",
              "block": {"us_per_call": block_us, "mean_accepted_len": mean_blk,
                        "bytes": 2 * B * (K - 1) * V * 4 + B * V * 8,
                        "note": "block verification of the same drafts: reads "
                                "the K-1 rows p_1..p_{K-1}, q_1..q_{K-1} in full"}}
    del target

    if rank == 0:
        line = {
            "metric": METRIC, "value": us_per_block, "unit": "us",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": False,
            "scaling": "weak",
            "vs_baseline": us_per_block / PAGES_US_B88,
            "dtype": "f32", "data": "synthetic",
            "config": dict(workload_desc(w), parallelism=f"replicas x{world}"),
            "block_hbm_gbs": block_gbs,
            "block_hbm_frac": block_gbs / peak,
            "compulsory_bytes_per_block": compulsory_bytes(w),
            "roofline": roofline,
            "clocks": clocks.summary(),
            "verify": verify,
            "target_sampler": sampler,
            # kernels of one block (counted by the profile pass) x steps
            "gpu_launches": args.steps * sum(v[1] for v in prof.values()) // prof_reps,
            "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "path": "dspark_draft_block_host: pinned-host drafter "
                            "logits copied per position on a second stream, "
                            "overlapped with the kernels; tokens copied back "
                            "to pinned host memory"},
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", choices=["bench", "ncu"], default="bench",
                    help="ncu: run a few eager blocks and exit (a small, "
                         "self-ending workload for profiler captures)")
    ap.add_argument("--positions", type=int, default=7,
                    help="draft positions K (7 = the benchmark workload; "
                         "fewer shrink the device footprint for captures)")
    ap.add_argument("--blocks", type=int, default=2,
                    help="eager blocks run by --mode ncu")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank = _env_int("RANK", 0)
    world = _env_int("WORLD_SIZE", args.gpus)
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world)


if __name__ == "__main__":
    sys.exit(main())
