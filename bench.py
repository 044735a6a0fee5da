"""Benchmark of the DSpark ancestral draft-block sampler on one GB300.

One step = one whole K=7 draft block (the memset of the error word and the
decision keys, every position kernel, the pick and the proposal writer) over
the B=88, V=200064, r=256 workload (float32 drafter logits, bfloat16 Markov
head, T=1, requests 80..87 are CUDA-graph padding rows), replayed from a
CUDA graph -- the configuration the throughput target is stated on.  Prints
one JSON line.  The other full-size configurations (B = 8, 44, 64) are
measured the same way under "per_config".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (test infrastructure) on the host cores
on the whole block.  Under torchrun (N > 1) every rank runs an independent
replica (no collective on the path); rank 0 prints.
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

    def __init__(self, gpu_id: str, period_ms: int = 20):
        self.gpu = gpu_id  # "GPU-<uuid>" (or an nvidia-smi index)
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


def nvsmi_gpu_id(local: int) -> str:
    """The identity nvidia-smi knows this CUDA device by: "GPU-<uuid>" from
    the device properties (CUDA_VISIBLE_DEVICES may renumber devices, so the
    CUDA index is not nvidia-smi's index); the CUDA index as a fallback."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        if u and u != "None":
            return u if u.startswith("GPU-") else "GPU-" + u
    except (AttributeError, RuntimeError):
        pass
    return str(local)


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
def oracle_block_seconds(w, threads: int):
    """Wall seconds for the oracle to draft the whole block (every request,
    all K positions each, in order) with `threads` host threads, requests
    dealt to the threads."""
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

    t0 = time.perf_counter()
    if threads == 1:
        for b in range(w.B):
            one(b)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, range(w.B)))
    return time.perf_counter() - t0


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w):
    """The oracle on the whole block: once with every host core (the
    reported value) and once single-threaded."""
    threads = cpu_threads()
    t_all = oracle_block_seconds(w, threads)
    t_one = oracle_block_seconds(w, 1)
    return {
        "value": t_all * 1e6, "unit": "us", "cores": threads,
        "kind": "oracle",
        "single_thread_us": t_one * 1e6,
        "sample": (f"the whole block ({w.B} requests x {w.K} positions) "
                   f"timed once with {threads} threads ({t_all:.2f} s) and "
                   f"once with 1 thread ({t_one:.2f} s)"),
    }


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from ancestral_draft_sampling_gb300 import workloads as wl
    w = wl.make_config(CONFIG_ID)
    threads = cpu_threads()
    for _ in range(args.warmup):
        oracle_block_seconds(w, threads)
    times = [oracle_block_seconds(w, threads) for _ in range(args.steps)]
    us = statistics.mean(times) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": us, "unit": "us",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": us / 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_desc(w),
        "cpu_baseline": {"value": us, "unit": "us", "cores": threads,
                         "kind": "oracle",
                         "sample": (f"each step: the whole block ({w.B} "
                                    f"requests x {w.K} positions) with "
                                    f"{threads} threads")},
        "e2e": {"value": us, "unit": "us", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- GPU arm
class GraphBlock:
    """One workload on the device with its outputs, its workspace and the
    draft block captured into a CUDA graph on a side stream."""

    def __init__(self, w, device):
        import torch

        import ancestral_draft_sampling_gb300 as pkg
        from ancestral_draft_sampling_gb300 import workloads as wl
        self.w = w
        self.dev = wl.to_device(w, device)
        B, K, V, r = w.B, w.K, w.V, w.r
        self.tokens = torch.empty((B, K), dtype=torch.int32, device=device)
        self.logits = torch.empty((B, K, V), dtype=torch.float32, device=device)
        self.probs = torch.empty((B, K, V), dtype=torch.float32, device=device)
        self.ws = pkg.DraftWorkspace(B, K, V, r, device=device)
        self.side = torch.cuda.Stream()
        self.side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(self.side):
            self.call(self.side)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.side):
            self.call(self.side)
        torch.cuda.synchronize()

    def kwargs(self):
        d = self.dev
        return dict(greedy=d["greedy"], pad_row=d["pad_row"], tokens=self.tokens,
                    logits=self.logits, draft_probs=self.probs,
                    workspace=self.ws)

    def args(self):
        d = self.dev
        return (d["base"], d["U"], d["Wb"], d["d0"], d["seed"], d["offset"],
                self.w.T)

    def call(self, stream=None):
        import ancestral_draft_sampling_gb300 as pkg
        pkg.draft_block(*self.args(), stream=stream, **self.kwargs())

    def time_replays(self, n):
        """Milliseconds of n back-to-back graph replays (CUDA events on the
        current stream)."""
        import torch
        cur = torch.cuda.current_stream()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(n):
            self.graph.replay()
        e1.record(cur)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    def timeline(self, replays):
        """(position chain ms, proposal writer ms) in the block's own
        schedule: dspark_draft_block_timeline's graph with event nodes."""
        import ancestral_draft_sampling_gb300 as pkg
        return pkg.draft_block_timeline(*self.args(), replays=replays,
                                        stream=self.side, **self.kwargs())

    def profile(self, reps):
        """Per-launch event brackets (dspark_draft_block_profile), summed
        over reps blocks: {class: [ms, launches]}."""
        import ancestral_draft_sampling_gb300 as pkg
        prof = {"position": [0.0, 0], "pick": [0.0, 0], "proposal": [0.0, 0]}
        for _ in range(reps):
            p = pkg.draft_block_profile(*self.args(), **self.kwargs())
            for key, (ms, n) in p.items():
                prof[key][0] += ms
                prof[key][1] += n
        return prof


def position_roofline(w, chain_ms, peak):
    """The position kernel in the block's schedule: the chain's time (the
    memset, K positions and the last pick) over K launches."""
    per_launch_ms = chain_ms / w.K
    alg = position_kernel_bytes(w)
    achieved = alg / (per_launch_ms * 1e-3) / 1e9
    return per_launch_ms, achieved, achieved / peak


def measure_config(cfg, steps, peak, device):
    """µs per block of configuration cfg from graph replays, its fraction of
    the compulsory-byte floor, and the position kernel's fraction."""
    import torch

    import ancestral_draft_sampling_gb300 as pkg
    from ancestral_draft_sampling_gb300 import workloads as wl
    w = wl.make_config(cfg)
    gb = GraphBlock(w, device)
    for _ in range(3):
        gb.graph.replay()
    torch.cuda.synchronize()
    n = max(20, steps)
    us = gb.time_replays(n) / n * 1e3
    chain_ms, prop_ms = gb.timeline(10)
    per_launch_ms, pos_gbs, pos_frac = position_roofline(w, chain_ms, peak)
    comp = compulsory_bytes(w)
    out = {
        "workload": (f"B={w.B} K={w.K} V={w.V} r={w.r}, "
                     f"{'f32' if w.base_dtype == 0 else 'bf16'} drafter logits, "
                     f"bf16 head, T={w.T}"
                     + (", 4 greedy rows" if w.greedy is not None else "")),
        "us_per_block": us, "replays": n,
        "compulsory_bytes": comp,
        "floor_us": comp / (peak * 1e9) * 1e6,
        "block_hbm_frac": comp / (us * 1e-6) / 1e9 / peak,
        "position": {"us_per_launch_in_chain": per_launch_ms * 1e3,
                     "alg_bytes_per_launch": position_kernel_bytes(w),
                     "achieved_gbs": pos_gbs, "frac": pos_frac},
        "proposal_us": prop_ms * 1e3,
    }
    if w.target is not None:
        # the configuration as configured: the drafts verified against its
        # target probabilities by both rules
        gb.graph.replay()
        torch.cuda.synchronize()
        rules = {}
        for name, fn in (("standard", pkg.verify_standard),
                         ("block", pkg.verify_block)):
            acc = torch.empty(w.B, dtype=torch.int32, device=device)
            emit = torch.empty(w.B, dtype=torch.int32, device=device)
            args = (gb.probs, gb.dev["target"], gb.tokens, gb.dev["seed"],
                    gb.dev["offset"])
            for _ in range(3):
                fn(*args, accepted_len=acc, emitted_token=emit)
            cur = torch.cuda.current_stream()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(cur)
            for _ in range(20):
                fn(*args, accepted_len=acc, emitted_token=emit)
            e1.record(cur)
            torch.cuda.synchronize()
            rules[name] = {"us_per_call": e0.elapsed_time(e1) / 20 * 1e3,
                           "mean_accepted_len": float(acc.float().mean())}
        out["verify"] = rules
    del gb
    torch.cuda.empty_cache()
    return out


def run_ours(args, rank, world):
    import numpy as np
    import torch

    import __graft_entry__
    __graft_entry__.build_library()
    import ancestral_draft_sampling_gb300 as pkg
    from ancestral_draft_sampling_gb300 import workloads as wl

    local = _env_int("LOCAL_RANK", 0)
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")

    w = wl.make_config(args.config if args.mode == "ncu" else CONFIG_ID)
    if args.mode == "ncu" and args.f32_head_rank > 0:
        # the same requests and drafter logits, a float32 head of that rank
        rng = np.random.default_rng(7000 + args.f32_head_rank)
        w.r = args.f32_head_rank
        w.U = rng.standard_normal((w.V, w.r), dtype=np.float32) * np.float32(0.02)
        w.Wb = rng.standard_normal((w.r, w.V), dtype=np.float32) * np.float32(0.02)
    if args.positions != w.K:
        w.K = args.positions
        w.base = np.ascontiguousarray(w.base[:, :w.K])
    B, K, V, r = w.B, w.K, w.V, w.r

    if args.mode == "ncu":
        # a small, self-ending workload for profiler captures: a few eager
        # blocks, then (--ncu-extra) one call of each verification rule and
        # of the target sampler on the block's outputs
        dev = wl.to_device(w, device)
        for _ in range(args.blocks):
            tokens, logits, probs = pkg.draft_block(
                dev["base"], dev["U"], dev["Wb"], dev["d0"], dev["seed"],
                dev["offset"], w.T, greedy=dev["greedy"], pad_row=dev["pad_row"])
        if args.ncu_extra:
            gen = torch.Generator(device=device)
            gen.manual_seed(5)
            tl = torch.cat([logits, logits[:, -1:]], dim=1)
            tl = tl + torch.randn(tl.shape, device=device, generator=gen)
            target = torch.softmax(tl.nan_to_num(neginf=-1e30), dim=-1)
            pkg.verify_standard(probs, target, tokens, dev["seed"], dev["offset"])
            pkg.verify_block(probs, target, tokens, dev["seed"], dev["offset"])
            del target
            rows = tl.reshape(B * (K + 1), V).contiguous()
            del tl
            pkg.sample_temperature(
                rows, dev["seed"].repeat_interleave(K + 1),
                dev["offset"].repeat_interleave(K + 1), T=1.0,
                position=torch.arange(K + 1, dtype=torch.int32,
                                      device=device).repeat(B))
        torch.cuda.synchronize()
        return 0

    gb = GraphBlock(w, device)
    dev = gb.dev
    for _ in range(args.warmup):
        gb.graph.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    cur = torch.cuda.current_stream()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(nvsmi_gpu_id(local)) as clocks:
        torch.cuda.synchronize()
        clocks.start()
        ev0.record(cur)
        for _ in range(args.steps):
            gb.graph.replay()
        ev1.record(cur)
        # the clock window: the same replays continue (no gap) for about a
        # second, so that the clock record holds many samples; its own time
        # is reported beside the timed region's
        cw_steps = max(args.steps, int(1.0 / 0.00048))
        ev2 = torch.cuda.Event(enable_timing=True)
        for _ in range(cw_steps):
            gb.graph.replay()
        ev2.record(cur)
        torch.cuda.synchronize()
        clocks.stop()
    ms_step, us_per_block = job_timing(ev0.elapsed_time(ev1), args.steps,
                                       world, dist, "cuda")
    clock_window_us = ev1.elapsed_time(ev2) / cw_steps * 1e3
    peak, peak_kind = measured_peaks()

    # the position kernel in the block's own schedule (graph replay, the
    # positions chained by programmatic dependent launch)
    chain_ms, prop_ms = gb.timeline(max(5, min(args.steps, 20)))
    per_launch_ms, achieved, frac = position_roofline(w, chain_ms, peak)
    # every launch bracketed by events (no overlap between launches)
    prof_reps = max(3, min(args.steps, 10))
    prof = gb.profile(prof_reps)
    iso_ms = {k: (v[0] / v[1] if v[1] else 0.0) for k, v in prof.items()}
    iso_gbs = position_kernel_bytes(w) / (iso_ms["position"] * 1e-3) / 1e9
    roofline = {
        "bound": "hbm", "kernel": "position_tc_kernel",
        "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
        "unit": "GB/s", "frac": frac,
        "traffic": ncu_traffic("position"),
        "alg_bytes_per_launch": position_kernel_bytes(w),
        "avg_launch_ms": per_launch_ms,
        "schedule": ("graph replay of the block, positions chained by "
                     "programmatic dependent launch; avg launch = (event "
                     "node before the memset .. event node after the last "
                     "pick) / K, so the memset and the pick are counted "
                     "against the position kernel (dspark_draft_block_timeline)"),
        "isolated": {
            "schedule": ("every launch bracketed by CUDA events, no overlap "
                         "between launches (dspark_draft_block_profile)"),
            "avg_launch_ms": iso_ms, "position_frac": iso_gbs / peak,
            "launches_per_block": {k: v[1] // prof_reps for k, v in prof.items()}},
        "proposal_ms_in_graph": prop_ms,
    }
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
    copy_stream = torch.cuda.Stream()
    host_ws = pkg.HostWorkspace(B, K, V, r)

    def e2e_step():
        # dspark_draft_block_host: drafter logits copied position by position
        # on copy_stream while earlier positions compute; tokens copied back
        pkg.draft_block_host(host_base, dev["U"], dev["Wb"], host_small["d0"],
                             host_small["seed"], host_small["offset"], w.T,
                             base_dev=dev["base"], logits=gb.logits,
                             draft_probs=gb.probs, tokens_host=host_tokens,
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
    assert torch.equal(host_tokens, gb.tokens.cpu()), "host-fed tokens differ"
    del host_base

    # secondary path: standard verification of this block's drafts against
    # target distributions softmax(l + N(0,1)) (timing inputs, made by torch)
    gen = torch.Generator(device=device)
    gen.manual_seed(5)
    tl = torch.cat([gb.logits, gb.logits[:, -1:]], dim=1)
    tl = tl + torch.randn(tl.shape, device=device, generator=gen)
    target = torch.softmax(tl.nan_to_num(neginf=-1e30), dim=-1)
    # temperature-only target sampling of the same B x (K+1) target rows
    tl_rows = tl.reshape(B * (K + 1), V).contiguous()
    del tl
    seed_rows = dev["seed"].repeat_interleave(K + 1)
    off_rows = dev["offset"].repeat_interleave(K + 1)
    pos_rows = torch.arange(K + 1, dtype=torch.int32, device=device).repeat(B)
    smp_tok = torch.empty(B * (K + 1), dtype=torch.int32, device=device)
    smp_probs = torch.empty_like(tl_rows)
    smp_ws = torch.empty(pkg._lib.load().dspark_sample_workspace_bytes(B * (K + 1), V),
                         dtype=torch.uint8, device=device)

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
               "compulsory_bytes": 2 * B * (K + 1) * V * 4,
               "note": "temperature-only sampling of the block's target rows "
                       "(token and probabilities per row); bytes: the three "
                       "launches' traffic (the logits read by the statistics "
                       "and again by the probability writer, the "
                       "probabilities written), compulsory_bytes: the logits "
                       "read once and the probabilities written once"}
    sampler["hbm_frac"] = sampler["bytes"] / (sampler["us_per_call"] * 1e-6) / 1e9 / peak
    sampler["hbm_frac_compulsory"] = (sampler["compulsory_bytes"] /
                                      (sampler["us_per_call"] * 1e-6) / 1e9 / peak)
    del tl_rows, smp_probs
    acc_len = torch.empty(B, dtype=torch.int32, device=device)
    emitted = torch.empty(B, dtype=torch.int32, device=device)

    def time_rule(fn, n_ver=20):
        for _ in range(3):
            fn(gb.probs, target, gb.tokens, dev["seed"], dev["offset"],
               accepted_len=acc_len, emitted_token=emitted)
        torch.cuda.synchronize()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(cur)
        for _ in range(n_ver):
            fn(gb.probs, target, gb.tokens, dev["seed"], dev["offset"],
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
    verify["block"]["hbm_frac"] = (verify["block"]["bytes"] /
                                   (block_us * 1e-6) / 1e9 / peak)
    del target

    per_config = None
    if world == 1 and not args.no_per_config:
        del gb
        torch.cuda.empty_cache()
        per_config = {str(c): measure_config(c, args.steps, peak, device)
                      for c in (2, 3, 5)}

    if rank == 0:
        clock = clocks.summary()
        clock["gpu"] = nvsmi_gpu_id(local)
        clock["window_note"] = (
            f"samples from the timed region and the clock window that follows "
            f"it without a gap ({cw_steps} more replays, "
            f"{clock_window_us:.1f} us per block)")
        launches_per_block = sum(v[1] for v in prof.values()) // prof_reps
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
            "clocks": clock,
            "verify": verify,
            "target_sampler": sampler,
            # kernels of one block (counted by the profile pass) x steps
            "gpu_launches": args.steps * launches_per_block,
            "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "path": "dspark_draft_block_host: pinned-host drafter "
                            "logits copied per position on a second stream, "
                            "overlapped with the kernels; tokens copied back "
                            "to pinned host memory"},
        }
        if per_config is not None:
            line["per_config"] = per_config
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
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the B = 8, 44, 64 configurations")
    ap.add_argument("--mode", choices=["bench", "ncu"], default="bench",
                    help="ncu: run a few eager blocks and exit (a small, "
                         "self-ending workload for profiler captures)")
    ap.add_argument("--positions", type=int, default=7,
                    help="draft positions K (7 = the benchmark workload; "
                         "fewer shrink the device footprint for captures)")
    ap.add_argument("--blocks", type=int, default=2,
                    help="eager blocks run by --mode ncu")
    ap.add_argument("--config", type=int, default=CONFIG_ID,
                    choices=[1, 2, 3, 4, 5],
                    help="workload of --mode ncu (4 = the benchmark block)")
    ap.add_argument("--ncu-extra", action="store_true",
                    help="--mode ncu: also one call of each verification "
                         "rule and of the target sampler")
    ap.add_argument("--f32-head-rank", type=int, default=0,
                    help="--mode ncu: the workload's shape with a float32 "
                         "head of this rank (the FFMA position kernel)")
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
