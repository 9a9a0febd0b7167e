#!/usr/bin/env python
"""Benchmark of the MoE expert-parallel hot path on GB300.

One step = one pass of the whole path over one synthetic batch:
ep_route -> ep_layout -> ep_dispatch -> ep_combine (the expert FFN between
dispatch and combine is outside the library; its output buffer y is filled once
before timing with the synthetic expert's rows for this batch, which are the
same every step because routing is deterministic).

Default workload: the largest single-GPU one, the sweep's T=32768 point with
Zipf 1.2 expert popularity (H=7168, E=256 over R=64, top-8; 8.5 GB moved per
layer). ``--config`` selects another workload.

Printed: one JSON line (rank 0). ``value`` is achieved algorithmic GB/s of the
whole step (bytes every step must move at least once / device time), ``e2e``
the same through the public API with the host<->device copies of the step's
inputs and result inside the timed region, ``roofline`` the dominant call
against the measured HBM copy bandwidth (and the 8 TB/s nominal figure),
``cpu_baseline`` the CPU oracle on a bounded sample of the same workload.
Unless ``--no-blocks``: ``workloads`` holds the same figures for prefill, mid
and the other large sweep points, and ``latency`` the per-layer latency at the
sweep's small T (1, 8, 64; uniform and Zipf) and at decode.

``--impl reference`` times the CPU oracle (the only reference implementation
of this path) on the same workload, each step a bounded token sample.

Multi-GPU (torchrun, one process per GPU): every rank runs its own batch of
the workload (data-parallel shards, no exchange between ranks); value = bytes
of all ranks / the slowest rank's time ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import pathlib
import statistics
import subprocess
import sys
import time

ROOT = pathlib.Path(__file__).resolve().parent
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))

METRIC = "dispatch+combine µs/layer and achieved HBM GB/s (fraction of GB300 peak), 1 GPU"
FALLBACK_HBM_GBS = 6800.0
SPEC_HBM_GBS = 8000.0  # the GB300's nominal HBM3e bandwidth (~8 TB/s), reported beside the measured copy peak
# The line's own workload: the largest single-GPU one (8.5 GB moved per layer).
DEFAULT_WORKLOAD = "sweep-zipf-T32768"
# The other workloads the >= 70 % target names, each reported in a block of the same line.
BLOCK_WORKLOADS = ("prefill", "mid", "sweep-uniform-T4096", "sweep-zipf-T4096", "sweep-uniform-T32768")
# The sweep's small-T latency floor, plus the decode shape.
LATENCY_WORKLOADS = ("sweep-uniform-T1", "sweep-zipf-T1", "sweep-uniform-T8", "sweep-zipf-T8",
                     "sweep-uniform-T64", "sweep-zipf-T64", "decode")
# The files whose contents fix each timed kernel (profiles/dram_traffic.txt keys).
KERNEL_SOURCES = {
    "route": ["route.cu", "route_token.cuh"],
    "layout": ["layout.cu", "block_common.cuh"],
    "dispatch": ["dispatch.cu"],
    # the call runs the fused kernel at small T, else route + layout + dispatch kernels
    "dispatch_fused": ["fused.cu", "fused_kernel.cuh", "block_common.cuh", "route_token.cuh", "route.cu", "layout.cu",
                       "dispatch.cu"],
    "combine": ["combine.cu"],
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    p.add_argument("--config", default=DEFAULT_WORKLOAD,
                   help="workload name (tiny, decode, prefill, mid, sweep-<dist>-T<n>)")
    p.add_argument("--no-blocks", action="store_true",
                   help="time only --config (default: also the other throughput workloads and the small-T latency "
                        "points, each in a block of its own)")
    p.add_argument("--latency-steps", type=int, default=100, help="replays per small-T latency point (at least --steps)")
    p.add_argument("--e2e-steps", type=int, default=None, help="steps of the end-to-end leg (default min(steps, 200))")
    p.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU work of the oracle baseline")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-clocks", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="time the per-step launches only (no CUDA graph)")
    p.add_argument("--data-as-flag", action="store_true",
                   help="also time dispatch + expert as two kernels (bulk-synchronous) and as one "
                        "sentinel-polling kernel (Data-as-Flag)")
    p.add_argument("--schedule-ablation", action="store_true",
                   help="also time the dispatch pulled by the chunk schedule under three tables (latency-"
                        "homogenized, one class, whole ranks per worker) beside the token-major dispatch")
    p.add_argument("--tff", action="store_true",
                   help="also time the Token-Flag Fusion block codec (encode and decode of the send buffer)")
    p.add_argument("--separate", action="store_true",
                   help="step = ep_route, ep_layout, ep_dispatch, ep_combine (default: ep_dispatch_fused, ep_combine)")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# distributed plumbing (barrier + max over ranks; no data-path collective)
# ---------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def rank_workload(w, rank: int):
    """Rank r's shard: the same shapes with its own seed (independent tokens)."""
    return w.with_(seed=w.seed + rank) if rank else w


def reduce_max(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (200 ms) during the timed region."""
    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, enabled: bool = True):
        self.proc = None
        self.idx = device_index
        if not enabled:
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={device_index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_samples(out)


def parse_clock_samples(out: str) -> dict:
    """Median SM clock, max clock and the throttle reasons seen in nvidia-smi
    CSV lines of ``ClockSampler.QUERY`` (noheader, nounits); lines that do not
    parse are skipped."""
    sm, smax, reasons = [], None, set()
    for line in out.strip().splitlines():
        f = [x.strip() for x in line.split(",")]
        if len(f) < 10:
            continue
        try:
            sm.append(float(f[2]))
            smax = float(f[3])
        except ValueError:
            continue
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for name, val in zip(names, f[6:10]):
            if val.lower() == "active":
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# roofline inputs
# ---------------------------------------------------------------------------

def measured_peak_gbs():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            return float(json.loads(p.read_text())["hbm_gbs"]), "measured"
        except (KeyError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """Source text without comments and blank space, so that an edit to a
    comment does not mark a captured kernel as changed."""
    import re

    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.strip() for line in text.splitlines() if line.strip())


def kernel_source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel] + ["ep_internal.cuh"]:
        h.update(_code_only((ROOT / "combine_router_softmax_gb300" / "csrc" / rel).read_text()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    this workload and the kernel source has not changed since."""
    p = ROOT / "profiles" / "dram_traffic.txt"
    if not p.exists():
        return None
    try:
        data = json.loads(p.read_text())
        ent = data[workload][kernel]
    except (KeyError, ValueError):
        return None
    # an entry summed from other kernels' captures (the dispatch call at large
    # T runs route, layout and dispatch kernels) is valid while all of them are
    parts = ent.get("components")
    if parts:
        if any(data[workload].get(c, {}).get("source_sha256_16") != kernel_source_hash(c) for c in parts):
            return None
    elif ent.get("source_sha256_16") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------

def oracle_sample_pass(orc, w, T_s: int, logits, x):
    """One pass of the oracle over the first T_s tokens of the workload."""
    return orc.run_path(logits[:T_s], x[:T_s], E=w.E, R=w.R, k=w.k, n_groups=w.n_groups,
                        topk_groups=w.topk_groups, renormalize=w.renormalize, ranks_per_node=w.ranks_per_node,
                        self_rank=w.self_rank, W=w.num_workers)


def pick_sample_tokens(orc, w, logits, x, target_s: float) -> int:
    T_s = min(w.T, 16)
    while True:
        t0 = time.perf_counter()
        oracle_sample_pass(orc, w, T_s, logits, x)
        dt = time.perf_counter() - t0
        if T_s >= w.T or dt >= target_s / 4:
            break
        T_s = min(w.T, T_s * 4)
    scale = target_s / max(dt, 1e-6)
    return max(1, min(w.T, int(T_s * scale)))


def cpu_baseline(w, seconds: float) -> dict:
    import ep_synth
    import oracle

    orc = oracle.get()
    T_probe = min(w.T, 4096)
    logits = ep_synth.gate_logits(w.seed, T_probe, w.E, w.zipf_s)
    x = ep_synth.hidden_bf16_bits(w.seed, T_probe, w.H)
    T_s = pick_sample_tokens(orc, w.with_(T=T_probe), logits, x, min(seconds / 3, 2.0))
    ws = w.with_(T=T_s)
    reps, t_total = 0, 0.0
    while t_total < seconds or reps < 1:
        t0 = time.perf_counter()
        oracle_sample_pass(orc, w, T_s, logits, x)
        t_total += time.perf_counter() - t0
        reps += 1
    gbs = ws.total_bytes() * reps / t_total / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {T_s} of {w.T} tokens of {w.name}, whole path (route, layout, schedule, dispatch, "
                      f"expert, combine), {reps} passes in {t_total:.1f} s, single-threaded C; "
                      f"host has {os.cpu_count()} cores"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import ep_synth
    import oracle

    w = ep_synth.get_workload(args.config)
    orc = oracle.get()
    T_probe = min(w.T, 4096)
    logits = ep_synth.gate_logits(w.seed, T_probe, w.E, w.zipf_s)
    x = ep_synth.hidden_bf16_bits(w.seed, T_probe, w.H)
    # each step a bounded sample: the whole --steps/--warmup run stays near two minutes
    per_step = min(0.5, 120.0 / max(1, args.steps + args.warmup))
    T_s = pick_sample_tokens(orc, w.with_(T=T_probe), logits, x, per_step)
    for _ in range(args.warmup):
        oracle_sample_pass(orc, w, T_s, logits, x)
    times = []
    t_all = time.perf_counter()
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_sample_pass(orc, w, T_s, logits, x)
        times.append(time.perf_counter() - t0)
    wall = time.perf_counter() - t_all
    ws = w.with_(T=T_s)
    gbs = ws.total_bytes() * len(times) / sum(times) / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * sum(times) / len(times), 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32/f64 (CPU oracle)",
        "data": "synthetic", "config": workload_config(w, args, extra={"sample_tokens": T_s}),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {T_s} of {w.T} tokens per step, whole path, single-threaded C"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 3),
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(w, args, extra=None) -> dict:
    cfg = {"workload": w.note or w.name, "name": w.name, "T": w.T, "H": w.H, "E": w.E, "R": w.R, "k": w.k,
           "n_groups": w.n_groups, "topk_groups": w.topk_groups, "renormalize": w.renormalize,
           "zipf_s": w.zipf_s, "ranks_per_node": w.ranks_per_node, "num_workers": w.num_workers,
           "bytes_per_step": w.total_bytes(), "parallelism": f"dp{args.gpus} (independent shards)",
           "l2": "flushed before every timed step: 2x L2 written, then another 2x L2 read (no dirty line "
                 "of the flush is written back inside the timed step)"}
    if extra:
        cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def capture_step_graph(buf, device, fused: bool, pre=None):
    """route -> layout -> dispatch -> combine captured once into a CUDA graph
    (after ``pre()``, e.g. an L2 flush, when given).

    Two eager passes on the capture stream first, so that every lazy set-up
    inside the library (attributes, occupancy, symbol addresses) happens
    outside the capture."""
    import torch

    cap = torch.cuda.Stream(device)
    cap.wait_stream(torch.cuda.current_stream(device))
    bound = buf.bind(cap)
    calls = step_calls(bound, fused)
    with torch.cuda.stream(cap):
        for _ in range(2):
            if pre is not None:
                pre()
            for _, fn in calls:
                fn()
    cap.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        if pre is not None:
            pre()
        for _, fn in calls:
            fn()
    torch.cuda.synchronize()
    return g


def capture_callable_graph(fn, device):
    """fn() (torch work on the current stream) captured once into a CUDA graph."""
    import torch

    cap = torch.cuda.Stream(device)
    cap.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(cap):
        fn()
    cap.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        fn()
    torch.cuda.synchronize()
    return g


def graph_call_ms(buf, device, fused: bool, flush_l2, K: int):
    """Per-call times of the step inside a CUDA graph: the step's graph with an
    event-record node before each call and after the last (events recorded as
    graph nodes), replayed K times after 3 warm-up replays, L2 flushed before
    each replay and the events read after it. Returns {call: [ms, ...]}, or
    None where this PyTorch cannot record events as graph nodes."""
    import torch

    cap = torch.cuda.Stream(device)
    cap.wait_stream(torch.cuda.current_stream(device))
    calls = step_calls(buf.bind(cap), fused)
    try:
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(calls) + 1)]
    except TypeError:
        return None
    with torch.cuda.stream(cap):
        for _ in range(2):
            for _, fn in calls:
                fn()
    cap.synchronize()
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g, stream=cap):
            for j, (_, fn) in enumerate(calls):
                evs[j].record(cap)
                fn()
            evs[-1].record(cap)
    except RuntimeError:
        return None
    torch.cuda.synchronize()
    per = {n: [] for n, _ in calls}
    for i in range(K + 3):
        flush_l2()
        g.replay()
        torch.cuda.synchronize()
        if i >= 3:
            for j, (n, _) in enumerate(calls):
                per[n].append(evs[j].elapsed_time(evs[j + 1]))
    del g
    return per


def step_calls(bound, fused: bool):
    """The C-ABI calls of one step, in order, with the names their bytes are booked under."""
    if fused:
        return [("dispatch_fused", bound.dispatch_fused), ("combine", bound.combine)]
    return [("route", bound.route), ("layout", bound.layout), ("dispatch", bound.dispatch),
            ("combine", bound.combine)]


def call_bytes(w, name: str) -> int:
    kb = w.algorithmic_bytes()
    if name == "dispatch_fused":
        return kb["route"] + kb["layout"] + kb["dispatch"]
    return kb[name]


def data_as_flag_leg(ep, buf, w, device, flush_l2, K: int) -> dict:
    """dispatch -> expert handed over three ways, each captured in a CUDA graph and
    replayed K times with L2 flushed in between:
      bsp: ep_dispatch, then ep_expert_scale (kernel boundary as the barrier);
      sp:  ep_dispatch_expert_sp (rows handed over by sentinel polling; each
           call re-arms send for the next);
      sw:  ep_dispatch_expert_sw (stop-and-wait: a per-row flag released after
           the row lands; two graphs with epochs 1 and 2 replayed in turn)."""
    import numpy as np
    import torch

    row = w.H * 2
    if w.k % 4 != 0 or not 1024 <= row <= 48 * 1024:
        return {"unsupported": "needs k % 4 == 0 and rows of 1..48 KiB"}
    scale = torch.from_numpy((np.arange(w.E, dtype=np.float32) + np.float32(1)) / np.float32(w.E)).to(device)
    cap = torch.cuda.Stream(device)
    cap.wait_stream(torch.cuda.current_stream(device))

    def bsp():
        buf.dispatch(cap)
        buf.expert_scale(scale, cap)

    def sp():
        buf.dispatch_expert_sp(scale, cap)

    flag = torch.zeros(w.T * w.k, dtype=torch.int32, device=device)

    def sw1():
        buf.dispatch_expert_sw(scale, flag, 1, cap)

    def sw2():
        buf.dispatch_expert_sw(scale, flag, 2, cap)

    graphs = {}
    with torch.cuda.stream(cap):
        buf.layout(cap)
        bsp()
        bsp()
        y_bsp = buf.y.clone()
        buf.sentinel_arm(cap)
        sp()
        sp()
    cap.synchronize()
    same = bool(torch.equal(y_bsp, buf.y))
    with torch.cuda.stream(cap):
        buf.y.zero_()
        sw1()
        sw2()
    cap.synchronize()
    same = same and bool(torch.equal(y_bsp, buf.y))
    for name, fn in (("bsp", bsp), ("sp", sp), ("sw1", sw1), ("sw2", sw2)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn()
        graphs[name] = g
    torch.cuda.synchronize()
    out = {}
    stream = torch.cuda.current_stream(device)
    for name in ("bsp", "sp", "sw"):
        if name == "sp":
            buf.sentinel_arm(stream)
        # stop-and-wait alternates two graphs (epochs 1 and 2) so that every
        # replay finds the other epoch in the flags
        seq = [graphs["sw1"], graphs["sw2"]] if name == "sw" else [graphs[name]]
        for i in range(4):
            flush_l2()
            seq[i % len(seq)].replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i, (a, b_) in enumerate(ev):
            flush_l2()
            a.record(stream)
            seq[i % len(seq)].replay()
            b_.record(stream)
        torch.cuda.synchronize()
        out[name + "_us"] = round(1e3 * sum(a.elapsed_time(b_) for a, b_ in ev) / K, 2)
    err = ep.ep_device_error()
    rows_b = w.T * w.k * row
    kb = w.algorithmic_bytes()
    out.update({
        "bsp_kernels": 2, "sp_kernels": 1, "sw_kernels": 1,
        "sw_bytes": kb["dispatch"] + 2 * rows_b + 2 * w.T * w.k * 4,
        "bsp_bytes": kb["dispatch"] + 2 * rows_b,
        "sp_bytes": kb["dispatch"] + 3 * rows_b,
        "same_output": same and err == 0,
        "device_error": err,
        "steps": K,
    })
    out["sp_speedup"] = round(out["bsp_us"] / out["sp_us"], 3)
    out["sp_vs_sw_latency_cut"] = round(1.0 - out["sp_us"] / out["sw_us"], 3)
    return out


def rank_static_table(rank_offset, W: int):
    """Ablation table: worker r mod W takes the whole send segment of rank r
    (no balancing)."""
    per = [[] for _ in range(W)]
    for r in range(len(rank_offset) - 1):
        n = int(rank_offset[r + 1] - rank_offset[r])
        if n:
            per[r % W].append([r % W, 0, r, int(rank_offset[r]), n])
    rows, wb = [], [0]
    for p in per:
        rows += p
        wb.append(len(rows))
    return rows, wb


def schedule_ablation_leg(ep, buf, w, device, flush_l2, K: int) -> dict:
    """The dispatch pulled by the chunk schedule (ep_dispatch_scheduled) under
    three tables over the same rows, beside the token-major ep_dispatch:
      homogenized : ep_layout's table (every worker an equal share of each hop class);
      one_class   : ep_layout's table with every rank in the sender's node (equal row
                    shares, classes ignored: the token-count-only split);
      rank_static : whole destination ranks per worker, no balancing.
    Each is timed as a CUDA graph replayed K times with L2 flushed in between; one
    more eager call records %globaltimer per CTA, from which the per-worker end
    times (max over a worker's CTAs, relative to the earliest CTA start) give the
    peak (the slowest worker) and its ratio to the mean."""
    import numpy as np
    import torch

    row = w.H * 2
    if row > 48 * 1024:
        return {"unsupported": "rows above 48 KiB"}
    cap = torch.cuda.Stream(device)
    cap.wait_stream(torch.cuda.current_stream(device))
    W = (ep.ep_schedule_capacity(buf.cfg) - w.R) // buf.cfg.hop_classes
    tables = {}
    with torch.cuda.stream(cap):
        buf.layout(cap)
    cap.synchronize()
    n = int(buf.n_chunks.item())
    tables["homogenized"] = (buf.chunks[:n].clone(), buf.worker_begin[:W + 1].clone())
    one = ep.EpConfig.from_workload(w, ranks_per_node=w.R, ranks_per_pod=0, self_rank=0)
    b1 = ep.LayerBuffers.allocate(one, device=device)
    b1.topk_idx.copy_(buf.topk_idx)
    with torch.cuda.stream(cap):
        b1.layout(cap)
    cap.synchronize()
    n1 = int(b1.n_chunks.item())
    tables["one_class"] = (b1.chunks[:n1].clone(), b1.worker_begin[:W + 1].clone())
    del b1
    rows, wb = rank_static_table(buf.rank_offset.cpu().numpy(), W)
    tables["rank_static"] = (torch.tensor(rows, dtype=torch.int32, device=device).reshape(-1, 5),
                             torch.tensor(wb, dtype=torch.int32, device=device))
    chunks = torch.zeros((max(t[0].shape[0] for t in tables.values()) + 1, 5), dtype=torch.int32, device=device)
    worker_begin = torch.zeros((W + 1,), dtype=torch.int32, device=device)
    n_chunks = torch.zeros((1,), dtype=torch.int32, device=device)
    ref_send = torch.empty_like(buf.send)
    with torch.cuda.stream(cap):
        buf.dispatch(cap)
    cap.synchronize()
    ref_send.copy_(buf.send)
    n_ctas = ep.ep_dispatch_scheduled_ctas(buf.cfg)
    ns = torch.zeros((n_ctas, 2), dtype=torch.int64, device=device)
    stream = torch.cuda.current_stream(device)

    def time_graph(fn):
        with torch.cuda.stream(cap):
            fn()
            fn()
        cap.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn()
        torch.cuda.synchronize()
        for _ in range(3):
            flush_l2()
            g.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for a, b_ in ev:
            flush_l2()
            a.record(stream)
            g.replay()
            b_.record(stream)
        torch.cuda.synchronize()
        return round(1e3 * sum(a.elapsed_time(b_) for a, b_ in ev) / K, 2)

    out = {"scatter_us": time_graph(lambda: ep.ep_dispatch(buf.cfg, buf.x, buf.slot, buf.send, buf.slot_meta, cap)),
           "workers": W, "ctas": n_ctas, "steps": K}
    for name, (ch, wbt) in tables.items():
        chunks.zero_()
        chunks[:ch.shape[0]].copy_(ch)
        worker_begin.copy_(wbt)
        n_chunks.fill_(ch.shape[0])

        def fn(ns_arg=None):
            ep.ep_dispatch_scheduled(buf.cfg, buf.x, buf.slot, chunks, n_chunks, worker_begin, buf.send,
                                     buf.slot_meta, ns_arg, cap)

        us = time_graph(fn)
        flush_l2()
        torch.cuda.synchronize()
        with torch.cuda.stream(cap):
            fn(ns)
        cap.synchronize()
        same = bool(torch.equal(buf.send, ref_send))
        t = ns.cpu().numpy().astype(np.int64)
        t0 = t[:, 0].min()
        end = np.zeros(W, np.int64)
        for c in range(n_ctas):
            end[c % W] = max(end[c % W], t[c, 1] - t0)
        end_us = end / 1e3
        rows_w = np.diff(wbt.cpu().numpy())  # chunks per worker (not rows)
        out[name] = {"us": us, "peak_us": round(float(end_us.max()), 2), "mean_us": round(float(end_us.mean()), 2),
                     "peak_over_mean": round(float(end_us.max() / max(end_us.mean(), 1e-9)), 3),
                     "idle_workers": int((rows_w == 0).sum()), "same_send": same}
    out["device_error"] = ep.ep_device_error()
    return out


def e2e_pipelined(ep, buf, cfg, device, fused: bool, use_graph: bool, h_logits, h_x, n: int) -> dict:
    """End-to-end steps through the public API with every step's host->device
    copy of its inputs and device->host copy of its result, overlapped across
    steps: buffer set i % 2 serves step i; step i's input copy waits until step
    i-2 has finished reading that set, its compute waits for its input copy and
    for the copy-out of step i-2's result, and its result copy waits for its
    compute. Returns the total time of n steps (after two warm-up steps) and
    checks the last result."""
    import torch

    sets = [buf, ep.LayerBuffers.allocate(cfg, device=device)]
    sets[1].y.copy_(buf.y)
    s_c = torch.cuda.current_stream(device)
    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)
    if use_graph:
        graphs = [capture_step_graph(b, device, fused) for b in sets]
        run = [g.replay for g in graphs]
    else:
        bound = [b.bind(s_c) for b in sets]
        run = [(lambda bb=bb: [fn() for _, fn in step_calls(bb, fused)]) for bb in bound]
    h_outs = [torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    warm = 2
    total = n + warm
    ev_in = [torch.cuda.Event() for _ in range(total)]
    ev_c = [torch.cuda.Event() for _ in range(total)]
    ev_out = [torch.cuda.Event() for _ in range(total)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    for i in range(total):
        j = i % 2
        if i >= 2:
            s_in.wait_event(ev_c[i - 2])
        if i == warm:
            t0.record(s_in)
        with torch.cuda.stream(s_in):
            sets[j].logits.copy_(h_logits, non_blocking=True)
            sets[j].x.copy_(h_x, non_blocking=True)
        ev_in[i].record(s_in)
        s_c.wait_event(ev_in[i])
        if i >= 2:
            s_c.wait_event(ev_out[i - 2])
        run[j]()
        ev_c[i].record(s_c)
        s_out.wait_event(ev_c[i])
        with torch.cuda.stream(s_out):
            h_outs[j].copy_(sets[j].out, non_blocking=True)
        ev_out[i].record(s_out)
    t1.record(s_out)
    torch.cuda.synchronize()
    last = (total - 1) % 2
    assert torch.equal(h_outs[last].to(device), sets[last].out)
    return {"total_ms": t0.elapsed_time(t1)}


def tff_leg(ep, buf, w, device, flush_l2, K: int) -> dict:
    """The Token-Flag Fusion codec on this step's send buffer: ep_tff_encode
    (rows -> 512-byte blocks of 32 B metadata + 480 B payload) and
    ep_tff_decode (back, checking every block's flag), each captured in a CUDA
    graph and replayed K times with L2 flushed in between. Reports the framed
    size over the payload size (the codec's bandwidth overhead) and each
    kernel's bytes moved per second."""
    import torch

    cfg = buf.cfg
    nbytes = ep.ep_tff_framed_bytes(cfg)
    framed = torch.empty((nbytes,), dtype=torch.uint8, device=device)
    rows_back = torch.empty_like(buf.send)
    bad = torch.zeros(1, dtype=torch.int32, device=device)
    cap = torch.cuda.Stream(device)
    cap.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(cap):
        buf.dispatch(cap)
        ep.ep_tff_encode(cfg, buf.send, framed, 1, cap)
        ep.ep_tff_decode(cfg, framed, 1, rows_back, bad, cap)
    cap.synchronize()
    same = bool(torch.equal(rows_back.view(torch.int16), buf.send.view(torch.int16))) and int(bad.item()) == 0
    stream = torch.cuda.current_stream(device)
    out = {}
    for name, fn in (("encode", lambda: ep.ep_tff_encode(cfg, buf.send, framed, 2, cap)),
                     ("decode", lambda: ep.ep_tff_decode(cfg, framed, 2, rows_back, bad, cap))):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn()
        for _ in range(3):
            flush_l2()
            g.replay()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for a, b_ in ev:
            flush_l2()
            a.record(stream)
            g.replay()
            b_.record(stream)
        torch.cuda.synchronize()
        us = 1e3 * sum(a.elapsed_time(b_) for a, b_ in ev) / K
        moved = nbytes + buf.send.numel() * 2
        out[name + "_us"] = round(us, 2)
        out[name + "_gbs"] = round(moved / (us * 1e-6) / 1e9, 1)
    out.update({"payload_bytes": buf.send.numel() * 2, "framed_bytes": nbytes,
                "overhead": round(nbytes / (buf.send.numel() * 2), 4), "roundtrip_exact": same,
                "bad_blocks": int(bad.item()), "steps": K})
    return out


def reduce_max_many(values: dict, world: int, device=None) -> dict:
    """Max over ranks of every value: one all_reduce(MAX) of a float64 vector
    whose entries follow the sorted keys (every rank passes the same keys)."""
    if world == 1:
        return {k: float(v) for k, v in values.items()}
    import torch
    import torch.distributed as dist

    keys = sorted(values)
    t = torch.tensor([float(values[k]) for k in keys], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return {k: float(v) for k, v in zip(keys, t.tolist())}


def whole_job(bytes_per_step: int, world: int, steps: int, slowest_total_ms: float) -> tuple[float, float]:
    """(GB/s of all ranks, ms per step) when every rank moves bytes_per_step in
    each of `steps` steps and the slowest rank takes slowest_total_ms for them."""
    ms = slowest_total_ms / steps
    return world * bytes_per_step / (ms * 1e-3) / 1e9, ms


def step_stats_us(per_step_ms: list) -> dict:
    q = sorted(per_step_ms)
    return {"median": round(1e3 * q[len(q) // 2], 2), "p10": round(1e3 * q[len(q) // 10], 2),
            "p90": round(1e3 * q[(9 * len(q)) // 10], 2), "min": round(1e3 * q[0], 2), "max": round(1e3 * q[-1], 2)}


class Flusher:
    """Write 2x L2, then read another 2x L2: the step starts with none of its
    data in L2 and no dirty line left to write back inside the timed region."""

    def __init__(self, device):
        import torch

        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        n = max(2 * l2, 256 << 20)
        self.w = torch.empty(n, dtype=torch.uint8, device=device)
        self.r = torch.ones(n // 4, dtype=torch.int32, device=device)
        self.sink = torch.empty((), dtype=torch.int64, device=device)

    def __call__(self):
        import torch

        self.w.fill_(1)
        torch.sum(self.r, dim=0, dtype=torch.int64, out=self.sink)


def prepare_layer(ep, w, device):
    """Buffers of one layer with this batch's inputs and its expert output y
    (the synthetic expert: each send row scaled by (e + 1) / E), made before timing."""
    import numpy as np
    import torch

    import ep_synth

    cfg = ep.EpConfig.from_workload(w)
    logits_np = ep_synth.gate_logits(w.seed, w.T, w.E, w.zipf_s)
    x_np = ep_synth.hidden_bf16_bits(w.seed, w.T, w.H)
    buf = ep.LayerBuffers.allocate(cfg, device=device)
    buf.logits.copy_(torch.from_numpy(logits_np))
    buf.x.copy_(torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16))
    buf.bind(torch.cuda.current_stream(device)).dispatch_fused()
    rows = torch.arange(w.T * w.k, device=device, dtype=torch.int32)
    e = torch.searchsorted(buf.expert_offset, rows, right=True) - 1
    buf.y.copy_((buf.send.float() * ((e + 1).float() / w.E)[:, None]).to(torch.bfloat16))
    del rows, e
    torch.cuda.synchronize()
    return cfg, buf, logits_np, x_np


def measure_workload(ep, w0, args, rank: int, world: int, device, flush_l2, K: int,
                     cpu_seconds: float) -> tuple[dict, object]:
    """Time one workload the way the JSON line reports it. Returns the
    workload's block (values already reduced over ranks) and its buffers."""
    import numpy as np
    import torch

    w = rank_workload(w0, rank)
    cfg, buf, logits_np, x_np = prepare_layer(ep, w, device)
    stream = torch.cuda.current_stream(device)
    bound = buf.bind(stream)
    fused = not args.separate
    calls = step_calls(bound, fused)

    def step():
        for _, fn in calls:
            fn()

    for _ in range(max(args.warmup, 0)):
        flush_l2()
        step()
    torch.cuda.synchronize()
    graph = None if args.no_graph else capture_step_graph(buf, device, fused)
    if graph is not None:
        for _ in range(max(args.warmup, 0)):
            flush_l2()
            graph.replay()
        torch.cuda.synchronize()

    # (1) the calls launched one by one, an event between consecutive calls
    nc = len(calls)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nc + 1)] for _ in range(K)]
    clocks = ClockSampler(torch.cuda.current_device(), enabled=not args.no_clocks)
    time.sleep(0.3 if not args.no_clocks else 0)
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(K):
        flush_l2()
        evs = ev[i]
        for j, (_, fn) in enumerate(calls):
            evs[j].record(stream)
            fn()
        evs[nc].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    per = {n: [] for n, _ in calls}
    step_ms = []
    for evs in ev:
        for j, (n, _) in enumerate(calls):
            per[n].append(evs[j].elapsed_time(evs[j + 1]))
        step_ms.append(evs[0].elapsed_time(evs[nc]))

    # (2) the same calls captured once in a CUDA graph, replayed K times
    if graph is not None:
        gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        clocks = ClockSampler(torch.cuda.current_device(), enabled=not args.no_clocks)
        time.sleep(0.3 if not args.no_clocks else 0)
        barrier(world)
        torch.cuda.synchronize()
        gwall0 = time.perf_counter()
        for a, b_ in gev:
            flush_l2()
            a.record(stream)
            graph.replay()
            b_.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        wall += time.perf_counter() - gwall0
        gclk = clocks.stop()
        if gclk is not None:
            clk = gclk
        per_step_ms = [a.elapsed_time(b_) for a, b_ in gev]
    else:
        per_step_ms = list(step_ms)

    # (3) end to end through the public API: pinned host inputs in, result out, every step
    E2E = args.e2e_steps if args.e2e_steps is not None else min(K, 200)
    h_logits = torch.from_numpy(logits_np).pin_memory()
    h_x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_out = torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory()
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(E2E)]
    for i in range(E2E + 3):
        flush_l2()
        if i >= 3:
            e2e_ev[i - 3][0].record(stream)
        buf.logits.copy_(h_logits, non_blocking=True)
        buf.x.copy_(h_x, non_blocking=True)
        if graph is not None:
            graph.replay()
        else:
            step()
        h_out.copy_(buf.out, non_blocking=True)
        if i >= 3:
            e2e_ev[i - 3][1].record(stream)
    torch.cuda.synchronize()
    assert torch.equal(h_out.to(device), buf.out)  # the result is the one the path computes
    pipe = e2e_pipelined(ep, buf, cfg, device, fused, graph is not None, h_logits, h_x, E2E)

    # slowest rank of every timed total
    tot = reduce_max_many({"stream": sum(step_ms), "step": sum(per_step_ms),
                           "e2e": sum(a.elapsed_time(b) for a, b in e2e_ev), "pipe": pipe["total_ms"]},
                          world, device)
    bytes_step = w.total_bytes()
    value, ms_per_step = whole_job(bytes_step, world, K, tot["step"])
    stream_gbs, stream_ms = whole_job(bytes_step, world, K, tot["stream"])
    e2e_val, e2e_ms = whole_job(bytes_step, world, E2E, tot["e2e"])
    pipe_val, pipe_ms = whole_job(bytes_step, world, E2E, tot["pipe"])

    launches_per_step = ep.ep_step_kernel_count(cfg, fused=fused)
    kb = {n: call_bytes(w, n) for n, _ in calls}
    eager_ms = {n: sum(v) / len(v) for n, v in per.items()}
    # per-call times inside the step's graph (as the step itself is timed), the
    # slowest rank's mean; the calls launched one by one as a fallback
    gper = graph_call_ms(buf, device, fused, flush_l2, K) if graph is not None else None
    if gper is not None:
        gmean = reduce_max_many({n: sum(v) / len(v) for n, v in gper.items()}, world, device)
        kern_ms, call_timing = gmean, "graph"
    else:
        kern_ms, call_timing = eager_ms, "eager"
    eager_ms = reduce_max_many(eager_ms, world, device)
    dom = max(kern_ms, key=kern_ms.get)
    peak, peak_kind = measured_peak_gbs()
    names = [n for n, _ in calls]
    multi = "dispatch_fused" if "dispatch_fused" in names else "layout"
    call_kernels = {n: 1 for n in names}
    call_kernels[multi] = launches_per_step - (len(names) - 1)
    by_call = {n: {"us": round(kern_ms[n] * 1e3, 2), "us_eager": round(eager_ms[n] * 1e3, 2),
                   "kernels": call_kernels[n],
                   "algorithmic_bytes": kb[n],
                   "achieved": round(kb[n] / (kern_ms[n] * 1e-3) / 1e9, 1),
                   "frac": round(kb[n] / (kern_ms[n] * 1e-3) / 1e9 / peak, 4),
                   "frac_of_spec": round(kb[n] / (kern_ms[n] * 1e-3) / 1e9 / SPEC_HBM_GBS, 4),
                   "traffic": ncu_traffic(n, w0.name)} for n in kern_ms}
    achieved = kb[dom] / (kern_ms[dom] * 1e-3) / 1e9
    block = {
        "value": round(value, 2),
        "unit": "GB/s",
        "ms_per_step": round(ms_per_step, 5),
        "config": workload_config(w0, args),
        "us_per_layer": round(ms_per_step * 1e3, 2),
        "timing": ("CUDA graph of the step's C-ABI calls, replayed per step" if graph is not None
                   else "the step's C-ABI calls launched per step"),
        "calls": names,
        "stream_us_per_layer": round(stream_ms * 1e3, 2),
        "us_per_layer_stats": step_stats_us(per_step_ms),
        "hbm_fraction": round(value / world / peak, 4),
        "hbm_fraction_of_spec": round(value / world / SPEC_HBM_GBS, 4),
        "kernel_us": {n: round(v * 1e3, 2) for n, v in kern_ms.items()},
        "kernel_us_eager": {n: round(v * 1e3, 2) for n, v in eager_ms.items()},
        "roofline": {
            "bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "frac_of_spec": round(achieved / SPEC_HBM_GBS, 4),
            "traffic": ncu_traffic(dom, w0.name),
            "algorithmic_bytes_per_launch": kb[dom], "kernels_in_call": call_kernels[dom],
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s",
            "spec_peak": SPEC_HBM_GBS,
            "by_call_timing": ("each call between event-record nodes of the step's CUDA graph (replayed after an "
                               "L2 flush)" if call_timing == "graph" else
                               "each call between events, the calls launched one by one after an L2 flush"),
            "by_call": by_call,
        },
        "e2e": {"value": round(pipe_val, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h_logits.numel() * 4 + h_x.numel() * 2,
                "d2h_bytes_per_step": h_out.numel() * 2, "ms_per_step": round(pipe_ms, 5), "steps": E2E,
                "mode": "pipelined: two buffer sets; the H2D copy of step i+1 and the D2H copy of step i-1 run on "
                        "their own streams while step i computes; timed from the first timed H2D to the last D2H",
                "serial": {"value": round(e2e_val, 2), "ms_per_step": round(e2e_ms, 5),
                           "mode": "copy in, step, copy out on one stream, L2 flushed before each step (untimed)"}},
        "gpu_launches": K * launches_per_step * (2 if graph is not None else 1),
        "clocks": clk,
        "wall_s": round(wall, 3),
    }
    if rank == 0 and not args.no_cpu_baseline:
        block["cpu_baseline"] = cpu_baseline(w0, cpu_seconds)
    del graph
    return block, buf


def latency_point(ep, w0, args, rank: int, world: int, device, flush_l2, K: int) -> dict:
    """Per-layer latency of one small batch: the step's graph replayed K times,
    L2 flushed before each replay (outside the events); median and spread over
    the replays, the slowest rank's median (``us_per_layer``). Also the step's
    marginal time inside a graph that holds the flush as well (``in_graph_us``,
    no graph launch of its own, as in a model that runs its layers in one graph),
    and the step timed right after the same step on another layer's buffers
    (``after_other_layer_us``: its data flushed, the kernels' code warm)."""
    import torch

    w = rank_workload(w0, rank)
    cfg, buf, _, _ = prepare_layer(ep, w, device)
    fused = not args.separate
    graph = capture_step_graph(buf, device, fused)
    stream = torch.cuda.current_stream(device)
    for _ in range(max(args.warmup, 3)):
        flush_l2()
        graph.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b_ in ev:
        flush_l2()
        a.record(stream)
        graph.replay()
        b_.record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b_) for a, b_ in ev]
    st = step_stats_us(ms)

    # The same step inside a graph that also holds the L2 flush, as a layer
    # runs inside a whole model's graph: its marginal time is the mean replay
    # time of [flush, step] minus that of [flush] alone (events around each
    # replay; the launch of the graph itself is paid by both).
    flush_step = capture_step_graph(buf, device, fused, pre=flush_l2)
    flush_only = capture_callable_graph(flush_l2, device)

    def mean_us(g, n):
        for _ in range(3):
            g.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for a, b_ in evs:
            a.record(stream)
            g.replay()
            b_.record(stream)
        torch.cuda.synchronize()
        return 1e3 * sum(a.elapsed_time(b_) for a, b_ in evs) / n

    NG = max(K, 200)
    in_graph = mean_us(flush_step, NG) - mean_us(flush_only, NG)

    # The step right after the same calls on another layer's buffers (same
    # shapes, its own inputs): L2 flushed before that other layer, so this
    # step's data is as cold as after the flush, but the kernels' code is warm,
    # as in a model whose layers run these kernels one after another.
    _, buf2, _, _ = prepare_layer(ep, rank_workload(w0.with_(seed=w0.seed + 1000), rank), device)
    other = capture_step_graph(buf2, device, fused)
    for _ in range(3):
        flush_l2()
        other.replay()
        graph.replay()
    ev2 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b_ in ev2:
        flush_l2()
        other.replay()
        a.record(stream)
        graph.replay()
        b_.record(stream)
    torch.cuda.synchronize()
    ms2 = [a.elapsed_time(b_) for a, b_ in ev2]

    red = reduce_max_many({"median": st["median"], "mean": 1e3 * sum(ms) / K, "in_graph": in_graph,
                           "other_median": step_stats_us(ms2)["median"], "other_mean": 1e3 * sum(ms2) / K},
                          world, device)
    peak, _ = measured_peak_gbs()
    out = {"us_per_layer": round(red["median"], 2), "us_mean": round(red["mean"], 2), "stats_us": st,
           "in_graph_us": round(red["in_graph"], 2), "in_graph_steps": NG,
           "after_other_layer_us": {"median": round(red["other_median"], 2), "mean": round(red["other_mean"], 2),
                                    "steps": K},
           "kernels": ep.ep_step_kernel_count(cfg, fused=fused), "bytes_per_step": w.total_bytes(),
           "hbm_fraction": round(w.total_bytes() / (red["median"] * 1e-6) / 1e9 / peak, 4), "steps": K,
           "T": w.T, "dist": "zipf 1.2" if w.zipf_s else "uniform"}
    del graph, flush_only, flush_step, buf, other, buf2
    return out


def run_gb300(args):
    import torch

    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    import combine_router_softmax_gb300 as ep
    import ep_synth

    flush_l2 = Flusher(device)
    K = args.steps
    w0 = ep_synth.get_workload(args.config)
    block, buf = measure_workload(ep, w0, args, rank, world, device, flush_l2, K, args.cpu_seconds)

    line = {
        "metric": METRIC,
        "value": block.pop("value"),
        "unit": block.pop("unit"),
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": block.pop("ms_per_step"),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 rows, fp32 routing and combine accumulation",
        "data": "synthetic",
        "config": block.pop("config"),
    }
    line.update(block)
    # the optional legs run on the main workload's buffers
    w = rank_workload(w0, rank)
    if args.schedule_ablation:
        line["schedule_ablation"] = schedule_ablation_leg(ep, buf, w, device, flush_l2, min(K, 500))
    if args.tff:
        line["tff"] = tff_leg(ep, buf, w, device, flush_l2, min(K, 500))
    if args.data_as_flag:
        line["data_as_flag"] = data_as_flag_leg(ep, buf, w, device, flush_l2, min(K, 500))
    del buf
    torch.cuda.empty_cache()

    if not args.no_blocks:
        # the other workloads the throughput target names, each timed the same way
        blocks = {}
        for name in BLOCK_WORKLOADS:
            if name == w0.name:
                continue
            b, bb = measure_workload(ep, ep_synth.get_workload(name), args, rank, world, device, flush_l2, K,
                                     args.cpu_seconds / 3)
            del bb
            torch.cuda.empty_cache()
            blocks[name] = b
        line["workloads"] = blocks
        # the sweep's latency floor at small T (and decode), in us per layer
        LK = max(K, args.latency_steps)
        line["latency"] = {name: latency_point(ep, ep_synth.get_workload(name), args, rank, world, device,
                                               flush_l2, LK) for name in LATENCY_WORKLOADS}
        torch.cuda.empty_cache()
    if ep.ep_device_error() != 0:
        raise RuntimeError("a kernel gave up on a bounded wait during the benchmark")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())
