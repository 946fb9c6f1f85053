#!/usr/bin/env python3
"""Throughput of the MoE token path on one GB300: route -> dispatch (layout,
pack, receiver permute) -> combine, on the prefill workload of the
a2a-backends page (4,096 tokens per rank, 5,120-wide bf16 rows, 384 experts
top-6 over 8 partitions of 48).

Prints ONE JSON line.  `value` is algorithmic GB/s of the whole step (bytes
each call must move, counted from the measured copies and pairs) divided by
the device time of the step (CUDA events, L2 flushed before every step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (single thread, this host) on the same
workload and metric; the default run also reports the oracle single-threaded
and on every core (one process per core) as cpu_baseline(_all_cores).  Under torchrun each rank runs an independent replica on
its own batch (weak scaling, no data-path collective); rank 0 prints.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import moe_synth as ms  # noqa: E402

METRIC = "dispatch+combine HBM GB/s and rows/s at 4096-token prefill; % of HBM peak"
FALLBACK_HBM_GBS = 6800.0
DOMINANT = "k_perm_copy"
# The kernel the roofline line reports for each variant (the longest one of the
# step) and the key of its algorithmic bytes per launch in algorithmic_bytes().
DOMINANT_BY_VARIANT = {"two_stage": ("k_combine_stage1", "stage1"),
                       # the dequantizing stand-in expert is harness, not a step of the
                       # path: the line reports the longest of the path's own kernels
                       "mxfp8": ("k_combine", "combine"),
                       "nvfp4": ("k_combine", "combine"),
                       "routed": ("k_routed_stage1", "stage1")}
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# dominant kernel in the prefill pipeline, from an ncu capture with the L2 left
# as the previous kernel left it (--cache-control none), with the SHA-256 prefix
# of the code (comments and whitespace removed, source_code_sha16) of the files
# the kernel is built from, as they were when it was captured.  The line
# reports null instead once one of those files has changed, so a stale capture
# is never quoted.
DOMINANT_TRAFFIC = {("k_perm_copy", "prefill"): {"bytes": 142.5e6 + 252.9e6,
                                                 "sources": ["combine_moe_route_06_gb300/csrc/permute.cu"],
                                                 "sha16": "63c0e1b6e21e91ff"},
                    ("k_pack_permute", "prefill"): {"bytes": 43.52e6 + 430.24e6,
                                                    "sources": ["combine_moe_route_06_gb300/csrc/dispatch.cu",
                                                                "combine_moe_route_06_gb300/csrc/row_move.cuh"],
                                                    "sha16": "49a45874c40ef65a"}}


def source_code_sha16(*paths: str) -> str:
    """SHA-256 prefix of C/C++ sources (in the order given) with their comments
    and whitespace removed, so that editing a comment does not mark a capture
    stale."""
    import hashlib
    import re
    h = hashlib.sha256()
    for path in paths:
        with open(path) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = re.sub(r"\s+", " ", text).strip()
        h.update(text.encode())
    return h.hexdigest()[:16]


def dominant_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` at `workload` if the capture is current, else None."""
    rec = DOMINANT_TRAFFIC.get((kernel, workload))
    if rec is None:
        return None
    try:
        sha = source_code_sha16(*[os.path.join(ROOT, p) for p in rec["sources"]])
    except OSError:
        return None
    return rec["bytes"] if sha == rec["sha16"] else None


# ------------------------------------------------------------ byte model --

def algorithmic_bytes(S, T, H, E, k, P, copies, copies_recv, pairs_recv, two_stage=False,
                      mxfp8=False, routed=False, nvfp4=False):
    """Bytes each call must read + write at minimum.

    copies: rows packed (sum of part_offsets[s][P]); copies_recv: packed rows
    bound for the receiving partition(s); pairs_recv: permuted pair rows.
    two_stage: the combine pre-adds per (token, partition) slot (copies_recv
    rows written and read back) before the per-token sum.
    mxfp8 / nvfp4: packed and permuted rows are MXFP8 records of H + H/32
    bytes (NVFP4: H/2 + H/16), and the stand-in expert that dequantizes them
    (pair records in, bf16 rows out) is part of the step.
    routed: rows carry the token's ids and weights (8 bytes per choice), nothing
    is permuted, the routed expert pre-adds straight from the received rows
    (copies_recv rows in and out) and the home side sums them (stage 2).
    """
    NT = S * T
    R = H + H // 32 if mxfp8 else (H // 2 + H // 16 if nvfp4 else 2 * H)   # bytes of a moved row
    b = {
        "route": NT * E * 4 + NT * k * 8,
        "layout": NT * k * 4 + NT * P * 4 + S * (E + 2 * P + 1) * 4,
        "pack": NT * H * 2 + copies * R + copies * 4,
        "permute": copies_recv * R + pairs_recv * R + NT * k * 8,
        "combine": pairs_recv * H * 2 + NT * k * 8 + NT * H * 2,
    }
    if mxfp8 or nvfp4:
        b["expert"] = pairs_recv * R + pairs_recv * H * 2
    if two_stage:
        b["combine"] = (pairs_recv * H * 2 + NT * k * 12 + copies_recv * H * 2      # stage 1
                        + copies_recv * H * 2 + NT * P * 4 + NT * H * 2)            # stage 2
        b["stage1"] = pairs_recv * H * 2 + NT * k * 12 + copies_recv * H * 2
    if routed:
        b["pack"] += copies * k * 8
        b["permute"] = 0
        b["stage1"] = copies_recv * (H * 2 + k * 8) + copies_recv * H * 2
        b["combine"] = b["stage1"] + copies_recv * H * 2 + NT * P * 4 + NT * H * 2
    b["dispatch_combine"] = b["layout"] + b["pack"] + b["permute"] + b["combine"] + b.get("expert", 0)
    b["step"] = b["route"] + b["dispatch_combine"]
    b["perm_copy"] = copies_recv * R + pairs_recv * R + NT * k * 8
    # moe_dispatch: the four calls in one; its pack + permute kernel reads each
    # receiving send row back right after storing it (an L2 hit), so the bytes it
    # must move through HBM are the pack's and the permute's less that re-read
    b["dispatch"] = b["route"] + b["layout"] + b["pack"] + b["permute"] - copies_recv * R
    b["pack_permute"] = b["pack"] + b["permute"] - copies_recv * R
    b["step_hbm_fused"] = b["step"] - copies_recv * R
    return b


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


def host_cpu() -> dict:
    """The host's architecture, logical CPU count and CPU model as /proc/cpuinfo
    names it (x86: `model name`; Arm: implementer and part numbers)."""
    import platform
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            fields = {}
            for line in f:
                if ":" in line:
                    k_, v_ = line.split(":", 1)
                    fields.setdefault(k_.strip(), v_.strip())
        if "model name" in fields:
            model = fields["model name"]
        elif "CPU implementer" in fields:
            model = f"implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    except OSError:
        pass
    return {"machine": platform.machine(), "logical_cpus": os.cpu_count(), "model": model}


# ------------------------------------------------------ distributed glue --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """Largest value over all ranks (the slowest rank sets the job time)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, dist, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def rank_workload(name: str, rank: int) -> ms.Workload:
    """Each rank gets its own batch of the same shape (distinct seeds)."""
    w = ms.workload(name)
    return w if rank == 0 else ms.workload(name, index=w.index + 1000 * rank)


# ------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed loop runs."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int, interval_ms: int = 20):
        self.cmd = ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + ",".join(self.FIELDS),
                    "--format=csv,noheader,nounits", "-lms", str(interval_ms)]
        self.lines = []
        self.proc = None
        self.th = None

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.th = threading.Thread(target=self._read, daemon=True)
        self.th.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0: float | None = None, t1: float | None = None):
        """Summary of the samples taken between host times t0 and t1 (the loop)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.th.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        # samples taken while the loop ran; a loop shorter than the sampling
        # interval takes the samples nearest to it (within 0.25 s) instead
        lines = [(ts, ln) for ts, ln in self.lines if t0 is None or t0 <= ts <= t1]
        window = "timed loop"
        if not lines and t0 is not None:
            lines = [(ts, ln) for ts, ln in self.lines if t0 - 0.25 <= ts <= t1 + 0.25]
            window = "within 0.25 s of the timed loop (shorter than the sampling interval)"
        for ts, ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


def physical_gpu_index(local: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [v.strip() for v in vis.split(",") if v.strip()]
    if ids and local < len(ids) and ids[local].isdigit():
        return int(ids[local])
    return local


# ------------------------------------------------------- CPU oracle arm --

def oracle_step(inp, w):
    """One pass of the whole path through the CPU oracle (identity expert)."""
    import oracle
    ids, wt = oracle.route_topk(inp["logits"], w.k)
    lay = oracle.dispatch_layout(ids, w.E, w.P)
    cap_send = w.T * min(w.k, w.P)
    send, _, _ = oracle.dispatch_pack(inp["x"], lay["token_slot"], cap_send)
    per = oracle.permute_to_experts(send, lay["token_slot"], ids, w.E, recv_part=w.recv_part)
    oracle.combine(per["recv"], per["pair_row"], wt.astype(np.float32))
    copies = int(lay["part_offsets"][:, -1].sum())
    L = w.E // w.P
    if w.recv_part < 0:
        copies_recv = copies
    else:
        copies_recv = int(lay["part_counts"][:, w.recv_part].sum())
    pairs_recv = int(per["expert_offsets"][-1])
    _ = L
    return copies, copies_recv, pairs_recv


def time_oracle(w, seconds: float, max_steps: int, min_steps: int = 1):
    inp = ms.gen_inputs(w)
    n = 0
    t0 = time.perf_counter()
    stats = None
    while True:
        stats = oracle_step(inp, w)
        n += 1
        el = time.perf_counter() - t0
        if n >= min_steps and (el >= seconds or n >= max_steps):
            break
    b = algorithmic_bytes(w.S, w.T, w.H, w.E, w.k, w.P, *stats)
    return n, el, b


def _oracle_worker(name, seconds, barrier, results):
    """One spawned process of the all-cores oracle timing: its own inputs, then
    whole steps of the unchanged oracle from the common start until `seconds`."""
    w = ms.workload(name)
    inp = ms.gen_inputs(w)
    oracle_step(inp, w)                      # loads the oracle library
    barrier.wait(timeout=600)
    n, t0 = 0, time.perf_counter()
    while True:
        stats = oracle_step(inp, w)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    results.put((n, el, stats))


def time_oracle_all_cores(w, seconds: float):
    """The oracle on every core this process may use: one spawned process per
    core, each running whole steps on its own copy of the workload (the oracle
    itself stays single-threaded).  Returns (cores, steps, seconds, bytes per
    step); throughput = steps x bytes / seconds of the longest process.  Raises
    RuntimeError (after stopping the processes it started) if a process fails
    or the run overstays its time."""
    import multiprocessing as mp
    import queue
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    ctx = mp.get_context("spawn")            # fresh interpreters: nothing inherited from CUDA
    barrier, results = ctx.Barrier(cores), ctx.Queue()
    procs = [ctx.Process(target=_oracle_worker, args=(w.name, seconds, barrier, results))
             for _ in range(cores)]
    for p_ in procs:
        p_.start()
    out = []
    deadline = time.monotonic() + 600 + 4 * seconds
    try:
        while len(out) < cores:
            try:
                out.append(results.get(timeout=1.0))
            except queue.Empty:
                if any(p_.exitcode not in (None, 0) for p_ in procs):
                    raise RuntimeError("an oracle process failed")
                if time.monotonic() > deadline:
                    raise RuntimeError("the all-cores oracle run overstayed its time")
    finally:
        for p_ in procs:
            if p_.is_alive() and len(out) < cores:
                p_.terminate()
            p_.join()
    steps = sum(n for n, _, _ in out)
    el = max(e for _, e, _ in out)
    b = algorithmic_bytes(w.S, w.T, w.H, w.E, w.k, w.P, *out[0][2])
    return cores, steps, el, b


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    full = ms.workload(args.workload)
    # bounded sample: shrink the token count so that W + K steps take ~2 minutes
    inp_full = ms.gen_inputs(full)
    t0 = time.perf_counter()
    oracle_step(inp_full, full)
    t_full = time.perf_counter() - t0
    frac = min(1.0, 120.0 / ((args.steps + args.warmup) * t_full))
    T = max(64, int(full.T * frac))
    w = ms.workload(args.workload, T=T) if T < full.T else full
    inp = ms.gen_inputs(w) if T < full.T else inp_full
    for _ in range(args.warmup):
        oracle_step(inp, w)
    times = []
    stats = None
    for _ in range(args.steps):
        t0 = time.perf_counter()
        stats = oracle_step(inp, w)
        times.append(time.perf_counter() - t0)
    b = algorithmic_bytes(w.S, w.T, w.H, w.E, w.k, w.P, *stats)
    tot = sum(times)
    value = b["step"] * args.steps / tot / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, "none (CPU)"),
        "rows_per_s": round(w.S * w.T * args.steps / tot, 1),
        "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "host": host_cpu(),
                         "sample": f"{args.steps} steps of the {w.name} workload with T={w.T} of "
                                   f"{full.T} tokens per source, single thread"},
        "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def stage_summary(stage_ms, b, peak, tokens, copies, pairs):
    """Per stage of the path: µs (sum of its calls' medians from the per-stage
    loop), algorithmic GB/s, fraction of the HBM peak and rows/s, rows being
    what the stage writes: route and layout tokens, pack copies, permute and
    expert pairs, combine tokens."""
    def group(name):
        if name == "route_topk":
            return "route"
        if name == "dispatch":
            return "dispatch"
        for g in ("layout", "pack", "permute", "expert"):
            if name.startswith(g):
                return g
        return "combine"                   # combine, its two stages, the routed pre-add
    us = {}
    for name, v in stage_ms.items():
        g = group(name)
        us[g] = us.get(g, 0.0) + 1e3 * statistics.median(v)
    rows = {"route": tokens, "layout": tokens, "pack": copies, "permute": pairs,
            "expert": pairs, "combine": tokens, "dispatch": pairs}
    out = {}
    for g, t in us.items():
        gbs = b[g] / (t * 1e-6) / 1e9 if g in b else None
        out[g] = {"us": round(t, 2), "gbs": round(gbs, 1) if gbs else None,
                  "frac_of_hbm_peak": round(gbs / peak, 4) if gbs else None,
                  "rows_per_s": round(rows[g] / (t * 1e-6), 1)}
    return out


def workload_config(w, l2, variant="contiguous"):
    scope = "route+layout+pack+permute+combine"
    if variant == "routed":
        scope = "route+layout+pack(rows with ids and weights)+routed pre-add+home sum"
    if variant == "nvfp4":
        scope = "route+layout+pack(NVFP4 records)+permute+dequantizing stand-in expert+combine"
    if variant == "mxfp8":
        scope = "route+layout+pack(MXFP8 records)+permute+dequantizing stand-in expert+combine"
    return {"workload": f"{w.name}: S={w.S} T={w.T} H={w.H} bf16, E={w.E} top-{w.k}, "
                        f"P={w.P} partitions, recv_part={w.recv_part}",
            "variant": variant,
            "tokens_per_rank": w.S * w.T, "hidden": w.H, "experts": w.E, "topk": w.k,
            "partitions": w.P, "l2": l2, "value_scope": scope}


# ------------------------------------------------------------ GPU arm --

VARIANTS = {
    "contiguous": {},
    "masked": {"layout": "masked"},
    "two_stage": {"combine": "two_stage"},
    "mxfp8": {"quant": "mxfp8"},
    "nvfp4": {"quant": "nvfp4"},
    "placed": {},          # placement planned from another batch; see plan_for()
    "routed": {"layout": "routed"},
}


def plan_for(m, torch, w, dev, spare):
    """Placement by load with `spare` copy slots per partition, planned from
    the routing of another batch of the same workload (a plan is made from
    past load and used on new traffic).  Returns the Placement and the
    receiving partition to time: the busiest one under the plan when the
    workload times a single receiver, else -1 (all partitions)."""
    past = dataclasses.replace(w, index=w.index + 7919)
    tmp = m.MoePath(w.S, w.T, w.H, w.E, w.k, w.P, device=dev)
    tmp.route(torch.from_numpy(ms.gen_logits(past)).to(dev))
    m.moe_dispatch_layout(tmp.topk_ids, w.E, w.P, tmp.expert_counts, tmp.expert_rank,
                          tmp.part_counts, tmp.part_offsets, tmp.token_slot, tmp.ws, tmp.dev_status)
    load = tmp.expert_counts.sum(dim=0).cpu().numpy().astype(np.int64)
    del tmp
    pl = m.moe_plan_placement(load, w.P, spare)
    recv_part = int(np.argmax(pl.part_load)) if w.recv_part >= 0 else -1
    return pl, recv_part


def path_kwargs(args, w):
    """MoePath options of the --variant.  Masked blocks default to room for four
    times the mean pairs per expert (at least 64 rows, at most every token of
    every source); the JSON line's dev_status shows whether any pair was dropped."""
    kw = dict(VARIANTS[args.variant])
    if args.dispatch != "auto":
        kw["dispatch"] = args.dispatch
    if kw.get("layout") == "masked":
        mean = -(-w.S * w.T * w.k // w.E)
        kw["block_rows"] = args.block_rows or min(w.S * w.T, max(64, 4 * mean))
    return kw


def run_profile(args, local):
    """Small, quiet run for ncu: warm-up + K steps of the bound path, no flush
    buffers, no e2e phase, no clock sampling, no oracle."""
    import torch

    import combine_moe_route_06_gb300 as m

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    m.load_library()
    w = ms.workload(args.workload)
    inp = ms.gen_inputs(w)
    stream = torch.cuda.Stream(device=dev)
    path = m.MoePath(w.S, w.T, w.H, w.E, w.k, w.P, recv_part=w.recv_part, device=dev,
                     **path_kwargs(args, w))
    logits = torch.from_numpy(inp["logits"]).to(dev)
    x = torch.from_numpy(inp["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    calls = path.bind(logits, x, stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup + args.steps):
            m.MoePath.run_bound(calls)
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": w.name, "steps": args.steps, "warmup": args.warmup,
                      "launches_per_step": path.launches_per_step(),
                      "dev_status": int(path.dev_status.item())}), flush=True)
    return 0


def bind_to_gpu_numa(torch, local):
    """Run this process on the CPUs next to the GPU, so that pinned host buffers
    (first touched by this process) sit in that node's memory and host<->device
    copies take the direct link.  Returns a note for the JSON line."""
    try:
        prop = torch.cuda.get_device_properties(local)
        bus = f"{prop.pci_domain_id:04x}:{prop.pci_bus_id:02x}:{prop.pci_device_id:02x}.0"
        base = f"/sys/bus/pci/devices/{bus}"
        with open(f"{base}/local_cpulist") as f:
            spec = f.read().strip()
        cpus = set()
        for part in spec.split(","):
            if "-" in part:
                lo, hi = part.split("-")
                cpus.update(range(int(lo), int(hi) + 1))
            elif part:
                cpus.add(int(part))
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return {"bound": False, "why": f"no usable CPU in {spec}"}
        os.sched_setaffinity(0, cpus)
        node = open(f"{base}/numa_node").read().strip() if os.path.exists(f"{base}/numa_node") else "?"
        return {"bound": True, "cpus": spec, "numa_node": node, "pci": bus}
    except (OSError, ValueError, AttributeError) as exc:
        return {"bound": False, "why": str(exc)[:80]}


def hold_stream(torch, steps: int) -> bool:
    """Keep the current stream busy (torch's device sleep, a bounded clock-cycle
    count) for about 25 us per step to come, so that the host has enqueued all of
    them before the first runs: steps timed back to back then carry no host gap.
    Returns False (and holds nothing) where this torch has no device sleep."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is None:
        return False
    sleep(int(steps * 25e-6 * 2.1e9))
    return True


def time_other_workload(m, torch, name, steps, dev, local, flush_l2, peak, variant_kw):
    """Step time of another workload on the same GPU, with the headline's protocol:
    the step recorded once into a CUDA graph and replayed, the L2 flushed before
    every timed step, CUDA events around each step, nvidia-smi clocks sampled
    meanwhile.  Returns the workload's summary for the JSON line."""
    w = ms.workload(name)
    inp = ms.gen_inputs(w)
    path = m.MoePath(w.S, w.T, w.H, w.E, w.k, w.P, recv_part=w.recv_part, device=dev,
                     **variant_kw)
    logits = torch.from_numpy(inp["logits"]).to(dev)
    x = torch.from_numpy(inp["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    del inp
    stream = torch.cuda.Stream(device=dev)
    calls = path.bind(logits, x, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush_l2()
            m.MoePath.run_bound(calls)
    torch.cuda.synchronize()
    path.dev_status.zero_()
    m.MoePath.run_bound(calls)
    torch.cuda.synchronize()
    status = int(path.dev_status.item())
    copies = int(path.part_offsets[:, -1].sum().item())
    copies_recv = copies if w.recv_part < 0 else int(path.part_counts[:, w.recv_part].sum().item())
    pairs_recv = int((path.pair_row >= 0).sum().item())
    per_part = path.expert_counts.sum(dim=0).cpu().numpy().reshape(w.P, -1).sum(axis=1)
    b = algorithmic_bytes(w.S, w.T, w.H, w.E, w.k, w.P, copies, copies_recv, pairs_recv)
    cap = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        m.MoePath.run_bound(path.bind(logits, x, cap))
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    sampler = ClockSampler(physical_gpu_index(local))
    sampler.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush_l2()
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    clocks = sampler.stop(t0, t1)
    # the same steps back to back without the flush (inputs left in L2)
    evw = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps + 3)]
    with torch.cuda.stream(stream):
        hold_stream(torch, steps + 3)
        for i in range(steps + 3):
            evw[i][0].record(stream)
            graph.replay()
            evw[i][1].record(stream)
    torch.cuda.synchronize()
    warm = [1e3 * a.elapsed_time(b_) for a, b_ in evw[3:]]
    graph = None
    torch.cuda.synchronize()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    tot_s = sum(step_ms) * 1e-3
    gbs = b["step"] * steps / tot_s / 1e9
    return {"workload": f"{w.name}: S={w.S} T={w.T} H={w.H} bf16, E={w.E} top-{w.k}, "
                        f"P={w.P} partitions, recv_part={w.recv_part}",
            "steps": steps, "step_us_median": round(1e3 * statistics.median(step_ms), 2),
            "step_us_mean": round(1e3 * statistics.fmean(step_ms), 2),
            "warm_l2_us_mean": round(statistics.fmean(warm), 2),
            "gbs": round(gbs, 2), "frac_of_hbm_peak": round(gbs / peak, 4),
            "rows_per_s": round(w.S * w.T * steps / tot_s, 1), "bytes_per_step": b["step"],
            "copies_per_token": round(copies / (w.S * w.T), 4), "pairs_recv": pairs_recv,
            "partition_load": {"pairs_max_over_mean": round(float(per_part.max() / max(per_part.mean(), 1e-9)), 4),
                               "busiest_partition": int(per_part.argmax())},
            "launches_per_step": path.launches_per_step(), "dispatch_mode": path.dispatch_mode,
            "dev_status": status,
            "clocks": clocks}


# variants whose decode step the 40-layer graph also times (their MoePath options
# are all in path_kwargs; the placed variant needs a plan, the routed one has no
# pair rows to count)
LAYERED_DECODE_VARIANTS = ("contiguous", "masked", "mxfp8", "nvfp4", "two_stage")


def time_decode_layers(m, torch, steps, dev, local, peak, variant_kw, layers=40, byte_flags=None):
    """Decode as an engine runs it: one CUDA graph holding the round trips of
    `layers` MoE layers (route ... combine per layer, each layer with its own
    logits, x and buffers), replayed `steps` times (ishwarj.com a2a post, §1.4:
    40 round trips per decode step, recorded once and replayed).  The layers'
    inputs and outputs together are several times the L2, so each layer finds
    its data in HBM without a flush between replays; the kernels' code stays
    cached, as it does in a model's graph.  Returns the per-layer figures."""
    w = ms.workload("decode")
    lg = ms.gen_logits(w, T=w.T * layers).reshape(layers, w.S, w.T, w.E)
    xs = ms.gen_x(w, T=w.T * layers).reshape(layers, w.S, w.T, w.H)
    paths, bound_args = [], []
    for i in range(layers):
        p = m.MoePath(w.S, w.T, w.H, w.E, w.k, w.P, recv_part=w.recv_part, device=dev,
                      **variant_kw)
        li = torch.from_numpy(np.ascontiguousarray(lg[i])).to(dev)
        xi = torch.from_numpy(np.ascontiguousarray(xs[i]).view(np.int16)).to(dev).view(torch.bfloat16)
        paths.append(p)
        bound_args.append((li, xi))
    del lg, xs
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(3):
            for p, (li, xi) in zip(paths, bound_args):
                m.MoePath.run_bound(p.bind(li, xi, stream))
    torch.cuda.synchronize()
    for p in paths:
        p.dev_status.zero_()
    copies = pairs_recv = 0
    for p, (li, xi) in zip(paths, bound_args):
        m.MoePath.run_bound(p.bind(li, xi, stream))
    torch.cuda.synchronize()
    status = max(int(p.dev_status.item()) for p in paths)
    b_layers = 0
    for p in paths:
        c = int(p.part_offsets[:, -1].sum().item())
        pr = int((p.pair_row >= 0).sum().item())
        copies += c
        pairs_recv += pr
        b_layers += algorithmic_bytes(w.S, w.T, w.H, w.E, w.k, w.P, c, c, pr,
                                      **(byte_flags or {}))["step"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    cap = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for p, (li, xi) in zip(paths, bound_args):
            m.MoePath.run_bound(p.bind(li, xi, cap))
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps + 3)]
    sampler = ClockSampler(physical_gpu_index(local))
    sampler.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        hold_stream(torch, steps + 3)
        for i in range(steps + 3):
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    clocks = sampler.stop(t0, t1)
    graph = None
    torch.cuda.synchronize()
    rep_ms = [e0.elapsed_time(e1) for e0, e1 in ev[3:]]
    tot_s = sum(rep_ms) * 1e-3
    us_layer = [1e3 * t / layers for t in rep_ms]
    return {"workload": f"decode: S={w.S} T={w.T} H={w.H} bf16, E={w.E} top-{w.k}, "
                        f"P={w.P} partitions, {layers} layers in one CUDA graph, "
                        f"each layer its own inputs and buffers",
            "layers": layers, "replays": steps,
            "us_per_layer_mean": round(statistics.fmean(us_layer), 2),
            "us_per_layer_median": round(statistics.median(us_layer), 2),
            "graph_us_mean": round(1e3 * statistics.fmean(rep_ms), 2),
            "gbs": round(b_layers * steps / tot_s / 1e9, 2),
            "frac_of_hbm_peak": round(b_layers * steps / tot_s / 1e9 / peak, 4),
            "rows_per_s": round(w.S * w.T * layers * steps / tot_s, 1),
            "bytes_per_layer_mean": round(b_layers / layers),
            "data_per_replay_over_l2": round(b_layers / l2, 2),
            "copies_per_token": round(copies / (w.S * w.T * layers), 4),
            "path_options": {key: val for key, val in variant_kw.items()
                             if isinstance(val, (str, int, float))},
            "launches_per_layer": paths[0].launches_per_step(),
            "dispatch_mode": paths[0].dispatch_mode, "dev_status": status,
            "l2_flush": "none: the replay's data is several times the L2",
            "clocks": clocks}


def run_ours(args, world, rank, local):
    import torch

    import combine_moe_route_06_gb300 as m

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    host_binding = bind_to_gpu_numa(torch, local)
    dist = dist_init(world, "nccl")
    m.load_library()

    w = rank_workload(args.workload, rank)
    inp = ms.gen_inputs(w)
    stream = torch.cuda.Stream(device=dev)
    pkw = path_kwargs(args, w)
    placement_info = None
    if args.variant == "placed":
        pl, rp = plan_for(m, torch, w, dev, args.spare)
        pkw["placement"] = pl
        w = dataclasses.replace(w, recv_part=rp)
        placement_info = {"spare_slots_per_partition": args.spare, "recv_part": rp,
                          "physical_experts": pl.E_phys, "copies": int(pl.copy_offsets[-1]) - w.E,
                          "learned_from": "expert counts of another batch of the workload (index + 7919)"}
    path = m.MoePath(w.S, w.T, w.H, w.E, w.k, w.P, recv_part=w.recv_part, device=dev, **pkw)
    logits = torch.from_numpy(inp["logits"]).to(dev)
    x = torch.from_numpy(inp["x"].view(np.int16)).to(dev).view(torch.bfloat16)
    flush = torch.empty(1 << 30, dtype=torch.uint8, device=dev)   # 1 GiB > L2 (~126 MiB)
    clean = torch.ones(1 << 26, dtype=torch.float32, device=dev)  # 256 MiB read after the write

    def flush_l2():
        """Evict the step's data from L2: write 1 GiB, then read 256 MiB so the
        lines left in L2 are clean (no write-back charged to the next step)."""
        flush.fill_(1)
        clean.sum()

    h_logits = torch.from_numpy(inp["logits"]).pin_memory()
    h_x = torch.from_numpy(inp["x"].view(np.int16)).pin_memory()
    h_out = torch.empty((w.S, w.T, w.H), dtype=torch.int16).pin_memory()
    launches = path.launches_per_step()

    calls = path.bind(logits, x, stream)

    def step():
        m.MoePath.run_bound(calls)

    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 3)):
            flush_l2()
            step()
        torch.cuda.synchronize()
        path.dev_status.zero_()
        step()
        torch.cuda.synchronize()
        status = int(path.dev_status.item())
        per_part = path.expert_counts.sum(dim=0).cpu().numpy().reshape(w.P, -1).sum(axis=1)
        partition_load = {"pairs_max_over_mean": round(float(per_part.max() / max(per_part.mean(), 1e-9)), 4),
                          "busiest_partition": int(per_part.argmax())}
        copies = int(path.part_offsets[:, -1].sum().item())
        copies_recv = copies if w.recv_part < 0 else int(path.part_counts[:, w.recv_part].sum().item())
        if args.variant == "routed":
            # no pair rows are formed: count the pairs whose expert the receivers hold
            ids_d = path.topk_ids
            if w.recv_part >= 0:
                L_ = w.E // w.P
                pairs_recv = int(((ids_d >= w.recv_part * L_) & (ids_d < (w.recv_part + 1) * L_)).sum().item())
            else:
                pairs_recv = int(((ids_d >= 0) & (ids_d < w.E)).sum().item())
        else:
            pairs_recv = int((path.pair_row >= 0).sum().item())
        b = algorithmic_bytes(w.S, w.T, w.H, w.E, w.k, w.P, copies, copies_recv, pairs_recv,
                              two_stage=(args.variant == "two_stage"),
                              mxfp8=(args.variant == "mxfp8"), routed=(args.variant == "routed"),
                              nvfp4=(args.variant == "nvfp4"))
        dom_name, dom_key = DOMINANT_BY_VARIANT.get(args.variant, (DOMINANT, "perm_copy"))
        if path.dispatch_mode == "fused":
            # the longest kernel of the fused step's own calls: pack + permute in one
            # pass (quantizing with MXFP8 / NVFP4 rows), or the whole dispatch in one
            # launch for a decode-sized batch of bf16 rows
            if path.quantized:
                dom_name, dom_key = f"k_pack_permute_{path.quant}", "pack_permute"
            elif path.layout == "masked":
                dom_name, dom_key = "k_pack_permute_masked", "pack_permute"
            elif (path.placement is None
                  and m.moe_dispatch_kernels(w.S, w.T, w.k, w.E, w.P) == 1):
                dom_name, dom_key = "k_dispatch_small", "dispatch"
            else:
                dom_name, dom_key = "k_pack_permute", "pack_permute"
        if placement_info is not None:
            # pairs per partition on the timed batch: contiguous blocks vs the placement
            ids_h = path.topk_ids.cpu().numpy()
            logical = np.bincount(ids_h[ids_h >= 0], minlength=w.E)
            contiguous = logical.reshape(w.P, -1).sum(axis=1)
            placed = path.expert_counts.sum(dim=0).cpu().numpy().reshape(w.P, -1).sum(axis=1)
            placement_info["pairs_per_partition"] = {
                "contiguous_max_over_mean": round(float(contiguous.max() / contiguous.mean()), 4),
                "placed_max_over_mean": round(float(placed.max() / placed.mean()), 4),
                "placed_max_partition": int(np.argmax(placed))}

        # ---------------- the step as a CUDA graph (fixed shapes and addresses) ---
        # The five calls are recorded once and replayed, as a serving engine
        # runs them (no host work inside a step).  The timed steps replay a
        # clean graph; the dominant kernel is timed in a second, instrumented
        # copy of the step whose event nodes bracket that kernel (event nodes
        # break the programmatic-launch edges on both sides of it, so they stay
        # out of the timed steps).
        K = args.steps
        graph = graph_dom = None
        m.trace_disable()
        if not args.eager:
            cap = torch.cuda.Stream(device=dev)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                m.MoePath.run_bound(path.bind(logits, x, cap))
            # the trace's events back the instrumented graph's event nodes: the
            # trace stays enabled until that graph is released
            m.trace_enable(dom_name, max_records=8)
            m.trace_reset()
            graph_dom = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph_dom, stream=cap):
                m.MoePath.run_bound(path.bind(logits, x, cap))
            torch.cuda.synchronize()

        def run_step():
            if graph is not None:
                graph.replay()
            else:
                for fn, a in calls:            # route, layout, pack, permute, combine
                    if fn(*a) != 0:
                        raise RuntimeError(m.load_library().moe_last_error_message().decode())

        def run_dom_step():
            """The instrumented step: returns the dominant kernel's event times (ms)."""
            if graph_dom is not None:
                graph_dom.replay()
                torch.cuda.current_stream().synchronize()
                return [ms_ for name, ms_ in m.trace_records() if name == dom_name]
            m.trace_enable(dom_name, max_records=8)
            m.trace_reset()
            m.MoePath.run_bound(calls)
            torch.cuda.current_stream().synchronize()
            out = [ms_ for name, ms_ in m.trace_records() if name == dom_name]
            m.trace_disable()
            return out

        # ---------------- timed region: K steps, L2 flushed before each ------
        # Between timed steps (outside their events) the instrumented step runs
        # once, after its own flush, for the dominant kernel's launch time.
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        sampler = ClockSampler(physical_gpu_index(local)) if rank == 0 else None
        recs = []
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        if sampler:
            sampler.start()
            time.sleep(0.5)
        t_loop0 = time.perf_counter()
        flush2 = torch.empty(2 << 30, dtype=torch.uint8, device=dev)
        flush2.fill_(2)                    # head start so the host enqueues ahead of the GPU
        t_host0 = time.perf_counter()
        for i in range(K):
            flush_l2()
            e = ev[i]
            e[0].record(stream)
            run_step()
            e[1].record(stream)
            flush_l2()
            recs += run_dom_step()
        host_enqueue_us = (time.perf_counter() - t_host0) * 1e6 / K
        torch.cuda.synchronize()
        t_loop1 = time.perf_counter()
        if dist is not None:
            dist.barrier()
        clocks = sampler.stop(t_loop0, t_loop1) if sampler else None
        del flush2
        graph_dom = None                   # then the trace (and its events) can go
        torch.cuda.synchronize()
        m.trace_disable()

        # ---------------- warm L2 (diagnostic) ------------------------------
        # The same step back to back without the flush, each step timed by its
        # own events: what a small step (decode, ~15 MB) costs when its inputs
        # are still in the 126 MB L2 from the step before.
        Kw = max(10, min(K, 200))
        evw = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Kw + 3)]
        with torch.cuda.stream(stream):
            hold_stream(torch, Kw + 3)             # the host enqueues every step meanwhile
            for i in range(Kw + 3):                # the first 3 refill the L2
                evw[i][0].record(stream)
                run_step()
                evw[i][1].record(stream)
        torch.cuda.synchronize()
        warm = [1e3 * e0.elapsed_time(e1) for e0, e1 in evw[3:]]
        warm_us = statistics.median(warm)
        warm_mean_us = statistics.fmean(warm)

        # ---------------- dispatch + combine alone (diagnostic) ---------------
        # The same calls without the route (its outputs stay in the buffers),
        # as a clean graph (or eager calls), each run after an L2 flush.
        # (With moe_dispatch the route runs inside the dispatch call, so this is the
        # whole step.)
        Kd = max(10, min(K, 500))
        dc_start = 1 if path.dispatch_mode == "separate" else 0
        if not args.eager:
            graph_dc = torch.cuda.CUDAGraph()
            cap_dc = torch.cuda.Stream(device=dev)
            with torch.cuda.graph(graph_dc, stream=cap_dc):
                m.MoePath.run_bound(path.bind(logits, x, cap_dc), start=dc_start)
            torch.cuda.synchronize()
            run_dc = graph_dc.replay
        else:
            run_dc = lambda: m.MoePath.run_bound(calls, start=dc_start)  # noqa: E731
        ev_dc = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Kd)]
        for i in range(Kd):
            flush_l2()
            ev_dc[i][0].record(stream)
            run_dc()
            ev_dc[i][1].record(stream)
        torch.cuda.synchronize()
        dc_ms = [e[0].elapsed_time(e[1]) for e in ev_dc]
        graph_dc = None

        step_ms = [e[0].elapsed_time(e[1]) for e in ev]
        total_ms = sum(step_ms)
        job_ms = max_over_ranks(total_ms, dist, dev)
        bytes_all = sum_over_ranks(float(b["step"]) * K, dist, dev)
        rows_all = sum_over_ranks(float(w.S * w.T) * K, dist, dev)
        value = bytes_all / (job_ms * 1e-3) / 1e9

        # ---------------- end to end: pinned host in, pinned host out --------
        # Through the package's HostPipeline, as a serving loop would run it:
        # every step copies its logits and x in from pinned host memory and its
        # output back out; three buffer sets, copies overlapping neighbouring
        # steps (three streams ordered by events).
        Ke = max(10, min(K, 200))
        NB = 3
        pipe = m.HostPipeline(w.S, w.T, w.H, w.E, w.k, w.P, sets=NB, graphs=not args.eager,
                              device=dev, recv_part=w.recv_part, **pkw)
        h_outs = [h_out] + [torch.empty_like(h_out).pin_memory() for _ in range(NB - 1)]
        for i in range(NB):                        # warm every set once
            pipe.submit(h_logits, h_x, h_outs[i])
        pipe.synchronize()
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        e_start.record(pipe.s_in)
        for i in range(Ke):
            pipe.submit(h_logits, h_x, h_outs[i % NB])
        e_end.record(pipe.s_out)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e_start.elapsed_time(e_end), dist, dev)
        e2e_bytes = sum_over_ranks(float(b["step"]) * Ke, dist, dev)
        e2e_value = e2e_bytes / (e2e_ms * 1e-3) / 1e9
        # every set's last output, as copied out, against the device buffer and the
        # graph-replay path's output (same inputs, so the same bytes)
        ref_out = path.out.view(torch.int16).cpu().numpy()
        out_ok = all(bool(np.array_equal(h_outs[b_].numpy(), ref_out) and
                          np.array_equal(pipe.paths[(Ke + b_) % NB].out.view(torch.int16).cpu().numpy(),
                                         ref_out))
                     for b_ in range(NB))
        pipe.release()
        del pipe

        # the link's own rate for the same bytes: plain copies in (inputs) and out
        # (output) on two streams at once, no kernels
        d_in = torch.empty(int(h_logits.numel() * 4 + h_x.numel() * 2), dtype=torch.uint8, device=dev)
        h_in_raw = torch.empty(d_in.numel(), dtype=torch.uint8).pin_memory()
        d_out = torch.empty(int(h_out.numel() * 2), dtype=torch.uint8, device=dev)
        h_out_raw = torch.empty(d_out.numel(), dtype=torch.uint8).pin_memory()
        s_a, s_b = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        l0.record(s_a)
        s_b.wait_event(l0)
        for _ in range(Ke):
            with torch.cuda.stream(s_a):
                d_in.copy_(h_in_raw, non_blocking=True)
            with torch.cuda.stream(s_b):
                h_out_raw.copy_(d_out, non_blocking=True)
        s_a.wait_stream(s_b)
        l1.record(s_a)
        torch.cuda.synchronize()
        link_us = 1e3 * l0.elapsed_time(l1) / Ke
        del d_in, h_in_raw, d_out, h_out_raw

        graph = None
        torch.cuda.synchronize()

        # ---------------- per-stage breakdown (diagnostic; events between calls) --
        Kb = max(10, min(K, 200))
        eb = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
              for _ in range(Kb)]
        torch.cuda.synchronize()
        for i in range(Kb):
            flush_l2()
            eb[i][0].record(stream)
            for c, (fn, a) in enumerate(calls):
                fn(*a)
                eb[i][c + 1].record(stream)
        torch.cuda.synchronize()
        names = [fn.__name__.replace("moe_", "").replace("dispatch_", "") for fn, _ in calls]
        stage_ms = {name: [e[c].elapsed_time(e[c + 1]) for e in eb]
                    for c, name in enumerate(names)}

        # ---------------- per-kernel times (diagnostic; events around every launch) --
        m.trace_enable(None, max_records=Kb * 16)
        m.trace_reset()
        torch.cuda.synchronize()
        for i in range(Kb):
            flush_l2()
            m.MoePath.run_bound(calls)
        torch.cuda.synchronize()
        kern = {}
        kern_recs = m.trace_records()
        for name, ms_ in kern_recs:
            kern.setdefault(name, []).append(ms_)
        m.trace_disable()
        # the launch count claimed per step must be what the library launched
        traced_per_step = len(kern_recs) / Kb
        if traced_per_step != launches:
            raise RuntimeError(f"{traced_per_step} kernels traced per step, {launches} expected")
        kernels_us = {name: round(1e3 * statistics.median(v), 2) for name, v in kern.items()}

        # ---------------- the other GPU workloads (same protocol, rank 0) --------
        others = None
        if rank == 0 and args.other_workloads and args.variant == "contiguous":
            peak_o, _ = measured_peak()
            others = {}
            for name in [n for n in ("decode", "large", "skewed", "skewed_perm") if n != w.name]:
                steps_o = {"decode": 500, "large": 200, "skewed": 100, "skewed_perm": 100}[name]
                others[name] = time_other_workload(m, torch, name, steps_o, dev, local, flush_l2,
                                                   peak_o, path_kwargs(args, ms.workload(name)))
                torch.cuda.empty_cache()
        if rank == 0 and args.other_workloads and args.variant in LAYERED_DECODE_VARIANTS:
            if others is None:
                others = {}
            others["decode_40_layers"] = time_decode_layers(
                m, torch, 200, dev, local, measured_peak()[0],
                path_kwargs(args, ms.workload("decode")),
                byte_flags={"two_stage": args.variant == "two_stage",
                            "mxfp8": args.variant == "mxfp8", "nvfp4": args.variant == "nvfp4"})
            torch.cuda.empty_cache()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peak, peak_src = measured_peak()
    hbm_step = b["step_hbm_fused"] if path.dispatch_mode == "fused" else b["step"]
    dom_ms = statistics.fmean(recs) if recs else None
    dom_achieved = (b[dom_key] / (dom_ms * 1e-3) / 1e9) if dom_ms else None
    dc_gbs = b["dispatch_combine"] * len(dc_ms) / (sum(dc_ms) * 1e-3) / 1e9

    cpu = cpu_all = None
    if world == 1 and not args.no_cpu_baseline:
        n, el, bb = time_oracle(ms.workload(args.workload), args.cpu_seconds, max_steps=100)
        cpu = {"value": round(bb["step"] * n / el / 1e9, 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle", "host": host_cpu(),
               "sample": f"{n} full steps of the {w.name} workload in {el:.1f} s (single thread)"}
        import platform
        try:
            nc, na, ela, ba = time_oracle_all_cores(ms.workload(args.workload), args.cpu_seconds / 2)
            cpu_all = {"value": round(ba["step"] * na / ela / 1e9, 4), "unit": "GB/s",
                       "cores": nc, "kind": "oracle", "machine": platform.machine(),
                       "sample": f"{na} full steps of the {w.name} workload in {ela:.1f} s over "
                                 f"{nc} processes of the single-threaded oracle, one per core"}
        except RuntimeError as exc:
            cpu_all = {"unavailable": str(exc)}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(job_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"mxfp8": "bf16/e4m3", "nvfp4": "bf16/e2m1"}.get(args.variant, "bf16"),
        "data": "synthetic",
        "config": workload_config(w, "flushed before every timed step: 1 GiB write, then 256 MiB read (clean lines)",
                                  args.variant),
        "rows_per_s": round(rows_all / (job_ms * 1e-3), 1),
        "frac_of_hbm_peak": round(value / peak, 4),
        "hbm_bytes_per_step": hbm_step,
        "frac_of_hbm_peak_on_hbm_bytes": round(hbm_step * K / (job_ms * 1e-3) / 1e9 / peak, 4),
        "bytes_note": ("value counts the byte table of the separate calls (the send rows are read "
                       "by the permute); through moe_dispatch that read-back is an L2 hit, so the "
                       "step's HBM bytes are hbm_bytes_per_step"),
        "dispatch_combine": {"gbs": round(dc_gbs, 2), "us_median": round(1e3 * statistics.median(dc_ms), 2),
                             "frac_of_hbm_peak": round(dc_gbs / peak, 4),
                             "bytes": b["dispatch_combine"],
                             "how": ("layout + pack + permute + combine as their own clean graph "
                                     "(route outputs kept), L2 flushed before each run"
                                     if dc_start == 1 else
                                     "the whole step (moe_dispatch routes inside the call), "
                                     "as its own clean graph, L2 flushed before each run")},
        "warm_l2": {"us_median": round(warm_us, 2), "us_mean": round(warm_mean_us, 2),
                    "gbs": round(b["step"] / (warm_mean_us * 1e-6) / 1e9, 2),
                    "how": "the same step back to back without the L2 flush (inputs and "
                           "buffers left in L2 by the step before), enqueued behind a device "
                           "sleep so no host gap falls between steps; events around each step"},
        "step_us": {"median": round(1e3 * statistics.median(step_ms), 2),
                    "min": round(1e3 * min(step_ms), 2), "max": round(1e3 * max(step_ms), 2)},
        "stages_us_median": {k_: round(1e3 * statistics.median(v), 2) for k_, v in stage_ms.items()},
        "stages_note": "separate loop with events between calls (breaks launch overlap)",
        "stages": stage_summary(stage_ms, b, peak, w.S * w.T, copies, pairs_recv),
        "kernels_us_median": kernels_us,
        "kernels_note": "separate loop with events around every launch (includes launch latency)",
        "stage_bytes": {k_: b[k_] for k_ in ("route", "layout", "pack", "permute", "expert", "combine")
                        if k_ in b},
        "copies_per_token": round(copies / (w.S * w.T), 4),
        "pairs_recv": pairs_recv,
        "partition_load": partition_load,
        "dev_status": status,
        "roofline": {"kernel": dom_name, "bound": "hbm",
                     "achieved": round(dom_achieved, 1) if dom_achieved else None,
                     "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                     "frac": round(dom_achieved / peak, 4) if dom_achieved else None,
                     "traffic": (dominant_traffic(dom_name, w.name) if args.variant == "contiguous"
                                 else None),
                     "bytes_per_launch": b[dom_key],
                     **({"bytes_per_launch_by_call_table": b["pack"] + b["permute"],
                         "frac_on_call_table": round((b["pack"] + b["permute"]) / (dom_ms * 1e-3) / 1e9
                                                     / peak, 4) if dom_ms else None,
                         "bytes_note": "bytes_per_launch = the kernel's HBM bytes (the receiving send "
                                       "rows are read back from L2); the call table counts that "
                                       "read-back as the permute's input, as the separate calls do"}
                        if dom_key == "pack_permute" else {}),
                     "us_per_launch": round(1e3 * dom_ms, 2) if dom_ms else None,
                     "launches_timed": len(recs),
                     "how": "CUDA events around the kernel in an instrumented copy of the step, "
                            "run after its own L2 flush between the timed steps (event nodes "
                            "break the programmatic-launch edges, so the timed steps carry none)"},
        "cpu_baseline": cpu,
        "cpu_baseline_all_cores": cpu_all,
        **({"placement": placement_info} if placement_info is not None else {}),
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(h_logits.numel() * 4 + h_x.numel() * 2),
                "d2h_bytes_per_step": int(h_out.numel() * 2), "steps": Ke,
                "ms_per_step": round(e2e_ms / Ke, 4), "readback_ok": out_ok,
                "link_us_per_step": round(link_us, 1),
                "frac_of_link": round(link_us / (1e3 * e2e_ms / Ke), 4),
                "host_binding": host_binding,
                "how": "HostPipeline: pinned H2D -> step -> D2H every step on 3 streams with 3 "
                       "buffer sets; no L2 flush (each step moves ~1 GB); link_us_per_step: "
                       "plain copies of the same bytes in and out at once, no kernels"},
        # the timed steps and, between them, the instrumented copies of the step
        "gpu_launches": 2 * launches * K,
        "gpu_launches_per_step": launches,
        "gpu_launches_per_step_traced": traced_per_step,
        "launch_mode": "eager" if args.eager else "cuda_graph_replay",
        "dispatch_mode": path.dispatch_mode,
        "host_enqueue_us_per_step": round(host_enqueue_us, 1),
        "clocks": clocks,
        "other_workloads": others,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill", choices=sorted(ms.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--variant", default="contiguous", choices=sorted(VARIANTS),
                    help="contiguous runs + one-stage combine (default), masked blocks, a "
                         "two-stage combine, MXFP8 or NVFP4 rows, experts placed by load with copies, or "
                         "routed rows (ids and weights with each row, no permute)")
    ap.add_argument("--spare", type=int, default=4,
                    help="spare copy slots per partition for --variant placed")
    ap.add_argument("--block-rows", type=int, default=0,
                    help="rows per expert block of the masked layout (default S*T)")
    ap.add_argument("--dispatch", choices=["auto", "fused", "separate"], default="auto",
                    help="moe_dispatch (route+layout+pack+permute in one call; the default for "
                         "contiguous bf16 rows) or the four separate calls")
    ap.add_argument("--no-other-workloads", dest="other_workloads", action="store_false",
                    help="skip timing the decode, large and skewed workloads after the headline")
    ap.add_argument("--eager", action="store_true",
                    help="launch the calls from the host every step instead of replaying a CUDA graph")
    ap.add_argument("--profile", action="store_true",
                    help="quiet run for ncu captures (no flush buffers, e2e, clocks or oracle)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.profile:
        return run_profile(args, local)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
