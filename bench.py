#!/usr/bin/env python
"""Benchmark of the DSA decode hot path on GB300.

A step is one pass of the whole path -- latent write (when the workload writes
new rows), indexer scores, top-k, FP8 gather-attend -- over one batch of the
named synthetic workload (default "single": 1 decode row at 32k context, 64
heads, index 32x128, topk 2048).  Inputs are resident in HBM; steps rotate over
enough copies of the inputs (distinct device addresses) that the working set of
a rotation exceeds twice the L2, so every step reads its keys and latent from
HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference     # the FP64 CPU oracle on the host cores
  python bench.py --workload proj_verify   # the K-token verify's batched projections

Under torchrun each rank runs its own copy of the workload on its own GPU
(weak scaling, no data exchange); timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "DSA decode rows/s (index+top-k+FP8 gather-attend) at 32k ctx; % HBM roofline"
UNIT = "rows/s"
DESCRIPTIONS = {
    "tiny": "tiny: 1 row, len 4096, 16 heads x 512 latent FP8 paged (block 64), index 8x64, topk 256",
    "single": "single decode: 1 row, len 32768, 64 heads x 512 latent FP8 paged (block 64), "
              "index 32x128, topk 2048",
    "batched": "batched decode: 32 seqs x 1 row, len U[8192,65536], 64 heads, index 32x128, topk 2048",
    "verify": "K-token verify: 8 seqs x 4 rows (len..len+3), base U[65536,131072], 64 heads, "
              "index 32x128, topk 2048",
    "long": "long-context batch: 64 seqs x 1 row, len log-U[4096,131072], 128 heads, index 64x128, "
            "topk 2048, latent write of the new row",
    "prefill": "prefill selection in one pass: 1 seq x 1024 query rows (lens 7977..9000 of a 9000-token "
               "prompt), 64 heads, index 32x128, topk 2048",
    "index_write": "indexer write side: 4 rows x (wk 128x4096 bf16 out, weights_proj 32x4096 fp32 out, "
                   "LayerNorm with bias + store into a 131072-token key arena), L2 flushed between steps",
    "proj_verify": "K-token verify projections: 4 rows x (q_a and kv_a stacked 2048x4096, absorbed q_b "
                   "32768x1536, absorbed o 4096x32768) bf16, one weight sweep per step",
}
IW_METRIC = ("indexer write rows/s (wk and weights_proj projections, k_norm LayerNorm with bias, "
             "store at the device-side position); % HBM roofline")
PROJ_METRIC = ("K-token verify projection rows/s (q_a, absorbed q_b, kv_a, absorbed o of one layer, "
               "64 heads; one bf16 weight sweep per step); % HBM roofline")
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")
TRAFFIC_NOTE = ("DRAM read+write bytes per launch of the stage's kernels from one ncu capture "
                "with --cache-control none (the merge's reads of the split partials are L2 hits, "
                "as in the chained step); null when the kernel source changed since the capture")


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="single", choices=sorted(DESCRIPTIONS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the batched / verify / long lines of the default run")
    ap.add_argument("--eager", action="store_true", help="launch every step eagerly (no CUDA graph)")
    return ap.parse_args()


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        hi = max(sm)
        loaded = [s for s in sm if s >= 0.5 * hi] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- helpers
def _peaks():
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def _source_hash(name):
    """Hash of a kernel source with its comments and blank space removed, so
    an edit of the comments alone keeps the captured counters valid."""
    p = os.path.join(ROOT, "sparse_attention_mla_dsa_gb300", "csrc", name)
    with open(p, encoding="utf-8") as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    src = "\n".join(ln.strip() for ln in src.splitlines() if ln.strip())
    return hashlib.sha256(src.encode()).hexdigest()[:16]


def _traffic(workload, stage):
    """DRAM bytes (read + write) per launch of a stage from the committed ncu
    table, valid only while the stage's kernel source is unchanged since the
    capture; None otherwise."""
    try:
        with open(TRAFFIC_FILE) as f:
            for ln in f:
                parts = ln.split()
                if not parts or parts[0].startswith("#") or len(parts) < 6:
                    continue
                w, st, src, sha, rd, wr = parts[:6]
                if w == workload and st == stage:
                    if _source_hash(src) != sha:
                        return None
                    return int(rd) + int(wr)
    except (OSError, ValueError):
        return None
    return None


def stage_bytes(wl):
    """Algorithmic bytes per launch of each stage for one step of ``wl``."""
    D = wl.index_dim
    keys = 0
    key_tokens = 0
    for g in range(0, wl.rows, wl.group_rows):
        lmax = int(wl.seq_lens[g:g + wl.group_rows].max())
        keys += lmax * (2 * D + 2)
        key_tokens += lmax
    sel = sum(min(wl.topk, int(L)) for L in wl.seq_lens)
    return {
        "latent_write": wl.rows * (512 * 2 + 512) if wl.has_write else 0,
        "index_scores": keys,
        "select_topk": sum(int(L) * 4 for L in wl.seq_lens) + wl.rows * wl.topk * 4,
        "mla_decode": sel * 512 + wl.rows * 2 * wl.heads * 512 * 2,
    }, key_tokens


# --------------------------------------------------------------------------- our arm
SECONDARY = ("batched", "verify", "long", "prefill")


def config_of(name, wl):
    """The workload's description; both arms print exactly this."""
    return {"workload": DESCRIPTIONS[name], "rows_per_step": wl.rows,
            "algorithmic_bytes_per_step": wl.algorithmic_bytes()}


def time_path(wl, dev, K, warmup, eager, world, api, path, shard):
    """Time K steps of the whole path on resident inputs.

    Steps rotate over enough input replicas (distinct device addresses) that
    one rotation touches more than 2x the L2.  The K timed steps are one CUDA
    graph of K consecutive steps (step s on replica s % n), the form a model
    gives a decode step that runs the path once per layer: the kernels of
    consecutive steps are chained by programmatic dependent launch like the
    stages inside a step.  A second pass replays one graph per step with
    timing events between the stages, for the per-stage breakdown (the event
    nodes serialise the chain, so the stages add up to more than a step)."""
    import torch
    sb, _ = stage_bytes(wl)
    alg_bytes = wl.algorithmic_bytes()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    first = path.DeviceWorkload(wl, dev)
    n_rep = max(2, min(64, math.ceil(2.0 * l2 / max(alg_bytes, 1)) + 1))
    reps = [first] + [first.clone() for _ in range(n_rep - 1)]
    stages = (["latent_write"] if wl.has_write else []) + ["index_scores", "select_topk", "mla_decode"]

    def one_step(dw, evs=None):
        s = torch.cuda.current_stream()
        calls = ([dw.latent_write] if wl.has_write else []) + [lambda: dw.index_scores(inputs_early=True),
                                                               dw.select_topk,
                                                               lambda: dw.mla_decode(q_early=True)]
        if evs is not None:
            evs[0].record(s)
        for j, call in enumerate(calls):
            call()
            if evs is not None:
                evs[j + 1].record(s)

    for i in range(max(3, warmup)):
        one_step(reps[i % n_rep])
    torch.cuda.synchronize()
    code, row, _ = api.dsa_get_error(reset=True)
    if code != 0:
        raise RuntimeError(f"device error during warm-up: {api.DEVERR.get(code)} row {row}")

    run_graph, staged, mode = None, [], "eager"
    if not eager:
        try:
            for dw in reps[:min(K, n_rep)]:
                evs = [torch.cuda.Event(enable_timing=True, external=True)
                       for _ in range(len(stages) + 1)]
                gs = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gs):
                    one_step(dw, evs)
                staged.append((gs, evs))
            run_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(run_graph):
                for i in range(K):
                    one_step(reps[i % n_rep])
            run_graph.replay()                     # untimed warm-up of the timed graph
            torch.cuda.synchronize()
            mode = f"one CUDA graph of the {K} timed steps"
        except (TypeError, RuntimeError) as ex:
            run_graph, staged = None, []
            torch.cuda.synchronize()
            print(f"cuda graph capture unavailable ({ex}); timing eager launches", file=sys.stderr)

    stream = torch.cuda.current_stream()
    eager_evs = None if run_graph is not None else [
        [torch.cuda.Event(enable_timing=True) for _ in range(len(stages) + 1)] for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        start.record(stream)
        if run_graph is not None:
            run_graph.replay()
        else:
            for i in range(K):
                one_step(reps[i % n_rep], eager_evs[i])
        end.record(stream)
        torch.cuda.synchronize()
        if staged:  # second pass: per-stage events (same rotation, same replicas)
            for i in range(K):
                staged[i % len(staged)][0].replay()
            torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = shard.max_over_ranks(start.elapsed_time(end))
    ev_sets = [evs for _, evs in staged] if staged else eager_evs
    stage_ms = {st: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev_sets)
                for j, st in enumerate(stages)}
    code, row, _ = api.dsa_get_error(reset=True)
    if code != 0:
        raise RuntimeError(f"device error during the timed steps: {api.DEVERR.get(code)} row {row}")
    peak, peak_kind = _peaks()
    dominant = max(stages, key=lambda st: stage_ms[st])
    ach = sb[dominant] / (stage_ms[dominant] / 1e3) / 1e9
    # The gather-attend is one kernel, plus a combine kernel when a row's
    # selection is cut into more than one split.
    launches = len(stages) + (1 if api.decode_splits(wl.heads, wl.topk) > 1 else 0)
    del run_graph, staged, reps
    return {"elapsed_ms": elapsed_ms, "stage_ms": stage_ms, "dominant": dominant,
            "achieved": ach, "peak": peak, "peak_kind": peak_kind, "stage_bytes": sb,
            "alg_bytes": alg_bytes, "n_rep": n_rep, "l2": l2, "mode": mode,
            "launches_per_step": launches, "clocks": clk.summary()}


def run_ours(args):
    import torch
    rank, world, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import __graft_entry__
    from sparse_attention_mla_dsa_gb300 import build as _b
    if rank == 0 and _b.is_stale():
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    from sparse_attention_mla_dsa_gb300 import api, path, shard, workloads

    K = args.steps
    wl = workloads.named(args.workload)
    t = time_path(wl, dev, K, args.warmup, args.eager, world, api, path, shard)
    elapsed_ms, stage_ms, dominant = t["elapsed_ms"], t["stage_ms"], t["dominant"]
    value = K * wl.rows * world / (elapsed_ms / 1e3)
    peak = t["peak"]
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": round(t["achieved"], 1),
                "peak": peak, "unit": "GB/s", "frac": round(t["achieved"] / peak, 4),
                "peak_source": t["peak_kind"], "traffic": _traffic(args.workload, dominant),
                "traffic_note": TRAFFIC_NOTE, "algorithmic_bytes": t["stage_bytes"][dominant],
                "stage_ms": {k: round(v, 5) for k, v in stage_ms.items()},
                "path_frac": round(t["alg_bytes"] / (elapsed_ms / K / 1e3) / 1e9 / peak, 4)}

    e2e = None
    if not args.no_e2e:
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        dec = path.DsaDecoder(wl, dev, replicas=t["n_rep"])
        dec.stage(wl)
        # Every replica's step graph is captured on its first use: warm up over
        # all of them so that no capture falls inside the timed steps.
        for i in range(max(3, args.warmup, t["n_rep"])):
            dec.decode()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(K):
            dec.decode()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = shard.max_over_ranks(e0.elapsed_time(e1))
        e2e = {"value": round(K * wl.rows * world / (ems / 1e3), 2), "unit": UNIT,
               "h2d_bytes_per_step": dec.h2d_bytes, "d2h_bytes_per_step": dec.d2h_bytes,
               "launch": "one CUDA graph per step: pinned H2D copy of the step's inputs, "
                         "the path, the output stored into pinned host memory"}
        del dec
        torch.cuda.empty_cache()

    secondary = None
    launches = K * t["launches_per_step"]
    if args.workload == "single" and not args.no_secondary:
        secondary = {}
        for name in SECONDARY:
            w2 = workloads.named(name)
            t2 = time_path(w2, dev, K, args.warmup, args.eager, world, api, path, shard)
            ms = t2["elapsed_ms"] / K
            secondary[name] = {
                "config": config_of(name, w2),
                "value": round(K * w2.rows * world / (t2["elapsed_ms"] / 1e3), 2), "unit": UNIT,
                "ms_per_step": round(ms, 5),
                "path_frac": round(t2["alg_bytes"] / (ms / 1e3) / 1e9 / t2["peak"], 4),
                "stage_ms": {k: round(v, 5) for k, v in t2["stage_ms"].items()},
                "dominant": t2["dominant"], "dominant_frac": round(t2["achieved"] / t2["peak"], 4),
                "traffic": _traffic(name, t2["dominant"]), "clocks": t2["clocks"]}
            launches += K * t2["launches_per_step"]
            del w2
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, rows_target=None)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_of(args.workload, wl),
        "timing": {"l2": f"rotating {t['n_rep']} input replicas at distinct addresses "
                         f"({t['n_rep'] * t['alg_bytes'] / 1e6:.0f} MB of touched inputs per "
                         f"rotation, L2 {t['l2'] / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "launch": t["mode"]},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "secondary": secondary,
        "gpu_launches": launches, "clocks": t["clocks"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# --------------------------------------------------------------------------- projections
def _proj_oracle_rows_per_s(pw, rows, threads):
    """The oracle's batched projection, every projection of the set, for the
    given activation rows (one task per row and projection)."""
    import numpy as np
    import oracle
    tasks = [(j, r) for r in rows for j in range(len(pw.shapes))]

    def one(t):
        j, r = t
        oracle.dense_mm(np.ascontiguousarray(pw.acts[j][r:r + 1]), pw.weights[j])

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(one, tasks))
    return len(rows) / (time.perf_counter() - t0)


def run_projections(args):
    """One step = one layer's four projections (q_a and kv_a stacked, they share
    the layer input) for the 4 rows of a K-token verify, each weight swept once
    (dsa_dense_mm_bf16, bf16 out)."""
    import torch
    rank, world, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    import __graft_entry__
    from sparse_attention_mla_dsa_gb300 import build as _b
    if rank == 0 and _b.is_stale():
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    from sparse_attention_mla_dsa_gb300 import api, shard, workloads
    api.load()
    pw = workloads.make_projections()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    wbytes = pw.weight_bytes()
    alg = pw.algorithmic_bytes()
    n_rep = max(2, math.ceil(2.0 * l2 / wbytes) + 1)
    names = [nm for nm, _, _ in pw.shapes]

    def dev16(a):
        return torch.from_numpy(a.view("int16")).to(dev)

    weights = [dev16(w) for w in pw.weights]
    reps = []
    for i in range(n_rep):
        ws = weights if i == 0 else [w.clone() for w in weights]
        acts = [dev16(a) for a in pw.acts]
        outs = [torch.empty((pw.rows, n), dtype=torch.int16, device=dev) for _, n, _ in pw.shapes]
        wsp = [torch.empty(max(256, api.dsa_dense_mm_workspace_bytes(n, k)), dtype=torch.uint8,
                           device=dev) for _, n, k in pw.shapes]
        reps.append((ws, acts, outs, wsp))

    def one_step(rep, evs=None):
        ws, acts, outs, wsp = rep
        s = torch.cuda.current_stream()
        if evs is not None:
            evs[0].record(s)
        for j in range(len(ws)):
            api.dsa_dense_mm_bf16(acts[j], ws[j], outs[j], wsp[j])
            if evs is not None:
                evs[j + 1].record(s)

    for i in range(max(3, args.warmup)):
        one_step(reps[i % n_rep])
    torch.cuda.synchronize()
    code, row, _ = api.dsa_get_error(reset=True)
    if code != 0:
        raise RuntimeError(f"device error during warm-up: {api.DEVERR.get(code)} ({row})")
    graphs, staged = [], []
    for rep in reps:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            one_step(rep)
        graphs.append(g)
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(names) + 1)]
        gs = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gs):
            one_step(rep, evs)
        staged.append((gs, evs))
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()

    K = args.steps
    stream = torch.cuda.current_stream()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        start.record(stream)
        for i in range(K):
            graphs[i % n_rep].replay()
        end.record(stream)
        torch.cuda.synchronize()
        for i in range(K):
            staged[i % n_rep][0].replay()
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    elapsed_ms = shard.max_over_ranks(start.elapsed_time(end))
    ev_sets = [evs for _, evs in staged[:min(K, n_rep)]]
    stage_ms = {nm: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in ev_sets)
                for j, nm in enumerate(names)}
    code, row, _ = api.dsa_get_error(reset=True)
    if code != 0:
        raise RuntimeError(f"device error during the timed steps: {api.DEVERR.get(code)} ({row})")

    value = K * pw.rows * world / (elapsed_ms / 1e3)
    peak, peak_kind = _peaks()
    stage_bytes = {nm: n * k * 2 + pw.rows * (n + k) * 2 for nm, n, k in pw.shapes}
    dominant = max(names, key=lambda nm: stage_ms[nm])
    ach = stage_bytes[dominant] / (stage_ms[dominant] / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": round(ach, 1), "peak": peak,
                "unit": "GB/s", "frac": round(ach / peak, 4), "peak_source": peak_kind,
                "traffic": _traffic(args.workload, dominant), "algorithmic_bytes": stage_bytes[dominant],
                "stage_ms": {k: round(v, 5) for k, v in stage_ms.items()},
                "path_frac": round(alg / (elapsed_ms / K / 1e3) / 1e9 / peak, 4)}

    e2e = None
    if not args.no_e2e:
        # Host-facing: the step's activations from pinned host memory, the four
        # projections, the outputs back to pinned host memory, one graph per replica.
        h_in = [torch.from_numpy(a.view("int16")).pin_memory() for a in pw.acts]
        h_out = [torch.empty((pw.rows, n), dtype=torch.int16).pin_memory() for _, n, _ in pw.shapes]

        def host_step(rep):
            ws, acts, outs, wsp = rep
            for j in range(len(ws)):
                acts[j].copy_(h_in[j], non_blocking=True)
            one_step(rep)
            for j in range(len(ws)):
                h_out[j].copy_(outs[j], non_blocking=True)

        hgraphs = []
        for rep in reps:
            host_step(rep)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                host_step(rep)
            hgraphs.append(g)
        for g in hgraphs:
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(K):
            hgraphs[i % n_rep].replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ems = shard.max_over_ranks(e0.elapsed_time(e1))
        e2e = {"value": round(K * pw.rows * world / (ems / 1e3), 2), "unit": UNIT,
               "h2d_bytes_per_step": sum(t.numel() * 2 for t in h_in),
               "d2h_bytes_per_step": sum(t.numel() * 2 for t in h_out)}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cores = os.cpu_count() or 1
        v = _proj_oracle_rows_per_s(pw, list(range(pw.rows)), cores)
        cpu = {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{pw.rows} rows x the projections, one (row, projection) per "
                         f"task over {cores} threads"}
    launches = sum(1 + (1 if api.dsa_dense_mm_workspace_bytes(n, k) > 0 else 0)
                   for _, n, k in pw.shapes)
    line = {
        "metric": PROJ_METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / K, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[args.workload], "rows_per_step": pw.rows,
                   "algorithmic_bytes_per_step": alg},
        "timing": {"l2": f"rotating {n_rep} weight replicas ({n_rep * wbytes / 1e6:.0f} MB per "
                         f"rotation, L2 {l2 / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "launch": "one CUDA graph per step"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": K * launches, "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_projections_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return
    from sparse_attention_mla_dsa_gb300 import workloads
    import oracle
    oracle.build()
    pw = workloads.make_projections()
    cores = os.cpu_count() or 1
    K = args.steps
    t0 = time.perf_counter()
    for _ in range(K):
        _proj_oracle_rows_per_s(pw, list(range(pw.rows)), cores)
    el = time.perf_counter() - t0
    value = K * pw.rows / el
    sample = f"{K} steps x {pw.rows} rows x the projections over {cores} threads"
    line = {"impl": "reference", "metric": PROJ_METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(el / K * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": DESCRIPTIONS[args.workload], "rows_per_step": pw.rows,
                       "algorithmic_bytes_per_step": pw.algorithmic_bytes()},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- indexer write side
IW_ROWS, IW_HIDDEN, IW_DIM, IW_HEADS, IW_TOKENS = 4, 4096, 128, 32, 131072


def _iw_inputs(seed=6):
    """Synthetic inputs of the indexer write step (weights_proj carries the
    index_heads^-0.5 scale, folded in as the pages fold it at load)."""
    import numpy as np
    from sparse_attention_mla_dsa_gb300 import workloads
    rng = np.random.default_rng(seed)
    f32 = np.float32
    hidden = workloads._bf16_bits(rng.standard_normal((IW_ROWS, IW_HIDDEN), dtype=f32))
    wk = workloads._bf16_bits(rng.standard_normal((IW_DIM, IW_HIDDEN), dtype=f32) / f32(IW_HIDDEN ** 0.5))
    wp = workloads._bf16_bits(rng.standard_normal((IW_HEADS, IW_HIDDEN), dtype=f32)
                              / f32(IW_HIDDEN ** 0.5) * f32(IW_HEADS ** -0.5))
    ln_w = workloads._bf16_bits(1.0 + 0.1 * rng.standard_normal(IW_DIM, dtype=f32))
    ln_b = workloads._bf16_bits(0.1 * rng.standard_normal(IW_DIM, dtype=f32))
    lens = rng.integers(IW_TOKENS // 8, IW_TOKENS // IW_ROWS, size=IW_ROWS)
    base = np.arange(IW_ROWS, dtype=np.int64) * (IW_TOKENS // IW_ROWS)
    return hidden, wk, wp, ln_w, ln_b, lens.astype(np.int32), base


def _iw_bytes():
    w = (IW_DIM + IW_HEADS) * IW_HIDDEN * 2
    return w + IW_ROWS * (IW_HIDDEN * 2 + IW_DIM * 2 * 2 + IW_DIM * 2 + IW_HEADS * 4)


def run_indexer_write(args):
    """One step = the indexer write side of 4 rows: the wk projection (bf16
    out) and the weights_proj projection (FP32 out, the head weights S1 reads)
    by dsa_dense_mm_bf16, then dsa_indexer_write.  The step's data is small
    and L2-resident, so L2 is flushed (a 2 x L2 buffer written) before every
    timed step and each step is timed on its own events."""
    import numpy as np
    import torch
    rank, world, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    import __graft_entry__
    from sparse_attention_mla_dsa_gb300 import build as _b
    if rank == 0 and _b.is_stale():
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    from sparse_attention_mla_dsa_gb300 import api, shard
    api.load()
    hidden, wk, wp, ln_w, ln_b, lens, base = _iw_inputs()
    d16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)
    t_hidden, t_wk, t_wp, t_lw, t_lb = d16(hidden), d16(wk), d16(wp), d16(ln_w), d16(ln_b)
    k_raw = torch.empty((IW_ROWS, IW_DIM), dtype=torch.int16, device=dev)
    head_w = torch.empty((IW_ROWS, IW_HEADS), dtype=torch.float32, device=dev)
    arena = torch.zeros((IW_TOKENS, IW_DIM), dtype=torch.int16, device=dev)
    ws1 = torch.empty(max(256, api.dsa_dense_mm_workspace_bytes(IW_DIM, IW_HIDDEN)), dtype=torch.uint8, device=dev)
    ws2 = torch.empty(max(256, api.dsa_dense_mm_workspace_bytes(IW_HEADS, IW_HIDDEN)), dtype=torch.uint8, device=dev)
    seq_lens = torch.from_numpy(lens).to(dev)
    positions = (seq_lens - 1).to(torch.int32)
    idx_base = torch.from_numpy(base).to(dev)
    rows = api.make_rows(seq_lens, positions=positions)

    def step():
        api.dsa_dense_mm_bf16(t_hidden, t_wk, k_raw, ws1)
        api.dsa_dense_mm_bf16(t_hidden, t_wp, head_w, ws2)
        api.dsa_indexer_write(rows, k_raw, t_lw, t_lb, 1e-6, idx_base, arena)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if api.dsa_get_error(reset=True)[0] != 0:
        raise RuntimeError("device error during warm-up")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    K = args.steps
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for i in range(K):
            flush.fill_(i & 0xFF)
            evs[i][0].record(stream)
            g.replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
    step_ms = shard.max_over_ranks(sum(a.elapsed_time(b) for a, b in evs) / K)
    if api.dsa_get_error(reset=True)[0] != 0:
        raise RuntimeError("device error during the timed steps")
    value = IW_ROWS * world / (step_ms / 1e3)
    peak, peak_kind = _peaks()
    alg = _iw_bytes()
    ach = alg / (step_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "index_write step", "achieved": round(ach, 1), "peak": peak,
                "unit": "GB/s", "frac": round(ach / peak, 4), "peak_source": peak_kind, "traffic": None,
                "algorithmic_bytes": alg}
    e2e = None
    if not args.no_e2e:
        h_in = torch.from_numpy(hidden.view(np.int16)).pin_memory()
        h_out = torch.empty((IW_ROWS, IW_HEADS), dtype=torch.float32).pin_memory()

        def host_step():
            t_hidden.copy_(h_in, non_blocking=True)
            step()
            h_out.copy_(head_w, non_blocking=True)

        host_step()
        torch.cuda.synchronize()
        hg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(hg):
            host_step()
        hevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush.fill_(i & 0xFF)
            hevs[i][0].record(stream)
            hg.replay()
            hevs[i][1].record(stream)
        torch.cuda.synchronize()
        ems = shard.max_over_ranks(sum(a.elapsed_time(b) for a, b in hevs) / K)
        e2e = {"value": round(IW_ROWS * world / (ems / 1e3), 2), "unit": UNIT,
               "h2d_bytes_per_step": h_in.numel() * 2, "d2h_bytes_per_step": h_out.numel() * 4}
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        v, cores = _iw_oracle_rows_per_s(1)
        cpu = {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": f"{IW_ROWS} rows: both projections and the norm, one task per row"}
    launches = 3 + sum(1 for n in (IW_DIM, IW_HEADS) if api.dsa_dense_mm_workspace_bytes(n, IW_HIDDEN) > 0)
    line = {
        "metric": IW_METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[args.workload], "rows_per_step": IW_ROWS,
                   "algorithmic_bytes_per_step": alg},
        "timing": {"l2": f"flushed before every step (a {2 * l2 / 1e6:.0f} MB buffer written)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "launch": "one CUDA graph per step"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": K * launches,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def _iw_oracle_rows_per_s(reps):
    import numpy as np
    import oracle
    oracle.build()
    hidden, wk, wp, ln_w, ln_b, lens, base = _iw_inputs()
    cores = os.cpu_count() or 1

    def one(r):
        row = np.ascontiguousarray(hidden[r:r + 1])
        c, _ = oracle.dense_mm(row, wk)
        oracle.dense_mm(row, wp)
        from sparse_attention_mla_dsa_gb300 import workloads
        oracle.layer_norm_row(workloads._bf16_bits(c[0]), ln_w, ln_b, 1e-6)

    rows = [r % IW_ROWS for r in range(reps * IW_ROWS)]
    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=cores) as ex:
        list(ex.map(one, rows))
    return len(rows) / (time.perf_counter() - t0), cores


def run_indexer_write_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return
    v, cores = _iw_oracle_rows_per_s(max(1, args.steps))
    line = {"impl": "reference", "metric": IW_METRIC, "value": round(v, 4), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(IW_ROWS / v * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": DESCRIPTIONS[args.workload], "rows_per_step": IW_ROWS,
                                            "algorithmic_bytes_per_step": _iw_bytes()},
            "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{args.steps} steps x {IW_ROWS} rows over {cores} threads"},
            "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- oracle (CPU)
def _oracle_rows_per_s(wl, rows, threads):
    import oracle

    t0 = time.perf_counter()
    oracle.run_path_rows(wl, rows=rows, threads=threads)
    return len(rows) / (time.perf_counter() - t0)


def cpu_baseline(wl, rows_target=None):
    """The oracle as it stands, rows in parallel over the host cores, on a
    bounded sample of the workload's rows (about 10-30 s of CPU work)."""
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    n = rows_target or max(1, min(2 * cores, 64))
    rows = [i % wl.rows for i in range(n)]
    v = _oracle_rows_per_s(wl, rows, cores)
    return {"value": round(v, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} rows of the same workload (index over the full context, full-sort "
                      f"top-k, gather-attend), rows spread over {cores} threads"}


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return
    from sparse_attention_mla_dsa_gb300 import workloads
    wl = workloads.named(args.workload)
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    for i in range(args.warmup):
        _oracle_rows_per_s(wl, [i % wl.rows], 1)
    # one step = one batch of rows; rows of the timed steps run over all cores
    K = args.steps
    rows_per_step = min(wl.rows, 4)
    rows = [i % wl.rows for i in range(K * rows_per_step)]
    t0 = time.perf_counter()
    import oracle as o
    o.run_path_rows(wl, rows=rows, threads=cores)
    el = time.perf_counter() - t0
    value = len(rows) / el
    sample = (f"{K} steps, each a bounded sample of {rows_per_step} of the workload's {wl.rows} "
              f"rows (index over the full context, full-sort top-k, gather-attend), rows over "
              f"{cores} threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": round(el / K * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(args.workload, wl),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = _args()
    if args.impl == "reference":
        if args.steps > 20:
            args.steps = 20     # the oracle is slow; keep the run within minutes
        if args.workload == "proj_verify":
            run_projections_reference(args)
        elif args.workload == "index_write":
            run_indexer_write_reference(args)
        else:
            run_reference(args)
    elif args.workload == "proj_verify":
        run_projections(args)
    elif args.workload == "index_write":
        run_indexer_write(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
