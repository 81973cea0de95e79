#!/usr/bin/env python
"""Benchmark of the UniPrefill token-selection path on one GB300 (or N replicas).

One step = one call of ``upf_select_tokens`` (score pass 1, score pass 2,
finalize + block means, top-p select, compaction, drop-history append) over one
batch of seeded synthetic inputs already resident in HBM.  Metric: prompt tokens
scored + selected + compacted per second.  The default workload is the 128K
LLaMA-3.1-8B-shaped full-attention layer (1 request, L=131072, H_q=32, H_kv=8,
d=128, hidden 4096, n=128, G=64, p=0.99).

Prints one JSON line (rank 0).  ``--impl reference`` times the float64 CPU
oracle on the host cores instead (the baseline arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from sparse_long_context_tail_gb300 import workload as wl  # noqa: E402

METRIC = "prompt tokens scored+selected+compacted/sec at 128K"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = "llama8b-L131072"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STAGES = ["describe", "score_pass1", "score_pass2", "finalize", "select", "compact_count", "compact_index",
          "compact_gather"]
# kernel sources per stage (for the traffic record's freshness check): the
# translation unit of the kernel the fused call launches plus the headers it
# includes from the package
_TC = ["score_tc.cu", "score_common.cuh", "sm100_ptx.cuh", "upf_internal.cuh"]
_TAIL = ["tail.cu", "select_core.cuh", "upf_internal.cuh"]
STAGE_SOURCES = {"score_pass1": _TC, "score_pass2": _TC, "finalize": _TAIL, "select": _TAIL,
                 "compact_gather": _TAIL, "compact_index": ["compact.cu", "upf_internal.cuh"],
                 "compact_count": ["compact.cu", "upf_internal.cuh"],
                 "describe": ["score_simt.cu", "upf_internal.cuh"]}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=wl.NAMED)
    ap.add_argument("--top-p", type=float, default=None, help="override p (e.g. 1.0 keeps every token)")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--stack", action="store_true",
                    help="instead of the bench line: a synthetic stack of later layers on the kept tokens")
    ap.add_argument("--stack-layers", type=int, default=48,
                    help="layers in the synthetic stack (48: a multiple of both schedules' periods)")
    ap.add_argument("--no-graph", action="store_true", help="skip timing the step replayed from a CUDA graph")
    ap.add_argument("--no-gather-p1", action="store_true", help="skip the supplementary all-kept gather point")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-flush", action="store_true", help="do not flush L2 between steps")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the other benchmark workloads after the headline one")
    ap.add_argument("--tp", action="store_true",
                    help="tensor-parallel mode: heads sharded over the ranks, one score all-reduce per step")
    return ap.parse_args()


# ------------------------------------------------------------ work counts ----

def algorithmic_work(spec, cu, kept_total, row_bytes, top_p):
    """Algorithmic flops / bytes per launch of each stage (what the method must do)."""
    H_q, H_kv, d, n = spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.n_tail
    L = np.diff(np.asarray(cu, dtype=np.int64))
    T = int(L.sum())
    vis = 0          # sum over requests and tail queries of visible keys (t_j + 1)
    for x in L:
        n_eff = min(n, int(x))
        vis += n_eff * int(x) - n_eff * (n_eff - 1) // 2
    flops_pass = 2.0 * d * H_q * vis
    k_bytes = 2.0 * T * H_kv * d
    q_bytes = 2.0 * H_q * d * sum(min(n, int(x)) for x in L)
    nb = sum(-(-int(x) // spec.block) for x in L)
    P = H_kv * max(1, math.ceil(H_q // H_kv * n / 512))
    return {
        "score_pass1": dict(bound="tensor", flops=flops_pass, bytes=k_bytes + q_bytes),
        "score_pass2": dict(bound="tensor", flops=flops_pass, bytes=k_bytes + q_bytes + 4.0 * P * T),
        "finalize": dict(bound="hbm", bytes=4.0 * P * T + 4.0 * T + 4.0 * nb + T / 8),
        "select": dict(bound="latency", bytes=4.0 * nb + T / 8),
        "compact_count": dict(bound="latency", bytes=T / 8),
        "compact_index": dict(bound="latency", bytes=T / 8 + 4.0 * kept_total),
        "compact_gather": dict(bound="hbm", bytes=kept_total * (2.0 * row_bytes + 32.0 + 4.0)),
        "describe": dict(bound="latency", bytes=0.0),
    }


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(stage):
    """First 16 hex digits of the SHA-256 of the stage's sources, concatenated."""
    files = STAGE_SOURCES.get(stage)
    if not files:
        return None
    h = hashlib.sha256()
    for name in files:
        src = os.path.join(ROOT, "sparse_long_context_tail_gb300", "csrc", name)
        if not os.path.isfile(src):
            return None
        with open(src, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record(stage, workload):
    """DRAM bytes per launch from a committed ncu summary, if it is still current."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            rec = json.load(f)
        r = rec.get(stage)
        sha = source_sha(stage)
        if r and sha is not None and r.get("workload") == workload and r.get("source_sha") == sha:
            return float(r["dram_bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        return None
    return None


# ------------------------------------------------------------- multi-GPU ----

def rank_spec(spec, rank):
    """The requests rank `rank` processes: the same workload shape with its own seed.

    Requests are independent, so N GPUs each take their own batch (weak
    scaling) and exchange nothing on the data path."""
    import dataclasses
    return spec if rank == 0 else dataclasses.replace(spec, seed=spec.seed + 100 * rank)


def aggregate_over_ranks(seconds_per_step, tokens, dist_mod=None, device=None):
    """Whole-job rate: units of all ranks / the slowest rank's step time.

    Returns (max seconds per step, total tokens per step, tokens/s)."""
    if dist_mod is not None and dist_mod.is_available() and dist_mod.is_initialized() and \
            dist_mod.get_world_size() > 1:
        import torch
        t = torch.tensor([float(seconds_per_step)], dtype=torch.float64, device=device)
        n = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
        dist_mod.all_reduce(t, op=dist_mod.ReduceOp.MAX)
        dist_mod.all_reduce(n, op=dist_mod.ReduceOp.SUM)
        seconds_per_step, tokens = float(t.item()), float(n.item())
    return seconds_per_step, tokens, tokens / seconds_per_step


# ----------------------------------------------------------------- clocks ----

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------ CPU oracle ----

def oracle_run(w, threads=None):
    """One whole pass of the float64 oracle over the workload.

    Returns (score seconds, rest seconds, threads used)."""
    import oracle
    s = w.spec
    thr = threads or min(32, os.cpu_count() or 1)
    t0 = time.perf_counter()
    scores = oracle.token_scores(w.k_bits, w.q_tail_bits, w.cu_seqlens, s.num_q_heads, s.num_kv_heads,
                                 s.head_dim, s.n_tail, None, s.kv_of_q, thr)
    t1 = time.perf_counter()
    sel = oracle.select(scores, w.cu_seqlens, s.block, s.top_p, s.sink_keep, s.tail_keep)
    oracle.compact(sel["mask"], w.cu_seqlens, w.hidden_bits(), w.positions(), w.slots(), 0)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1, thr


def cpu_baseline(w, budget_s=15.0):
    """Time the oracle as it stands on the host cores: whole passes until ~budget_s elapse (max 3)."""
    runs = []
    thr = None
    t_start = time.perf_counter()
    while len(runs) < 3:
        ts, tr, thr = oracle_run(w)
        runs.append(ts + tr)
        if time.perf_counter() - t_start > budget_s:
            break
    per = statistics.median(runs)
    return {"value": w.total_tokens / per, "unit": UNIT, "cores": thr, "kind": "oracle",
            "sample": f"{len(runs)} full pass(es) of the float64 oracle over the whole workload "
                      f"({w.spec.name}, {w.total_tokens} tokens, all {w.spec.num_q_heads} q-heads); "
                      f"median {per:.2f} s per pass"}


def run_reference(args):
    """The baseline arm: the float64 oracle as it stands, whole passes over the
    workload on the host cores (each step is one complete pass: scores of
    every q-head and tail query, block means, top-p + exempt mask, compaction
    with the hidden rows, positions and slots)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    spec = wl.named_spec(args.workload)
    if args.top_p is not None:
        spec.top_p = args.top_p
    w = wl.generate(spec)
    w.hidden_bits()
    thr = None
    for _ in range(args.warmup):
        oracle_run(w)
    per_step = []
    for _ in range(args.steps):
        ts, tr, thr = oracle_run(w)
        per_step.append(ts + tr)
    per = statistics.mean(per_step)
    value = w.total_tokens / per
    sample = (f"each step: one whole pass of the float64 oracle over {spec.name} ({w.total_tokens} tokens, all "
              f"{spec.num_q_heads} q-heads and {spec.n_tail} tail queries, selection and compaction); "
              f"{args.steps} timed passes after {args.warmup} untimed, mean {per:.2f} s per pass")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(spec, w, args), "gpu_launches": 0,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_of(spec, w, args):
    tp_mode = getattr(args, "tp", False)
    return {"workload": spec.name, "requests": len(spec.lengths), "total_tokens": w.total_tokens,
            "num_q_heads": spec.num_q_heads, "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim,
            "hidden": spec.hidden, "n_tail": spec.n_tail, "block": spec.block, "top_p": spec.top_p,
            "sink_keep": spec.sink_keep, "tail_keep": spec.tail_keep,
            "l2": "flushed between steps (512 MiB write)" if not args.no_flush else "not flushed",
            "parallelism": (f"tp{args.gpus} (heads sharded over ranks, one sum all-reduce of the fp32 scores)"
                            if tp_mode else f"replicas x{args.gpus} (requests sharded per GPU, no collective)")}


# -------------------------------------------------------------- rooflines ----

def scoring_bound(work_stage, peaks):
    """'tensor' when the pass's arithmetic intensity (flop per DRAM byte of K
    and tail Q) is above the ridge of the measured peaks, else 'hbm'."""
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    return "tensor" if work_stage["flops"] / max(1.0, work_stage["bytes"]) >= ridge else "hbm"


def kernel_roofline(stage, work, sec_per_launch, peaks, peak_kind, workload_name):
    """Roofline entry of one kernel: algorithmic work per launch / its mean
    launch time, against the measured peak of the unit that bounds it.

    The scoring passes are timed alone (one launch of well under a
    millisecond), so a tensor-bound pass takes the burst bf16 peak; the
    sustained figure is given beside it, labelled."""
    wk = work[stage]
    if stage in ("score_pass1", "score_pass2"):
        bound = scoring_bound(wk, peaks)
    else:
        bound = "hbm"
    if bound == "tensor":
        achieved = wk["flops"] / sec_per_launch / 1e12
        peak, unit, key = peaks["bf16_tflops"], "TFLOP/s", "bf16_tflops"
    else:
        achieved = wk["bytes"] / sec_per_launch / 1e9
        peak, unit, key = peaks["hbm_gbs"], "GB/s", "hbm_gbs"
    r = {"bound": bound, "kernel": stage, "achieved": achieved, "peak": peak, "unit": unit,
         "frac": achieved / peak, "peak_source": f"{peak_kind} {key}" + (" (burst)" if bound == "tensor" else ""),
         "traffic": traffic_record(stage, workload_name), "us_per_launch": sec_per_launch * 1e6,
         "algorithmic_bytes_per_launch": wk["bytes"]}
    if "flops" in wk:
        r["algorithmic_flops_per_launch"] = wk["flops"]
        r["tflops"] = wk["flops"] / sec_per_launch / 1e12
        r["gbs"] = wk["bytes"] / sec_per_launch / 1e9
        if bound == "tensor" and "bf16_tflops_sustained" in peaks:
            r["frac_of_sustained_peak"] = achieved / peaks["bf16_tflops_sustained"]
    return r


# ------------------------------------------------------------ one workload ----

class DeviceInputs:
    """A workload's inputs resident in HBM (the tail Q rows inside a [T, H_q, d]
    tensor, K, hidden rows, positions, slot ids, cu_seqlens)."""

    def __init__(self, torch, w, dev, hidden_from_host=True):
        spec = w.spec
        T = w.total_tokens
        self.q = torch.zeros((T, spec.num_q_heads, spec.head_dim), dtype=torch.bfloat16, device=dev)
        q_tail = torch.from_numpy(w.q_tail_bits.view(np.int16)).view(torch.bfloat16)
        self.q[torch.from_numpy(w.tail_rows).to(dev)] = q_tail.to(dev)
        self.k = torch.from_numpy(w.k_bits.view(np.int16)).to(dev).view(torch.bfloat16)
        if hidden_from_host:
            self.hidden = torch.from_numpy(w.hidden_bits().view(np.int16)).to(dev)
        else:   # contents do not affect the path (bit-copied rows): device zeros, no host generation
            self.hidden = torch.zeros((T, spec.hidden), dtype=torch.int16, device=dev)
        self.pos = torch.from_numpy(w.positions()).to(dev)
        self.slot = torch.from_numpy(w.slots()).to(dev)
        self.cu = torch.from_numpy(w.cu_seqlens).to(dev)


LEAD_CYCLES = 400000   # ~0.2 ms of GPU sleep before each timed step


def timed_loop(torch, fn, stream, steps, flush, lead_cycles=LEAD_CYCLES):
    """Per-step device ms of `steps` calls of fn, CUDA events on `stream`, L2
    flushed between steps (outside the events).

    Before each step's start event the stream sleeps for `lead_cycles` GPU
    cycles (a bounded sleep kernel): meanwhile the host enqueues the step, so
    the events time the step's kernels on the device rather than the host's
    launch path catching up with an idle GPU (the end-to-end figure carries
    the host path)."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        if lead_cycles:
            torch.cuda._sleep(lead_cycles)
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
        if flush is not None:
            flush.zero_()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def traced_loop(torch, B, sel, fn, stream, steps, flush):
    """The same steps with an event pair around every launch (library tracing):
    per-stage launches and summed ms, plus the traced step times."""
    B.upf_profile_read(sel.ctx)
    B.upf_profile_enable(sel.ctx, True)
    traced = timed_loop(torch, fn, stream, steps, flush)
    launches, stage_ms = B.upf_profile_read(sel.ctx)
    B.upf_profile_enable(sel.ctx, False)
    return launches, stage_ms, traced


def stage_table(work, launches, stage_ms):
    tot_ms = sum(stage_ms) or 1.0
    stages = {}
    for i, nm in enumerate(STAGES):
        n_l = max(1, launches[i])
        per = stage_ms[i] / n_l
        entry = {"launches": launches[i], "ms_per_launch": per, "share": stage_ms[i] / tot_ms}
        wk = work[nm]
        if per > 0:
            if "flops" in wk:
                entry["tflops"] = wk["flops"] / (per / 1e3) / 1e12
            entry["gbs"] = wk["bytes"] / (per / 1e3) / 1e9
        stages[nm] = entry
    return stages


def run_per_config(torch, B, sel, names, dev, stream, flush, peaks, peak_kind, steps=10, warmup=3):
    """tokens/s, per-stage us and the scoring passes' roofline fractions of the
    other benchmark workloads (the headline line measures only its own).
    Inputs are the seeded workloads (hidden rows are device zeros: the path
    bit-copies them, so their values change nothing but are never read as
    numbers)."""
    out = {}
    for name in names:
        t0 = time.time()
        spec = wl.named_spec(name)
        w = wl.generate(spec)
        x = DeviceInputs(torch, w, dev, hidden_from_host=False)
        cu = w.cu_seqlens
        params = B.make_params(spec.n_tail, spec.block, spec.sink_keep, spec.tail_keep, spec.top_p)
        o = sel.alloc_outputs(cu, spec.block, x.hidden, x.pos, x.slot)

        def step(o=o, x=x, spec=spec, cu=cu, params=params):
            return sel.select_tokens(x.q, x.k, cu, x.cu, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                                     x.hidden, x.pos, x.slot, layer_id=0, params=params, kv_of_q=spec.kv_of_q,
                                     out=o)

        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
        status = sel.status()
        kept = int(o.total_kept.item())
        ms = timed_loop(torch, step, stream, steps, flush)
        launches, stage_ms, _ = traced_loop(torch, B, sel, step, stream, steps, flush)
        graph = graph_replay(torch, step, stream, steps, flush)
        T = w.total_tokens
        work = algorithmic_work(spec, cu, kept, x.hidden.stride(0) * 2, spec.top_p)
        # median over the steps: one step delayed by the host (a rare stall of
        # a millisecond or more) must not stand for the workload
        entry = {"tokens": T, "requests": len(spec.lengths), "ms_per_step": statistics.median(ms),
                 "mean_ms": statistics.mean(ms), "tokens_per_s": T / (statistics.median(ms) / 1e3),
                 "graph_ms_per_step": graph["median_ms"], "kept_tokens": kept, "kept_fraction": kept / T,
                 "status": B.STATUS_NAMES.get(status, status),
                 "stage_us": {nm: 1e3 * stage_ms[i] / max(1, launches[i]) for i, nm in enumerate(STAGES)
                              if launches[i]},
                 "stage_sum_us": 1e3 * sum(stage_ms) / steps}
        for nm in ("score_pass1", "score_pass2"):
            i = STAGES.index(nm)
            if launches[i] and stage_ms[i] > 0:
                rf = kernel_roofline(nm, work, stage_ms[i] / launches[i] / 1e3, peaks, peak_kind, name)
                entry[nm] = {k: rf[k] for k in ("bound", "achieved", "unit", "frac", "tflops", "gbs",
                                                "us_per_launch")}
        out[name] = entry
        log(f"[bench] per-config {name}: {entry['ms_per_step'] * 1e3:.1f} us/step "
            f"({time.time() - t0:.1f} s incl. generation)")
        del x, o, w
        torch.cuda.empty_cache()
    return out


PER_CONFIG = ["small-L4096", "llama8b-L32768", "llama8b-batch16"] + list(wl.SWEEP_NAMES)


# ----------------------------------------------------------------- ours -----

def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.stack:
        return run_stack(args)
    if args.tp:
        return run_tp(args)
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from sparse_long_context_tail_gb300 import _binding as B
    from sparse_long_context_tail_gb300.selector import TokenSelector

    spec = rank_spec(wl.named_spec(args.workload), rank)
    if args.top_p is not None:
        spec.top_p = args.top_p
    t0 = time.time()
    w = wl.generate(spec)
    w.hidden_bits()
    log(f"[bench] generated {spec.name} in {time.time() - t0:.1f} s")
    cu = w.cu_seqlens
    T = w.total_tokens
    params = B.make_params(spec.n_tail, spec.block, spec.sink_keep, spec.tail_keep, spec.top_p)

    x = DeviceInputs(torch, w, dev)          # inputs resident in HBM
    q_dev, k_dev, hid_dev, pos_dev, slot_dev, cu_dev = x.q, x.k, x.hidden, x.pos, x.slot, x.cu
    sel = TokenSelector(local)
    out = sel.alloc_outputs(cu, spec.block, hid_dev, pos_dev, slot_dev)
    flush = None if args.no_flush else torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def step(o=out):
        return sel.select_tokens(q_dev, k_dev, cu, cu_dev, spec.num_q_heads, spec.num_kv_heads, spec.head_dim,
                                 hid_dev, pos_dev, slot_dev, layer_id=0, params=params, kv_of_q=spec.kv_of_q,
                                 out=o)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    status = sel.status()
    if status != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES.get(status)} during warm-up")
    kept_total = int(out.total_kept.item())

    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    B.upf_profile_read(sel.ctx)          # reset counters
    # Headline loop: tracing off, so consecutive kernels of a step overlap
    # their launch with the predecessor's tail (programmatic dependent launch).
    wall0 = time.perf_counter()
    step_ms = timed_loop(torch, step, stream, args.steps, flush)
    wall = time.perf_counter() - wall0
    launches, _ = B.upf_profile_read(sel.ctx)
    # Breakdown loop: the same steps with an event pair around every launch.
    _, stage_ms, traced = traced_loop(torch, B, sel, step, stream, args.steps, flush)
    # The same step captured once in a CUDA graph and replayed (launches keep
    # their programmatic-dependent-launch edges inside the graph).
    graph = None
    if not args.no_graph:
        graph = graph_replay(torch, step, stream, args.steps, flush)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    sec, _, value = aggregate_over_ranks(statistics.mean(step_ms) / 1e3, T, dist if world > 1 else None, dev)
    ms = sec * 1e3

    # roofline of the dominant kernel (largest share of device time), and of both scoring passes
    work = algorithmic_work(spec, cu, kept_total, hid_dev.stride(0) * 2, spec.top_p)
    peaks, peak_kind = load_peaks()
    stages = stage_table(work, launches, stage_ms)
    dom = max(range(len(STAGES)), key=lambda i: stage_ms[i])
    roofline = kernel_roofline(STAGES[dom], work, stage_ms[dom] / max(1, launches[dom]) / 1e3, peaks, peak_kind,
                               spec.name)
    roofline["passes"] = {}
    for nm in ("score_pass1", "score_pass2"):
        i = STAGES.index(nm)
        if launches[i]:
            roofline["passes"][nm] = kernel_roofline(nm, work, stage_ms[i] / launches[i] / 1e3, peaks, peak_kind,
                                                     spec.name)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, torch, sel, spec, w, cu, params, q_dev, k_dev, hid_dev, pos_dev, slot_dev, cu_dev, out,
                      dev, world)

    # supplementary gather point: the mask all ones (p = 1), full traffic
    gather_p1 = None
    if not args.no_gather_p1:
        gather_p1 = run_gather_p1(torch, sel, spec, w, cu, cu_dev, hid_dev, pos_dev, slot_dev, out, peaks)

    # the other workloads (one GPU only: they are not the headline)
    per_config = None
    if rank == 0 and world == 1 and not args.no_per_config:
        del x
        torch.cuda.empty_cache()
        names = [n for n in PER_CONFIG if n != spec.name]
        per_config = run_per_config(torch, B, sel, names, dev, stream, flush, peaks, peak_kind)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded bf16 N(0,1) + planted blocks)",
                "config": config_of(spec, w, args),
                "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms),
                            "traced_mean": statistics.mean(traced), "stage_sum": sum(stage_ms) / args.steps},
                "kept_tokens": kept_total, "kept_fraction": kept_total / T,
                "roofline": roofline, "stages": stages, "cpu_baseline": cpu, "e2e": e2e, "gather_p1": gather_p1,
                "graph": graph, "per_config": per_config,
                "gpu_launches": int(sum(launches)), "clocks": clk, "wall_s": wall}
        print(json.dumps(line), flush=True)
    sel.close()
    if world > 1:
        dist.destroy_process_group()
    return 0


# --------------------------------------------------- tensor-parallel mode ----

def tp_shard_inputs(w, rank, world):
    """This rank's head slices of a workload: (q-head slice, kv-head slice,
    tail Q bits [n_rows, H_q/P, d], K bits [T, H_kv/P, d])."""
    from sparse_long_context_tail_gb300 import tp
    s = w.spec
    qs, ks = tp.shard_heads(s.num_q_heads, s.num_kv_heads, rank, world)
    return qs, ks, np.ascontiguousarray(w.q_tail_bits[:, qs]), np.ascontiguousarray(w.k_bits[:, ks])


def tp_masks_agree(keep_bits, dist_mod, group=None):
    """True when every rank of the group holds the same keep mask (all-gather
    of the mask words, compared on every rank)."""
    import torch
    if not (dist_mod.is_available() and dist_mod.is_initialized()) or dist_mod.get_world_size(group) == 1:
        return True
    world = dist_mod.get_world_size(group)
    gathered = [torch.empty_like(keep_bits) for _ in range(world)]
    dist_mod.all_gather(gathered, keep_bits, group=group)
    return all(torch.equal(gathered[0], g) for g in gathered[1:])


def run_tp(args):
    """Tensor-parallel selection: the heads of one batch sharded over N ranks
    (rank r holds only its q and kv heads), each rank scores its heads, one
    sum all-reduce of the fp32 [T] scores over NCCL, then every rank selects
    and compacts its own copy of the hidden rows.  The total work is fixed
    (strong scaling); value = tokens of the batch / the slowest rank's step."""
    import torch
    import torch.distributed as dist
    from sparse_long_context_tail_gb300 import _binding as B
    from sparse_long_context_tail_gb300 import tp
    from sparse_long_context_tail_gb300.selector import TokenSelector

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    spec = wl.named_spec(args.workload)
    if args.top_p is not None:
        spec.top_p = args.top_p
    w = wl.generate(spec)                     # the same batch on every rank
    qs, ks, q_bits, k_bits = tp_shard_inputs(w, rank, world)
    hq_l, hkv_l = qs.stop - qs.start, ks.stop - ks.start
    T = w.total_tokens
    q_local = torch.zeros((T, hq_l, spec.head_dim), dtype=torch.bfloat16, device=dev)
    q_local[torch.from_numpy(w.tail_rows).to(dev)] = torch.from_numpy(q_bits.view(np.int16)).view(
        torch.bfloat16).to(dev)
    k_local = torch.from_numpy(k_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    hid = torch.from_numpy(w.hidden_bits().view(np.int16)).to(dev)
    pos = torch.from_numpy(w.positions()).to(dev)
    slot = torch.from_numpy(w.slots()).to(dev)
    cu = w.cu_seqlens
    cu_dev = torch.from_numpy(cu).to(dev)
    params = B.make_params(spec.n_tail, spec.block, spec.sink_keep, spec.tail_keep, spec.top_p)
    sel = TokenSelector(local)
    out = sel.alloc_outputs(cu, spec.block, hid, pos, slot)
    flush = None if args.no_flush else torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    def step():
        return tp.tp_select_tokens(sel, q_local, k_local, cu, cu_dev, hq_l, hkv_l, spec.head_dim, hid, pos, slot,
                                   layer_id=0, params=params, out=out)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    status = sel.status()
    if status != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES.get(status)} during warm-up")
    agree = tp_masks_agree(out.keep_bits, dist)
    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    B.upf_profile_read(sel.ctx)
    step_ms = timed_loop(torch, step, stream, args.steps, flush)
    launches, _ = B.upf_profile_read(sel.ctx)
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    sec = statistics.mean(step_ms) / 1e3
    if world > 1:
        t = torch.tensor([sec], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        sec = float(t.item())
    kept = int(out.total_kept.item())
    if rank == 0:
        line = {"metric": METRIC, "value": T / sec, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "strong",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded bf16 N(0,1) + planted blocks)",
                "mode": "tp", "config": config_of(spec, w, args), "masks_agree_across_ranks": agree,
                "kept_tokens": kept, "kept_fraction": kept / T, "allreduce_bytes_per_step": 4 * T,
                "gpu_launches": int(sum(launches)), "clocks": clk}
        print(json.dumps(line), flush=True)
    sel.close()
    if world > 1:
        dist.destroy_process_group()
    return 0 if agree else 1


def graph_replay(torch, step, stream, steps, flush):
    """Capture one step in a CUDA graph and time `steps` replays (same inputs
    and outputs; the L2 flush stays outside the graph, between replays)."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()                      # one eager step on the capture stream first
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    cur = torch.cuda.current_stream()
    for i in range(steps):
        torch.cuda._sleep(LEAD_CYCLES)   # the replay is enqueued before its start event is reached
        starts[i].record(cur)
        g.replay()
        ends[i].record(cur)
        if flush is not None:
            flush.zero_()
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    return {"ms_per_step": statistics.mean(ms), "median_ms": statistics.median(ms), "steps": steps}


def full_attention_layers(layers, every):
    """Indices of the full-attention layers of an (every-1):1 hybrid stack: the
    last layer of every group of `every`."""
    return [i for i in range(layers) if (i + 1) % every == 0]


def run_stack(args):
    """Cumulative savings of token selection over a stack of later layers.

    The layers are modelled by their token-proportional part only: a gated FFN
    (LLaMA-3.1-8B sizes: hidden 4096, intermediate 14336; random bf16 weights
    shared by all layers; residual add), run with cuBLAS through torch.  In a
    hybrid schedule r:1, every (r+1)-th layer is a full-attention layer, where
    the selection runs on the current tokens before its FFN and every later
    layer sees only the kept ones.  The selection's inputs at every
    full-attention layer are the workload's own tail queries and keys,
    restricted to the surviving tokens (its planted structure stands in for a
    trained model's attention, so the kept fraction is the synthetic
    workload's, not a model's).  Attention and the linear-attention mixers are
    not modelled.  The dense baseline runs the same layers on every token."""
    import torch
    from sparse_long_context_tail_gb300 import _binding as B
    from sparse_long_context_tail_gb300.selector import TokenSelector
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    spec = wl.named_spec(args.workload)
    w = wl.generate(spec)
    cu = w.cu_seqlens
    T, Hd, Hi = w.total_tokens, spec.hidden, 14336
    params = B.make_params(spec.n_tail, spec.block, spec.sink_keep, spec.tail_keep, spec.top_p)
    q_all = torch.zeros((T, spec.num_q_heads, spec.head_dim), dtype=torch.bfloat16, device=dev)
    q_all[torch.from_numpy(w.tail_rows).to(dev)] = torch.from_numpy(w.q_tail_bits.view(np.int16)).view(
        torch.bfloat16).to(dev)
    k_all = torch.from_numpy(w.k_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    x0 = torch.from_numpy(w.hidden_bits().view(np.int16)).to(dev).view(torch.bfloat16)
    g = torch.Generator(device=dev).manual_seed(7)
    wg = (torch.randn((Hi, Hd), generator=g, device=dev) / math.sqrt(Hd)).to(torch.bfloat16)
    wu = (torch.randn((Hi, Hd), generator=g, device=dev) / math.sqrt(Hd)).to(torch.bfloat16)
    wd = (torch.randn((Hd, Hi), generator=g, device=dev) / math.sqrt(Hi)).to(torch.bfloat16)
    sel = TokenSelector(0)
    F = torch.nn.functional

    def ffn(x):
        return x + F.linear(F.silu(F.linear(x, wg)) * F.linear(x, wu), wd)

    def run(full_every):
        x, idx, cu_cur = x0, None, cu
        tokens, sel_ms = [], 0.0
        full = set(full_attention_layers(args.stack_layers, full_every)) if full_every else set()
        for layer in range(args.stack_layers):
            if layer in full:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                q = q_all if idx is None else q_all.index_select(0, idx)
                k = k_all if idx is None else k_all.index_select(0, idx)
                out = sel.select_tokens(q, k, cu_cur, torch.from_numpy(cu_cur).to(dev), spec.num_q_heads,
                                        spec.num_kv_heads, spec.head_dim, x.view(torch.int16), params=params,
                                        kv_of_q=spec.kv_of_q)
                e1.record()
                kept = int(out.total_kept.item())
                cu_cur = out.cu_seqlens_out.cpu().numpy().astype(np.int32)
                ki = out.kept_index[:kept].long()
                idx = ki if idx is None else idx.index_select(0, ki)
                x = out.hidden_out[:kept].view(torch.bfloat16)
                sel_ms += e0.elapsed_time(e1)
            x = ffn(x)
            tokens.append(int(x.shape[0]))
        return tokens, sel_ms

    def timed(full_every, reps=2):
        run(full_every)                                   # warm-up (allocations, cuBLAS plans)
        best = None
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            tokens, sel_ms = run(full_every)
            torch.cuda.synchronize()
            dt = (time.perf_counter() - t0) * 1e3
            best = dt if best is None or dt < best else best
        return best, tokens, sel_ms

    dense_ms, _, _ = timed(0)
    flop_layer = 2.0 * 3 * Hd * Hi
    result = {"mode": "stack", "workload": spec.name, "layers": args.stack_layers,
              "ffn": {"hidden": Hd, "intermediate": Hi, "gemm": "cuBLAS bf16 via torch"},
              "dense_ms": dense_ms, "dense_ffn_tflops": flop_layer * T * args.stack_layers / dense_ms / 1e9,
              "schedules": {}}
    for name, every in (("3:1", 4), ("5:1", 6)):
        ms, tokens, sel_ms = timed(every)
        full = full_attention_layers(args.stack_layers, every)
        result["schedules"][name] = {
            "full_attention_layers": full, "ms": ms, "speedup_vs_dense": dense_ms / ms,
            "saved_fraction": 1.0 - ms / dense_ms, "selection_ms": sel_ms,
            "tokens_after_each_full_layer": [tokens[i] for i in full],
            "token_layers_fraction": sum(tokens) / float(T * args.stack_layers)}
    result["note"] = ("layers modelled by their gated FFN only (the token-proportional part); selection at each "
                      "full-attention layer on the synthetic workload's own queries and keys; kept fractions are "
                      "the synthetic workload's, not a trained model's")
    print(json.dumps(result), flush=True)
    sel.close()
    return 0


def run_gather_p1(torch, sel, spec, w, cu, cu_dev, hid_dev, pos_dev, slot_dev, out, peaks, launches=5):
    """The compaction with every token kept (upf_compact with an all-ones mask on
    the same batch): the gather kernel then moves 2 T (row_bytes + 16) bytes, far
    more than L2, so its time is the HBM bound of the compaction at full traffic."""
    from sparse_long_context_tail_gb300 import _binding as B
    T = w.total_tokens
    row_bytes = hid_dev.stride(0) * hid_dev.element_size()
    bits = torch.full(((T + 31) // 32,), -1, dtype=torch.int32, device=hid_dev.device)
    batch, keep = B.make_batch(cu_dev.data_ptr(), cu, spec.num_q_heads, spec.num_kv_heads, spec.head_dim)
    nbytes = B.upf_workspace_bytes(batch, B.make_params())
    ws = sel.workspace(nbytes)
    io = B.make_compact_io(row_bytes=row_bytes, hidden_in=hid_dev.data_ptr(), hidden_out=out.hidden_out.data_ptr(),
                           pos_in=pos_dev.data_ptr(), pos_out=out.pos_out.data_ptr(), slot_in=slot_dev.data_ptr(),
                           slot_out=out.slot_out.data_ptr(), kept_index=out.kept_index.data_ptr(),
                           cu_seqlens_out=out.cu_seqlens_out.data_ptr(), total_kept=out.total_kept.data_ptr())
    stream = torch.cuda.current_stream().cuda_stream
    B.upf_compact(sel.ctx, batch, bits.data_ptr(), io, ws.data_ptr(), ws.numel(), stream)   # warm-up
    torch.cuda.synchronize()
    B.upf_profile_read(sel.ctx)
    B.upf_profile_enable(sel.ctx, True)
    for _ in range(launches):
        B.upf_compact(sel.ctx, batch, bits.data_ptr(), io, ws.data_ptr(), ws.numel(), stream)
    torch.cuda.synchronize()
    n_l, ms = B.upf_profile_read(sel.ctx)
    B.upf_profile_enable(sel.ctx, False)
    kept = int(out.total_kept.item())
    assert kept == T, (kept, T)
    gi = STAGES.index("compact_gather")
    per = ms[gi] / max(1, n_l[gi])
    moved = 2 * T * (row_bytes + 16)
    gbs = moved / (per / 1e3) / 1e9
    del keep
    return {"kept_tokens": kept, "bytes_per_launch": moved, "gather_ms_per_launch": per, "achieved_gbs": gbs,
            "peak_gbs": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"],
            "compaction_ms_per_launch": sum(ms[STAGES.index(k)] for k in ("compact_count", "compact_index",
                                                                         "compact_gather")) / launches}


def run_e2e(args, torch, sel, spec, w, cu, params, q_dev, k_dev, hid_dev, pos_dev, slot_dev, cu_dev, out, dev, world):
    """Same metric through TokenSelector.select_tokens with host (pinned) inputs and outputs.

    K, the tail query rows and cu_seqlens are copied to the device (scoring
    reads them twice); the hidden rows, positions and slots stay in page-locked
    host memory, which the compaction's gather reads and writes directly, so
    only the kept rows cross the host link.  Steps run as a serving loop
    would: step i+1's inputs are copied on a copy stream into the other of two
    device buffers while step i computes; every step's copies and its result
    readback are inside the timed loop.  The serial form (copy, call, read
    back, one step at a time) is reported beside it."""
    import dataclasses
    q_tail_h = torch.from_numpy(w.q_tail_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    tail_idx = torch.from_numpy(w.tail_rows).to(dev)
    k_h = torch.from_numpy(w.k_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    hid_h = torch.from_numpy(w.hidden_bits().view(np.int16)).pin_memory()
    pos_h = torch.from_numpy(w.positions()).pin_memory()
    slot_h = torch.from_numpy(w.slots()).pin_memory()
    cu_h = torch.from_numpy(cu).pin_memory()
    T = w.total_tokens
    row_bytes = hid_h.stride(0) * hid_h.element_size()
    # two sets of device inputs and of outputs (device mask/counts, host rows)
    k_b = [k_dev, torch.empty_like(k_dev)]
    q_b = [q_dev, q_dev.clone()]
    qt_b = [torch.empty_like(q_tail_h, device=dev) for _ in range(2)]
    cu_b = [cu_dev, torch.empty_like(cu_dev)]
    outs = [dataclasses.replace(sel.alloc_outputs(cu, params.block), hidden_out=torch.empty_like(hid_h).pin_memory(),
                                pos_out=torch.empty_like(pos_h).pin_memory(),
                                slot_out=torch.empty_like(slot_h).pin_memory()) for _ in range(2)]
    small_h = [dict(bits=torch.empty_like(o.keep_bits, device="cpu").pin_memory(),
                    cnt=torch.empty_like(o.kept_count, device="cpu").pin_memory(),
                    cuo=torch.empty_like(o.cu_seqlens_out, device="cpu").pin_memory(),
                    tot=torch.empty(1, dtype=torch.int32).pin_memory()) for o in outs]
    copy_s = torch.cuda.Stream(dev)
    main_s = torch.cuda.current_stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    computed = [torch.cuda.Event() for _ in range(2)]
    copy_bytes = q_tail_h.numel() * 2 + k_h.numel() * 2 + cu_h.numel() * 4

    def issue_copy(b):
        copy_s.wait_event(computed[b])          # the step that last used buffer b is done
        with torch.cuda.stream(copy_s):
            k_b[b].copy_(k_h, non_blocking=True)
            qt_b[b].copy_(q_tail_h, non_blocking=True)
            cu_b[b].copy_(cu_h, non_blocking=True)
            copied[b].record(copy_s)

    def issue_step(b):
        main_s.wait_event(copied[b])
        q_b[b].index_copy_(0, tail_idx, qt_b[b])
        o = outs[b]
        sel.select_tokens(q_b[b], k_b[b], cu, cu_b[b], spec.num_q_heads, spec.num_kv_heads, spec.head_dim, hid_h,
                          pos_h, slot_h, layer_id=0, params=params, kv_of_q=spec.kv_of_q, out=o)
        h = small_h[b]
        h["bits"].copy_(o.keep_bits, non_blocking=True)
        h["cnt"].copy_(o.kept_count, non_blocking=True)
        h["cuo"].copy_(o.cu_seqlens_out, non_blocking=True)
        h["tot"].copy_(o.total_kept, non_blocking=True)
        computed[b].record(main_s)

    for b in range(2):
        computed[b].record(main_s)
    # serial: one step at a time
    serial = []
    for i in range(3):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        issue_copy(0)
        issue_step(0)
        computed[0].synchronize()
        if i:
            serial.append(time.perf_counter() - t0)
    # pipelined loop (one untimed round first)
    times = []
    for rnd in range(2):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        issue_copy(0)
        for i in range(args.e2e_steps):
            if i + 1 < args.e2e_steps:
                issue_copy((i + 1) % 2)
            issue_step(i % 2)
        torch.cuda.synchronize()
        if rnd:
            times.append((time.perf_counter() - t0) / args.e2e_steps)
    total = int(small_h[0]["tot"][0])
    for b in range(2):
        assert int(small_h[b]["tot"][0]) == total
    kept_bytes = total * (row_bytes + 16)   # hidden row + position + slot per kept token
    h2d = copy_bytes + kept_bytes
    d2h = 4 + small_h[0]["bits"].numel() * 4 + small_h[0]["cnt"].numel() * 4 + small_h[0]["cuo"].numel() * 4 + \
        kept_bytes
    import torch.distributed as dist
    per, _, rate = aggregate_over_ranks(statistics.mean(times), T, dist if world > 1 else None, dev)
    return {"value": rate, "unit": UNIT, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": per * 1e3, "steps": args.e2e_steps, "serial_ms_per_step": statistics.mean(serial) * 1e3,
            "note": "wall clock of a loop of steps, each copying K, the tail Q rows and cu_seqlens from pinned host "
                    "memory (the next step's copy overlaps the current step's call), calling select_tokens (whose "
                    "gather reads the kept hidden rows, positions and slots from page-locked host memory and "
                    "writes them to page-locked host outputs), and reading back the mask, counts, offsets and "
                    "total; bytes count the copies plus the kept rows moved over the host link"}


if __name__ == "__main__":
    sys.exit(main())
