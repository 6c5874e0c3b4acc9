"""Benchmark: striped absorbed-MLA decode + exact LSE merge on one GB300 (per rank).

One step = the whole hot path over one batch: slot map + KV append of the
step's new tokens, the shard-local decode over all c shards, and the LSE
merge.  Inputs are resident in HBM when the timed region starts; the KV cache
of every workload except "tiny" is larger than L2, and for "tiny" L2 is
flushed between timed steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config bimodal] [--impl reference]

Prints one JSON line (rank 0).  The headline is the bimodal agentic batch, the
workload with the most KV bytes per step; at N = 1 the other four workloads
are timed after it the same way and reported under "per_workload".  With
N > 1 (torchrun) every rank runs an independent replica on its own GPU:
requests are independent and the path has no exchange step, so there is no
collective on the data path.
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
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import dcp_workloads as W  # noqa: E402

METRIC = "KV GB/s & % of HBM roofline for striped MLA decode+LSE merge; tokens/s"
L2_BYTES = 129 * 1024 * 1024


# ---------------------------------------------------------------------------
# Accounting (algorithmic bytes and FLOPs)
# ---------------------------------------------------------------------------
def flops_per_key_head() -> int:
    """FLOPs per (visible key, query row): 576-d dot product + 512-d weighted sum."""
    return 2 * W.D_K + 2 * W.D_LATENT


def q_o_bytes_per_head(q_bytes=2, o_bytes=2) -> int:
    return W.D_K * q_bytes + W.D_LATENT * o_bytes


def visible_keys(w: W.Workload, lens) -> int:
    """Sum over requests and query rows of the keys each row attends (causal for Tq > 1)."""
    tot = 0
    for L in lens:
        for t in range(w.Tq):
            tot += (L - w.Tq + t + 1) * w.H
    return tot


def accounting(w: W.Workload, lens, max_pages: int) -> dict:
    kv = sum(lens) * w.kv_bytes_per_token()
    q = w.B * w.Tq * w.H * W.D_K * 2
    out = w.B * w.Tq * w.H * (W.D_LATENT + 1) * 4
    tables = w.B * max_pages * 4 + w.B * 4
    append_rows = w.B * w.Tq * (w.kv_bytes_per_token() + 4 + 8)
    flops = visible_keys(w, lens) * flops_per_key_head()
    return dict(kv_bytes=kv, q_bytes=q, out_bytes=out, table_bytes=tables,
                append_bytes=append_rows,
                decode_bytes=kv + q + tables,
                step_bytes=kv + q + tables + out + append_rows,
                flops=flops)


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        rows = [s for (t, s) in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        window = "timed region"
        if not rows and self.samples:
            rows = [s for (_, s) in self.samples]
            window = "whole run (timed region shorter than the sampling interval)"
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for nm, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "window": window}


# ---------------------------------------------------------------------------
# Helpers
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, ws: int) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_gbs(bytes_per_rank: float, ms_step: float, ws: int) -> float:
    """Whole-job throughput: every rank moves bytes_per_rank per step; ms_step is the
    slowest rank's step time (weak scaling, one replica per GPU)."""
    return bytes_per_rank * ws / (ms_step * 1e-3) / 1e9


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_source_sha(paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if taken on the current source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}/{workload}")
    if not e:
        return None
    if e.get("source_sha") != kernel_source_sha(e.get("sources", [])):
        return None
    return e.get("dram_bytes_per_launch")


DECODE_KERNELS = {1: "decode_fh_bf16_kernel + fh_combine_kernel (tokens as MMA M)",
                  2: "decode_tc_bf16/e4m3_kernel (128-row tiles)",
                  3: "decode_fma_kernel (CUDA cores)"}

DECODE_SOURCES = ["decode_context_mla_gb300/csrc/decode_fewhead.cu",
                  "decode_context_mla_gb300/csrc/decode_tc.cu",
                  "decode_context_mla_gb300/csrc/sm100.cuh",
                  "decode_context_mla_gb300/csrc/decode_fma.cu",
                  "decode_context_mla_gb300/csrc/decode.cu",
                  "decode_context_mla_gb300/csrc/decode.cuh",
                  "decode_context_mla_gb300/csrc/common.cuh"]


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample
# ---------------------------------------------------------------------------
def oracle_sample(w: W.Workload, budget_s: float, max_requests: int = 256):
    """Time the fp64 oracle (striped decode + merge) on whole requests until the budget is spent."""
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle_ref import OracleWorkload
    ow = OracleWorkload(w)
    lens = ow.lens
    order = sorted(range(w.B), key=lambda b: lens[b])
    pick = [order[len(order) // 2]] + [b for b in order if b != order[len(order) // 2]]
    done_bytes, t_sum, n = 0, 0.0, 0
    wall0 = time.perf_counter()
    for b in pick[:max_requests]:
        if n and time.perf_counter() - wall0 > 2 * budget_s:
            break
        ow.load(b)
        t0 = time.perf_counter()
        ow.decode(b)
        t_sum += time.perf_counter() - t0
        done_bytes += lens[b] * w.kv_bytes_per_token()
        n += 1
        if t_sum >= budget_s:
            break
    return done_bytes, t_sum, n


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# Reference arm: the oracle, timed on the host cores
# ---------------------------------------------------------------------------
def run_reference(args, w: W.Workload):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle_ref import OracleWorkload
    ow = OracleWorkload(w)
    lens = ow.lens
    # each step: the oracle on one whole request (cycling over two requests)
    reqs = sorted(range(w.B), key=lambda b: lens[b])[: min(2, w.B)]
    for b in reqs:
        ow.load(b)
    for i in range(args.warmup):
        ow.decode(reqs[i % len(reqs)])
    t, nbytes, toks = 0.0, 0, 0
    for i in range(args.steps):
        b = reqs[i % len(reqs)]
        t0 = time.perf_counter()
        ow.decode(b)
        t += time.perf_counter() - t0
        nbytes += lens[b] * w.kv_bytes_per_token()
        toks += lens[b] * w.Tq
    gbs = nbytes / t / 1e9
    sample = (f"{args.steps} steps, each the fp64 oracle on one whole request "
              f"(requests {reqs}, {[lens[b] for b in reqs]} tokens) of the {w.name} workload")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_obj(w), "attended_tokens_per_s": round(toks / t, 1),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": cpu_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_obj(w: W.Workload) -> dict:
    return {"workload": w.name, "description": w.description, "B": w.B, "H": w.H, "Tq": w.Tq,
            "c": w.c, "P": w.P, "kv_dtype": w.kv_dtype, "lse_base": w.lse_base,
            "seq_len": w.L if w.L else "bimodal", "parallelism": "replicas (one per GPU)",
            "l2": ("KV cache larger than L2" if sum(w.seq_lens()) * w.kv_bytes_per_token()
                   > 4 * L2_BYTES else "L2 flushed between timed steps")}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------
def measure_step(args, w: W.Workload, ws: int, local: int, with_e2e: bool) -> dict:
    """Build the workload, capture its step as graphs and time `args.steps` replays.

    Returns the step and decode-launch times (max over ranks for the step), the roofline
    and tensor figures of the decode launch, the clocks seen during the timed region and,
    when asked, the end-to-end figure from pinned host buffers."""
    import dcp_harness as Hn
    from decode_context_mla_gb300 import binding as B

    dw = Hn.build(w, fused=args.fused)
    step = dw.step
    lens = dw.lens
    acc = accounting(w, lens, step.page_table.shape[1])
    small = acc["kv_bytes"] <= 4 * L2_BYTES
    flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device="cuda") if small else None

    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    # warm-up eagerly once (sets kernel attributes), then capture the step's three phases as
    # graphs: slot map + append, the decode (the dominant kernel), the merge
    with torch.cuda.stream(stream):
        step.run()
    torch.cuda.synchronize()
    graphs = []
    for phase in (step.run_append, step.run_decode, step.run_merge):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            phase()
        graphs.append(g)
    g_pre, g_dec, g_post = graphs
    c = dw.cache
    path, dec_launches = B.dcpmla_decode_path(w.B, w.Tq, w.H, w.P, w.c, w.c, c.kv_dtype,
                                              step.page_table.shape[1])
    torch.cuda.synchronize()

    def replay_step():
        g_pre.replay()
        g_dec.replay()
        g_post.replay()

    def timed(k):
        """(step ms summed over k steps, decode-launch ms summed over k steps), device clocks.

        Events on the launching stream bracket every step and, inside it, the decode
        launch; with a small cache L2 is flushed between steps, outside the brackets."""
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(k)]
        with torch.cuda.stream(stream):
            for i in range(k):
                if flush is not None:
                    flush.add_(1)
                ev[i][0].record(stream)
                g_pre.replay()
                ev[i][1].record(stream)
                g_dec.replay()
                ev[i][2].record(stream)
                g_post.replay()
                ev[i][3].record(stream)
        ev[-1][3].synchronize()
        dec = sum(e[1].elapsed_time(e[2]) for e in ev)
        if flush is None:
            tot = ev[0][0].elapsed_time(ev[-1][3])
        else:
            tot = sum(e[0].elapsed_time(e[3]) for e in ev)
        return tot, dec

    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            replay_step()
    torch.cuda.synchronize()
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    sampler = ClockSampler(vis.split(",")[local].strip() if vis else str(local))
    sampler.start()
    time.sleep(0.3)
    for _ in range(args.warmup):        # bring the clocks back up after the pause
        with torch.cuda.stream(stream):
            replay_step()
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    ms_total, ms_dec_total = timed(args.steps)
    t_wall1 = time.time()
    torch.cuda.synchronize()
    barrier(ws)
    ms_dec = ms_dec_total / args.steps
    time.sleep(0.15)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    err = c.check_errors()
    if err:
        raise RuntimeError(f"device error bits {err} ({w.name})")

    ms_step = max_over_ranks(ms_total / args.steps, ws)
    peaks = measured_peaks()
    achieved = acc["decode_bytes"] / (ms_dec * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": recorded_traffic(w.name, "decode"),
                "kernel": "dcpmla_decode (all c shards): " + DECODE_KERNELS[path],
                "kernel_ms": round(ms_dec, 4),
                "algorithmic_bytes": acc["decode_bytes"],
                "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst copy)"}
    tflops = acc["flops"] / (ms_dec * 1e-3) / 1e12
    tensor_info = {"achieved_tflops": round(tflops, 2), "peak_tflops": peaks["bf16_tflops"],
                   "frac": round(tflops / peaks["bf16_tflops"], 4),
                   "algorithmic_flops": acc["flops"]}
    e2e = run_e2e(args, w, dw, stream, acc, ws) if with_e2e else None

    # slot map + append (when the step appends), the decode's kernels, the merge
    # (fused: the decode's own merge kernel replaces the split merge and the LSE merge on
    # the bf16 tensor-core paths; E4M3 on the 128-row path decodes, then runs the LSE merge)
    if not args.fused:
        dec_step = dec_launches
    elif path == 2:
        dec_step = dec_launches + (1 if w.kv_dtype == "e4m3" else 0)
    else:
        dec_step = 2
    launches_per_step = (2 if step.do_append else 0) + dec_step
    if not args.fused:
        launches_per_step += 1
    res = dict(acc=acc, lens=lens, ms_step=ms_step, ms_dec=ms_dec, roofline=roofline,
               tensor=tensor_info, clocks=clocks, e2e=e2e, launches_per_step=launches_per_step,
               value=whole_job_gbs(acc["kv_bytes"], ms_step, ws))
    del graphs, g_pre, g_dec, g_post, dw, step, c, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


# The benchmark's headline workload: the one with the most KV bytes per step, on which the
# KV-GB/s metric is largest (the bimodal agentic mix); the others are reported beside it.
HEADLINE = "bimodal"


def run_ours(args, w: W.Workload):
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    from __graft_entry__ import build
    build()

    head = measure_step(args, w, ws, local, with_e2e=True)
    lens, acc, ms_step = head["lens"], head["acc"], head["ms_step"]

    # CPU baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        nb, t, n = oracle_sample(w, args.cpu_budget_s)
        cpu = {"value": round(nb / t / 1e9, 4), "unit": "GB/s", "cores": cpu_cores(),
               "kind": "oracle",
               "sample": f"fp64 oracle (striped decode + merge) on {n} whole request(s) of the "
                         f"{w.name} workload, {t:.1f} s of CPU work"}

    # the other workloads of the benchmark, each timed the same way (N = 1 only: with more
    # GPUs the run times the headline replicas alone)
    per_workload = None
    if ws == 1 and not args.no_per_workload and not args.batch and not args.interleave:
        per_workload = {}
        for name in W.WORKLOADS:
            if name == w.name:
                continue
            r = measure_step(args, W.WORKLOADS[name], ws, local, with_e2e=True)
            per_workload[name] = {
                "value": round(r["value"], 2), "unit": "GB/s", "ms_per_step": round(r["ms_step"], 4),
                "kernel_ms": r["roofline"]["kernel_ms"],
                "hbm_frac": r["roofline"]["frac"], "tensor_frac": r["tensor"]["frac"],
                "achieved_gbs": r["roofline"]["achieved"],
                "achieved_tflops": r["tensor"]["achieved_tflops"],
                "kernel": r["roofline"]["kernel"], "traffic": r["roofline"]["traffic"],
                "attended_tokens_per_s": round(sum(r["lens"]) * W.WORKLOADS[name].Tq
                                               / (r["ms_step"] * 1e-3), 1),
                "clocks": r["clocks"], "gpu_launches": r["launches_per_step"] * args.steps,
                "e2e": {k: r["e2e"][k] for k in ("value", "unit", "ms_per_step", "h2d_bytes_per_step",
                                                 "d2h_bytes_per_step")},
            }

    if rank == 0:
        peaks = measured_peaks()
        line = {
            "metric": METRIC, "value": round(head["value"], 2), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.kv_dtype == "bf16" else "e4m3", "data": "synthetic",
            "config": dict(config_obj(w), step="decode + merge fused" if args.fused else "decode, then merge"),
            "attended_tokens_per_s": round(sum(lens) * w.Tq * ws / (ms_step * 1e-3), 1),
            "decode_tokens_per_s": round(w.B * w.Tq * ws / (ms_step * 1e-3), 1),
            "step_hbm_frac": round(acc["step_bytes"] / (ms_step * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "roofline": head["roofline"], "tensor": head["tensor"], "cpu_baseline": cpu,
            "e2e": head["e2e"], "gpu_launches": head["launches_per_step"] * args.steps,
            "clocks": head["clocks"],
        }
        if per_workload is not None:
            line["per_workload"] = per_workload
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, w, dw, stream, acc, ws):
    """Same metric through the public step call from pinned host buffers (copies timed)."""
    import dcp_harness as Hn
    step = dw.step
    q_h = W.q_tensor(w, "cpu").pin_memory()
    rows, scales = Hn.new_rows_host(w, dw.lens)
    ckv_h = rows[:, :W.D_LATENT].contiguous().pin_memory()
    krope_h = rows[:, W.D_LATENT:].contiguous().pin_memory()
    sc_h = None if scales is None else scales.pin_memory()
    o_h = torch.empty(step.o.shape, dtype=torch.float32).pin_memory()
    lse_h = torch.empty(step.lse.shape, dtype=torch.float32).pin_memory()

    def one():
        with torch.cuda.stream(stream):
            step.run_host(q_h, ckv_h, krope_h, sc_h, o_h, lse_h)

    for _ in range(max(3, args.warmup)):
        one()
    torch.cuda.synchronize()
    barrier(ws)
    k = args.steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(k):
        one()
    e1.record(stream)
    e1.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / k, ws)
    return {"value": round(whole_job_gbs(acc["kv_bytes"], ms, ws), 2), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": step.h2d_bytes(),
            "d2h_bytes_per_step": step.d2h_bytes(),
            "path": "DecodeStep.run_host: pinned host inputs -> slot map, append, decode, merge "
                    "-> pinned host outputs, eager launches"}


# ---------------------------------------------------------------------------
# The layout calls around the decode (one call per step, large synthetic input)
# ---------------------------------------------------------------------------
def _event_time(fn, k, stream):
    """Mean ms of fn() over k calls on `stream`, CUDA events on that stream.  The call is
    captured once as a CUDA graph and replayed, so host-side call overhead (which would
    dominate a call of some tens of microseconds) stays out of the device time."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()                                # one untimed replay
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(k):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / k


def run_op(args, w: W.Workload):
    """Relayout, gather, E4M3 quantising append or HiCache filter: HBM GB/s moved."""
    from __graft_entry__ import build
    build()
    from decode_context_mla_gb300 import binding as B
    dev = "cuda"
    stream = torch.cuda.Stream()
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    peaks = measured_peaks()
    g = torch.Generator(device=dev).manual_seed(w.seed)
    lens = w.seq_lens()
    P, c, I = w.P, w.c, w.interleave
    sample = ""
    if args.op in ("relayout", "gather"):
        dpages = [(L + P - 1) // P for L in lens]
        vpages = [(L + P * c - 1) // (P * c) for L in lens]
        dpt = torch.full((w.B, max(dpages)), -1, dtype=torch.int32)
        vpt = torch.full((w.B, max(vpages)), -1, dtype=torch.int32)
        dperm = torch.randperm(sum(dpages), generator=torch.Generator().manual_seed(1)).to(torch.int32)
        vperm = torch.randperm(sum(vpages), generator=torch.Generator().manual_seed(2)).to(torch.int32)
        k0 = k1 = 0
        for b in range(w.B):
            dpt[b, :dpages[b]] = dperm[k0:k0 + dpages[b]]
            vpt[b, :vpages[b]] = vperm[k1:k1 + vpages[b]]
            k0 += dpages[b]
            k1 += vpages[b]
        dense = torch.randint(-30000, 30000, (sum(dpages) * P, W.D_K), dtype=torch.int16, device=dev,
                              generator=g).view(torch.bfloat16)
        pools = [torch.empty((sum(vpages) * P, W.D_K), dtype=torch.bfloat16, device=dev) for _ in range(c)]
        dpt_d, vpt_d = dpt.to(dev), vpt.to(dev)
        lens_d = torch.tensor(lens, dtype=torch.int32, device=dev)
        B.dcpmla_relayout_dense_to_striped(dense, None, dpt_d, pools, None, B.KV_BF16, vpt_d, lens_d, P, c,
                                           err, stream, interleave=I)
        if args.op == "relayout":
            fn = lambda: B.dcpmla_relayout_dense_to_striped(dense, None, dpt_d, pools, None, B.KV_BF16, vpt_d,
                                                            lens_d, P, c, err, stream, interleave=I)
        else:
            out = torch.empty((w.B, max(lens), W.D_K), dtype=torch.bfloat16, device=dev)
            fn = lambda: B.dcpmla_gather_unstriped(pools, None, B.KV_BF16, vpt_d, lens_d, P, c, out, None, err,
                                                   stream, interleave=I)
        moved = 2 * sum(lens) * W.D_K * 2
        units, unit = sum(lens), "tokens"
        sample = "oracle relayout of 4096 tokens of request 0"
        def cpu_leg():
            import oracle as O
            n = 4096
            rows = np.zeros((n, W.D_K), np.uint16)
            dpt_h = np.arange((n + P - 1) // P)[None, :]
            vpt_h = np.arange((n + P * c - 1) // (P * c))[None, :]
            pools_h = [np.zeros(((n // c) + 2 * P, W.D_K), np.uint16) for _ in range(c)]
            t0 = time.perf_counter()
            O.relayout_dense_to_striped(rows, None, dpt_h, [n], vpt_h, pools_h, None, c, P, I)
            return n * W.D_K * 2 * 2 / (time.perf_counter() - t0) / 1e9
    elif args.op == "append_e4m3":
        n = 1 << 20
        pages = (n + P - 1) // P + 1
        pools = [torch.empty((pages * P, W.D_K), dtype=torch.uint8, device=dev) for _ in range(c)]
        spools = [torch.empty(pages * P, dtype=torch.float32, device=dev) for _ in range(c)]
        rows = torch.randn((n, W.D_K), generator=g, device=dev).to(torch.bfloat16)
        own = (torch.arange(n, device=dev) % c).to(torch.int32)
        phys = (torch.arange(n, device=dev) // c).to(torch.int64)
        fn = lambda: B.dcpmla_kv_append_e4m3(pools, spools, own, phys, rows[:, :512], rows[:, 512:], err, stream)
        moved = n * (W.D_K * 2 + 4 + 8 + W.D_K + 4)
        units, unit = n, "rows"
        sample = "oracle quantisation of 2048 rows"
        def cpu_leg():
            import oracle as O
            r = np.random.default_rng(0).integers(0, 1 << 15, (2048, W.D_K)).astype(np.uint16)
            t0 = time.perf_counter()
            O.quantize_e4m3_rows(r)
            return 2048 * (W.D_K * 2 + W.D_K + 4) / (time.perf_counter() - t0) / 1e9
    elif args.op == "hicache":
        n = 1 << 24
        # slots of the widened-page space of a 2^31-slot virtual capacity
        idx = torch.randint(0, 1 << 31, (n,), dtype=torch.int64, device=dev, generator=g)
        out = torch.empty(n, dtype=torch.int64, device=dev)
        cnt = torch.zeros(1, dtype=torch.int64, device=dev)
        ws = torch.empty(max(16, B.dcpmla_hicache_filter_workspace_size(n)), dtype=torch.uint8, device=dev)
        fn = lambda: B.dcpmla_hicache_filter(idx, c, 0, out, cnt, ws, err, stream, interleave=I)
        moved = n * 8 + (n // c) * 8           # the list read once, the kept slots written
        units, unit = n, "indices"
        sample = "oracle filter of 1M indices"
        def cpu_leg():
            import oracle as O
            x = np.random.default_rng(0).integers(0, 1 << 40, 1 << 20)
            t0 = time.perf_counter()
            O.hicache_filter(x, c, 0, I)
            return (1 << 20) * 8 * (1 + 1 / c) / (time.perf_counter() - t0) / 1e9
    else:
        raise ValueError(args.op)
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            fn()
    torch.cuda.synchronize()
    ms = _event_time(fn, args.steps, stream)
    if int(err.item()):
        raise RuntimeError(f"device error bits {int(err.item())}")
    gbs = moved / (ms * 1e-3) / 1e9
    cpu = None
    if not args.no_cpu_baseline:
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        cpu = {"value": round(cpu_leg(), 4), "unit": "GB/s", "cores": cpu_cores(), "kind": "oracle",
               "sample": sample}
    line = {"metric": f"{args.op}: HBM GB/s moved", "value": round(gbs, 2), "unit": "GB/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if args.op != "hicache" else "int64", "data": "synthetic",
            "config": {"workload": f"{args.op} on {w.name}" if args.op in ("relayout", "gather") else args.op,
                       "units_per_step": units, "unit": unit, "c": c, "P": P, "interleave": I},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": None,
                         "algorithmic_bytes": moved},
            "cpu_baseline": cpu, "e2e": None, "gpu_launches": args.steps}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=HEADLINE, choices=sorted(W.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time only --config (by default the other workloads are timed after it "
                         "and reported under per_workload)")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--op", default="step", choices=["step", "relayout", "gather", "append_e4m3", "hicache"],
                    help="what to time: the decode step (default) or one of the layout calls")
    ap.add_argument("--interleave", type=int, default=0, help="override the interleave size")
    ap.add_argument("--fused", action="store_true",
                    help="decode and merge in one call (dcpmla_decode_merged) instead of decode + merge")
    ap.add_argument("--batch", type=int, default=0,
                    help="run the workload with this many requests (small profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = W.WORKLOADS[args.config]
    if args.batch:
        w = W.scaled(w, B=args.batch, name=f"{w.name}_b{args.batch}")
    if args.interleave:
        w = W.scaled(w, interleave=args.interleave, name=f"{w.name}_i{args.interleave}")
    if args.op != "step":
        run_op(args, w)
        return
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
