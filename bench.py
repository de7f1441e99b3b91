"""Benchmark of the EP Normal MoE token pipeline on GB300.

One step = the whole hot path on one synthetic batch: dispatch layout ->
notify -> dispatch (INT8 quantisation when the workload has it) -> combine,
with inputs already resident in HBM.  ``value`` is tokens per second over
the step (T tokens per step, summed over ranks); per-stage times, achieved
HBM bandwidth and the roofline fraction of the dominant kernel (combine) are
reported next to it.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload dsv3]
    python bench.py --impl reference ...   # the CPU oracle, as it stands

Multi-GPU runs (torchrun, one rank per GPU) are independent replicas: each
rank runs the full R-logical-rank problem on its own GPU and there is no
data-path collective; ranks only meet in a barrier and a max-reduction of
the step time ("weak" scaling).
"""
import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

L2_FLUSH_BYTES = 256 << 20          # > 129 MB of L2
SWIGLU_INTERMEDIATE = 2048          # expert intermediate size (DeepSeek-V3)
EXTRA_STEPS = 50                    # timed iterations of the extra kernels
FALLBACK_HBM_GBS = 6800.0
E2E_TRIALS = 3                     # end-to-end trials (median reported)
KERNEL_SOURCES = {                  # kernel -> source file (traffic staleness)
    "combine": "combine_moe_dispatch_layout_gb300/csrc/combine.cu",
    "dispatch": "combine_moe_dispatch_layout_gb300/csrc/dispatch.cu",
    "combine_quant": "combine_moe_dispatch_layout_gb300/csrc/combine_quant.cu",
    "swiglu_quant": "combine_moe_dispatch_layout_gb300/csrc/swiglu.cu",
}
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,"
               "clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,"
               "clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,"
               "clocks_event_reasons.sw_power_cap")


# ---------------------------------------------------------------------------
# algorithmic bytes (what each stage must move at minimum)
# ---------------------------------------------------------------------------

def row_bytes(w):
    return ((w.H + 31) // 32 * 32 + 32) if w.quant else 2 * w.H


def alg_bytes(w):
    """Per launch: x read once + k rows written (+ indices) for dispatch;
    k rows read + one row written (+ indices, weights) for combine."""
    es = 2
    dispatch = (w.T * w.H * es + w.P * row_bytes(w) + w.P * 8
                + w.E * w.R * 4 + (w.R + 1) * 8)
    combine = w.P * w.H * es + w.P * 12 + w.T * w.H * es
    combine_quant = w.P * row_bytes(w.with_(quant=True)) + w.P * 12 + w.T * w.H * es
    layout = w.P * 8 + w.R * w.E * 4 + w.R * w.R * 4
    notify = 2 * w.R * w.E * 4 + w.E * 4 + w.R * 4 + (w.R + 1) * 8
    return dict(layout=layout, notify=notify, dispatch=dispatch,
                combine=combine, combine_quant=combine_quant)


def workload_desc(w):
    return ("%s: R=%d E=%d (%d/rank) bs=%d T=%d H=%d k=%d %s %s" % (
        w.name, w.R, w.E, w.epr, w.bs, w.T, w.H, w.k,
        "bf16" if w.dtype == W.BF16 else "fp16",
        "int8-quant" if w.quant else "verbatim"))


def step_config(w, world):
    """The `config` object of the step, the same on both arms (the reference
    arm runs the identical workload on the host cores)."""
    return {
        "workload": workload_desc(w),
        "step": "layout+notify+dispatch+combine, inputs resident in HBM",
        "l2": "flushed between steps (256 MiB write outside the step events)",
        "parallelism": "replicas" if world > 1 else "single GPU",
        "io_dtype": "bf16" if w.dtype == W.BF16 else "fp16",
        "recv_rows": "int8 + fp32 1/scale" if w.quant else "verbatim",
    }


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """(burst, sustained) dense bf16 TFLOP/s from MEASURED_PEAKS.json, else
    the fallback figures."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, "fallback"


def _file_hash(rel):
    with open(os.path.join(ROOT, rel), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel, workload, key="traffic_bytes_per_launch"):
    """Bytes per launch from the committed ncu record, if it was taken on the
    current source of that kernel (else None).  key: traffic_bytes_per_launch
    (DRAM reads + the SMs' writes into L2) or dram_bytes_per_launch (DRAM
    reads + DRAM writes; writes still in L2 at kernel end are missing)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        ent = d[kernel][workload]
        if ent["source_sha256_16"] != _file_hash(KERNEL_SOURCES[kernel]):
            return None
        return float(ent[key])
    except (OSError, KeyError, ValueError):
        return None


TRAFFIC_NOTE = ("traffic = DRAM reads + the bytes the SMs wrote into L2 (ncu, a small case "
                "scaled to a launch); traffic_dram = DRAM reads + DRAM writes")


# ---------------------------------------------------------------------------
# distributed helpers (replicas: a barrier and a max of the step time)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def reduce_max(value, world, device=None):
    """Max of a float over ranks (value on every rank)."""
    if world == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_tokens_per_s(tokens_per_rank, world, max_seconds):
    """Whole-job throughput: the tokens all ranks processed over the slowest
    rank's time."""
    return tokens_per_rank * world / max_seconds


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    def __init__(self, gpu_index, path=None):
        self.proc = None
        self.path = path or "/tmp/moe_ep_clocks_%d.csv" % os.getpid()
        self.gpu = gpu_index

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + CLOCK_QUERY,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
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
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def _events(n):
    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _mean_us(pairs):
    return float(np.mean([a.elapsed_time(c) for a, c in pairs])) * 1e3


def measure_pipeline(w, dev, stream, flush, x, idx, wt, y, steps, warmup,
                     barrier_fn=None):
    """The four-stage step on one workload: per-stage device times (CUDA
    events on the launching stream, L2 flushed before every step), the same
    step replayed from a CUDA graph, and the one-launch dispatch against the
    three separate launches (eager and graph-replayed).  Returns (record,
    buffers)."""
    from combine_moe_dispatch_layout_gb300 import pipeline as pl
    b = pl.PipelineBuffers(w.R, w.bs, w.k, w.epr, w.H, w.dtype, w.quant,
                           device=dev)

    def step(evs=None, st=None, upto=4):
        st = stream if st is None else st
        if evs:
            evs[0].record(st)
        pl.moe_dispatch_layout(b.shape, idx, b.count, b.rank_send, b.send_idx,
                               b.workspace, b.dev_status, st)
        if evs:
            evs[1].record(st)
        pl.moe_notify_dispatch(b.shape, b.count, b.put_offset, b.total_recv,
                               b.rank_recv_base, b.recv_per_expert, b.max_bs,
                               b.dev_status, st)
        if evs:
            evs[2].record(st)
        pl.run_dispatch(b, x, idx, st)
        if evs:
            evs[3].record(st)
        if upto > 3:
            pl.run_combine(b, y, idx, wt, st)
            if evs:
                evs[4].record(st)

    def check(what):
        torch.cuda.synchronize()
        if b.status() != 0:
            raise RuntimeError("%s: device status %d in %s" % (w.name, b.status(), what))

    for i in range(warmup):
        flush.fill_(i & 0xff)
        step()
    check("warm-up")
    evs = [_events(5) for _ in range(steps)]
    if barrier_fn:
        barrier_fn()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        flush.fill_(i & 0xff)        # between steps, outside the events
        step(evs[i])
    check("timed steps")
    if barrier_fn:
        barrier_fn()
    wall = time.perf_counter() - t0
    stage_ms = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(4)]
                         for i in range(steps)])

    def graph_of(fn):
        gs = torch.cuda.Stream(dev)
        gs.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            with torch.cuda.graph(g, stream=gs):
                fn(gs)
        stream.wait_stream(gs)
        return g

    def timed(fn, n):
        pairs = []
        for i in range(n):
            flush.fill_(i & 0xff)
            a0, a1 = _events(2)
            a0.record(stream)
            fn()
            a1.record(stream)
            pairs.append((a0, a1))
        return pairs

    n_extra = min(steps, EXTRA_STEPS)
    g_step = graph_of(lambda st: step(st=st))
    graph_step = timed(g_step.replay, n_extra)
    check("graph replay")
    del g_step
    for i in range(3):
        pl.run_dispatch_fused(b, x, idx, stream)
    check("one-launch dispatch")
    fused = timed(lambda: pl.run_dispatch_fused(b, x, idx, stream), n_extra)
    check("one-launch dispatch")
    g_fused = graph_of(lambda st: pl.run_dispatch_fused(b, x, idx, st))
    g_sep = graph_of(lambda st: step(st=st, upto=3))
    fused_graph = timed(g_fused.replay, n_extra)
    sep_graph = timed(g_sep.replay, n_extra)
    check("graph replay of the dispatch paths")
    del g_fused, g_sep
    stage_mean = stage_ms.mean(axis=0)
    rec = {"steps": steps, "stage_ms": stage_mean, "step_ms": stage_ms.sum(axis=1),
           "stage_ms_median": np.median(stage_ms, axis=0),
           "wall_s": wall,
           "graph_step_us": _mean_us(graph_step),
           "dispatch_fused": {
               "us": _mean_us(fused),
               "separate_us": float(stage_mean[0] + stage_mean[1] + stage_mean[2]) * 1e3,
               "graph_us": _mean_us(fused_graph),
               "separate_graph_us": _mean_us(sep_graph),
               "note": "layout+notify+dispatch in one cooperative launch vs three "
                       "launches; graph_us / separate_graph_us: the same replayed "
                       "from CUDA graphs (device time without host enqueue)"}}
    return rec, b


def config_record(w, m, peak, peak_kind, cpu=None):
    """The per-workload object of the JSON line from measure_pipeline's
    record: step and stage times, tokens/s, and dispatch / combine against
    the HBM roofline."""
    stage_mean = m["stage_ms"]
    names = ["layout", "notify", "dispatch", "combine"]
    ab = alg_bytes(w)
    step_ms = float(m["step_ms"].mean())

    def roof(n, j):
        ms = float(stage_mean[j])
        gbs = ab[n] / (ms * 1e-3) / 1e9
        return {"kernel": n, "bound": "hbm", "achieved": gbs, "peak": peak,
                "peak_source": peak_kind, "unit": "GB/s", "frac": gbs / peak,
                "traffic": recorded_traffic(n, w.name),
                "traffic_dram": recorded_traffic(n, w.name, "dram_bytes_per_launch"),
                "traffic_note": TRAFFIC_NOTE, "algorithmic_bytes": ab[n],
                "avg_launch_ms": ms, "tokens_per_s": w.T / (ms * 1e-3)}
    disp, comb = roof("dispatch", 2), roof("combine", 3)
    return {
        "workload": workload_desc(w),
        "steps": m["steps"],
        "step_us": step_ms * 1e3,
        "tokens_per_s": w.T / (step_ms * 1e-3),
        "dispatch_combine_tokens_per_s": w.T / ((stage_mean[2] + stage_mean[3]) * 1e-3),
        "stages_us": {n: float(stage_mean[j] * 1e3) for j, n in enumerate(names)},
        "step_us_median": float(np.median(m["step_ms"])) * 1e3,
        "stages_us_median": {n: float(m["stage_ms_median"][j] * 1e3)
                             for j, n in enumerate(names)},
        "stages_gbs": {n: ab[n] / (stage_mean[j] * 1e-3) / 1e9 for j, n in enumerate(names)},
        "roofline": comb if comb["avg_launch_ms"] >= disp["avg_launch_ms"] else disp,
        "roofline_dispatch": disp,
        "roofline_combine": comb,
        "graph_step_us": m["graph_step_us"],
        "dispatch_fused": m["dispatch_fused"],
        "cpu_baseline": cpu,
    }


def run_gpu(args, w):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    import combine_moe_dispatch_layout_gb300 as ep  # noqa: F401 (loads the .so)
    from combine_moe_dispatch_layout_gb300 import pipeline as pl
    dev = torch.device("cuda", local)
    peak, peak_kind = measured_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline

    idx_h, wt_h = W.routing(w)
    x_h = W.tokens(w)
    idx, wt, x = idx_h.to(dev), wt_h.to(dev), x_h.to(dev)
    y = W.expert_outputs_device(w, dev)

    clocks = ClockSampler(local, args.clocks_csv)
    clocks.start()
    m, b = measure_pipeline(w, dev, stream, flush, x, idx, wt, y, args.steps,
                            args.warmup, barrier_fn=lambda: barrier(world))
    clk = clocks.stop()
    stage_mean = m["stage_ms"]
    mean_step_ms = float(m["step_ms"].mean())
    max_step_ms = reduce_max(mean_step_ms, world, dev)
    value = aggregate_tokens_per_s(w.T, world, max_step_ms / 1e3)
    ab = alg_bytes(w)
    gbs = {n: ab[n] / (stage_mean[j] * 1e-3) / 1e9
           for j, n in enumerate(["layout", "notify", "dispatch", "combine"])}

    # ---- combine over INT8 expert outputs (moe_combine_quant) -------------
    def timed(fn, n):
        pairs = []
        for i in range(n):
            flush.fill_(i & 0xff)
            a0, a1 = _events(2)
            a0.record(stream)
            fn()
            a1.record(stream)
            pairs.append((a0, a1))
        torch.cuda.synchronize()
        return _mean_us(pairs)
    n_extra = min(args.steps, EXTRA_STEPS)
    cq = None
    if w.quant:
        yq = W.expert_outputs_int8(w).to(dev)
        for i in range(3):
            pl.run_combine_quant(b, yq, idx, wt, stream)
        cq_us = timed(lambda: pl.run_combine_quant(b, yq, idx, wt, stream), n_extra)
        if b.status() != 0:
            raise RuntimeError("device status %d in combine_quant" % b.status())
        cq_bytes = ab["combine_quant"]
        cq = {"us": cq_us, "achieved_gbs": cq_bytes / (cq_us * 1e-6) / 1e9,
              "algorithmic_bytes": cq_bytes,
              "traffic": recorded_traffic("combine_quant", w.name),
              "traffic_dram": recorded_traffic("combine_quant", w.name,
                                               "dram_bytes_per_launch"),
              "frac": cq_bytes / (cq_us * 1e-6) / 1e9 / peak,
              "tokens_per_s": w.T / (cq_us * 1e-6)}
        del yq

    # ---- GMM1 epilogue (moe_swiglu_quant): one row per dispatched pair, I=2048
    sw = None
    if w.quant:
        I = SWIGLU_INTERMEDIATE
        acc_h, ws_h, ts_h = W.gmm1_accumulators(w.P, I)
        acc_d, ws_d, ts_d = acc_h.to(dev), ws_h.to(dev), ts_h.to(dev)
        del acc_h
        sw_out = torch.empty((w.P, (I + 31) // 32 * 32 + 32), dtype=torch.uint8,
                             device=dev)
        for i in range(3):
            ep.moe_swiglu_quant(acc_d, ws_d, ts_d, sw_out, b.dev_status, stream)
        sw_us = timed(lambda: ep.moe_swiglu_quant(acc_d, ws_d, ts_d, sw_out,
                                                  b.dev_status, stream), n_extra)
        if b.status() != 0:
            raise RuntimeError("device status %d in swiglu_quant" % b.status())
        sw_bytes = w.P * (8 * I + (I + 31) // 32 * 32 + 32 + 4) + 8 * I
        sw = {"us": sw_us, "rows": w.P, "I": I, "algorithmic_bytes": sw_bytes,
              "traffic": recorded_traffic("swiglu_quant", w.name),
              "traffic_dram": recorded_traffic("swiglu_quant", w.name,
                                               "dram_bytes_per_launch"),
              "achieved_gbs": sw_bytes / (sw_us * 1e-6) / 1e9,
              "frac": sw_bytes / (sw_us * 1e-6) / 1e9 / peak}
        del acc_d, sw_out

    # ---- token-level layout (moe_token_layout) ------------------------------
    tpr = torch.empty((w.R, w.R), dtype=torch.int32, device=dev)
    inr = torch.empty((w.T, w.R), dtype=torch.uint8, device=dev)
    for i in range(3):
        ep.moe_token_layout(b.shape, idx, tpr, inr, b.dev_status, stream)
    tl_us = timed(lambda: ep.moe_token_layout(b.shape, idx, tpr, inr, b.dev_status,
                                              stream), n_extra)
    if b.status() != 0:
        raise RuntimeError("device status %d in token_layout" % b.status())
    del tpr, inr

    # ---- fused deep MoE (dispatch -> GMM1 -> DeqSwigluQuant -> GMM2 ->
    #      DeqCombine) on the same routing and tokens ------------------------
    deep = None
    if w.quant and w.E <= 256 and not args.no_deep_moe:   # weights: E x 44 M codes
        deep = run_deep_moe_bench(args, w, ep, pl, x, idx, wt, stream, dev, flush)

    # ---- end to end through the public API with host buffers --------------
    e2e = run_e2e(args, w, b, pl, idx_h, wt_h, x_h, y, stream, dev, flush)
    e2e_max_ms = reduce_max(e2e["ms_per_step"], world, dev)
    y_h = y.cpu() if want_cpu else None
    del b, y
    torch.cuda.empty_cache()

    cpu = None
    if want_cpu:
        cpu = cpu_baseline(w, idx_h, wt_h, x_h, y_h, args.cpu_seconds)
    del y_h
    head = config_record(w, m, peak, peak_kind, cpu)

    # ---- the other workloads, measured the same way -------------------------
    per_config = {}
    if not args.no_per_config and world == 1:
        for name in W.ORDER:
            if name == w.name:
                per_config[name] = head
                continue
            per_config[name] = run_other_config(args, W.WORKLOADS[name], dev, stream,
                                                flush, peak, peak_kind, want_cpu)

    if rank != 0:
        return None
    rec = {
        "metric": "dispatch+combine tokens/s",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": max_step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded: routing, weights and x drawn on the host, "
                "expert outputs drawn on the device)",
        "config": step_config(w, world),
        "roofline": dict(head["roofline_combine"]),
        "roofline_dispatch": head["roofline_dispatch"],
        "combine_quant": cq,
        "token_layout_us": tl_us,
        "graph_step_us": m["graph_step_us"],
        "swiglu_quant": sw,
        "deep_moe": deep,
        "dispatch_fused": m["dispatch_fused"],
        "stages_us": head["stages_us"],
        "stages_us_median": head["stages_us_median"],
        "step_us_median": head["step_us_median"],
        "stages_gbs": gbs,
        "dispatch_combine_tokens_per_s": head["dispatch_combine_tokens_per_s"],
        "e2e": {"value": aggregate_tokens_per_s(w.T, world, e2e_max_ms / 1e3),
                "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": e2e_max_ms, "steps": e2e["steps"],
                "link_ms_per_step": e2e["link_ms_per_step"],
                "frac_of_link": e2e["link_ms_per_step"] / e2e["ms_per_step"],
                "trials": e2e["trials"],
                "note": "every step copies x, topk_idx, topk_weights from pinned "
                        "host memory and out back inside the timed region; copies "
                        "of neighbouring steps overlap compute (3 streams); expert "
                        "outputs y stay on the device (they are produced there). "
                        "link_ms_per_step: the same copies on the same streams and "
                        "buffers with no kernels, timed just before each trial; "
                        "ms_per_step and link_ms_per_step are the medians of the "
                        "trials (each listed)"},
        "gpu_launches": 4 * args.steps,
        "clocks": clk,
        "wall_s_timed_region": m["wall_s"],
        "cpu_baseline": cpu,
        "per_config": per_config,
    }
    return rec


def run_other_config(args, w, dev, stream, flush, peak, peak_kind, want_cpu):
    """One non-headline workload: inputs drawn, the four-stage step timed
    (fewer steps than the headline), the oracle timed beside it."""
    idx_h, wt_h = W.routing(w)
    x_h = W.tokens(w)
    idx, wt, x = idx_h.to(dev), wt_h.to(dev), x_h.to(dev)
    y = W.expert_outputs_device(w, dev)
    steps = max(3, min(args.steps, args.per_config_steps))
    m, b = measure_pipeline(w, dev, stream, flush, x, idx, wt, y, steps, 3)
    y_h = y.cpu() if want_cpu else None
    del b, x, y, idx, wt
    torch.cuda.empty_cache()
    cpu = None
    if want_cpu:
        cpu = cpu_baseline(w, idx_h, wt_h, x_h, y_h, args.cpu_seconds)
    return config_record(w, m, peak, peak_kind, cpu)


def run_deep_moe_bench(args, w, ep, pl, x, idx, wt, stream, dev, flush):
    """Times the deep MoE pipeline stage by stage (CUDA events on the
    stream) with synthetic INT8 expert weights drawn on the device; the two
    grouped GEMMs are reported against the dense bf16 tensor peak."""
    I = SWIGLU_INTERMEDIATE
    w1, ws1, w2, ws2 = W.moe_weights(w.E, w.H, I, seed=31, device=dev)
    wts = pl.DeepMoeWeights(w1, ws1, w2, ws2, stream, interleaved=False)
    torch.cuda.synchronize()
    del w1, w2
    b = pl.DeepMoeBuffers(w.R, w.bs, w.k, w.epr, w.H, I, w.dtype, device=dev)
    P, H = w.P, w.H
    names = ["layout+notify", "dispatch_expand", "group_offsets", "gemm1",
             "swiglu_quant_bf16", "gemm2+dequant", "combine_f32"]

    def step(evs=None):
        def mark(j):
            if evs:
                evs[j].record(stream)
        mark(0)
        pl.run_layout_notify(b, idx, stream)
        mark(1)
        pl.run_dispatch_expand(b, x, idx, stream)
        mark(2)
        ep.moe_group_offsets(b.recv_per_expert, b.group_off, b.dev_status, stream)
        mark(3)
        ep.moe_grouped_gemm_i8(b.a1, wts.w1, b.recv_per_expert, b.acc1, b.dev_status,
                               stream)
        mark(4)
        ep.moe_swiglu_quant_grouped_bf16(b.acc1, wts.ws1, b.group_off, (b.ts1, 0, 4), b.a2,
                                         b.ts2, b.dev_status, stream)
        mark(5)
        ep.moe_grouped_gemm_i8_dequant(b.a2, wts.w2, b.recv_per_expert, wts.ws2,
                                       (b.ts2, 0, 4), b.y2, b.dev_status, stream)
        mark(6)
        pl.run_deep_combine(b, idx, wt, stream)
        mark(7)

    for i in range(3):
        step()
    torch.cuda.synchronize()
    if b.status() != 0:
        raise RuntimeError("device status %d in the deep MoE" % b.status())
    n = max(3, min(args.steps, 10))
    all_evs = []
    for i in range(n):
        flush.fill_(i & 0xff)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
        step(evs)
        all_evs.append(evs)
    torch.cuda.synchronize()
    if b.status() != 0:
        raise RuntimeError("device status %d in the deep MoE" % b.status())
    st_ms = np.array([[e[j].elapsed_time(e[j + 1]) for j in range(len(names))]
                      for e in all_evs])
    mean = st_ms.mean(axis=0)
    burst, sustained, src = measured_bf16_tflops()
    flops1 = 2.0 * P * H * 2 * I
    flops2 = 2.0 * P * I * H

    def gemm(flops, ms):
        tf = flops / (ms * 1e-3) / 1e12
        return {"us": ms * 1e3, "flops": flops, "achieved": tf, "unit": "TFLOP/s",
                "bound": "tensor", "peak": sustained, "frac": tf / sustained,
                "frac_of_burst": tf / burst, "peak_source": src,
                "note": "bf16 tensor-core MMA on int8-valued operands (exact int32)"}
    res = {
        "config": {"rows": P, "H": H, "I": I, "experts": w.E,
                   "weights": "synthetic int8 codes U[-127,127], bf16 copies resident"},
        "step_ms": float(mean.sum()),
        "tokens_per_s": w.T / (mean.sum() * 1e-3),
        "stages_us": {nm: float(mean[j] * 1e3) for j, nm in enumerate(names)},
        "gemm1": gemm(flops1, float(mean[3])),
        "gemm2": gemm(flops2, float(mean[5])),
        "steps": n,
    }
    del b, wts
    torch.cuda.empty_cache()
    return res


def run_gemm_only(args):
    """--gemm G,ROWS,N,K: times moe_grouped_gemm_i8 alone on G groups of ROWS
    rows (int8-valued bf16 operands drawn on the device) and prints one JSON
    line.  A kernel benchmark, not the step contract."""
    import combine_moe_dispatch_layout_gb300 as ep
    G, rows, N, K = (int(v) for v in args.gemm.split(","))
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    M = G * rows
    a = torch.randint(-127, 128, (M, K), generator=g, device=dev).to(torch.bfloat16)
    w = torch.randint(-127, 128, (G, N, K), generator=g, device=dev).to(torch.bfloat16)
    gr = torch.full((G,), rows, dtype=torch.int32, device=dev)
    c = torch.empty((M, N), dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cs = torch.rand((G, N), generator=g, device=dev) * 1e-4 + 1e-4
    rs = torch.rand((M,), generator=g, device=dev) * 0.01 + 0.01
    mode = args.gemm_epilogue
    h = torch.empty((M, N // 2), dtype=torch.float32, device=dev) if mode == "swiglu" else None

    def gemm():
        if mode == "int32":
            ep.moe_grouped_gemm_i8(a, w, gr, c, st, stream)
        elif mode == "dequant":
            ep.moe_grouped_gemm_i8_dequant(a, w, gr, cs, (rs, 0, 4), c.view(torch.float32), st,
                                           stream)
        else:
            ep.moe_grouped_gemm_i8_swiglu(a, w, gr, cs, (rs, 0, 4), h, st, stream)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        gemm()
    evs = []
    for i in range(args.steps):
        flush.fill_(i & 0xff)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        gemm()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize()
    if int(st.item()) != 0:
        raise RuntimeError("device status %d" % int(st.item()))
    us = float(np.mean([x.elapsed_time(y) for x, y in evs])) * 1e3
    burst, sustained, src = measured_bf16_tflops()
    tf = 2.0 * M * N * K / (us * 1e-6) / 1e12
    print(json.dumps({"kernel": "grouped_gemm_i8", "epilogue": mode, "groups": G,
                      "rows_per_group": rows,
                      "N": N, "K": K, "us": us, "tflops": tf, "frac_of_burst": tf / burst,
                      "peak_source": src, "steps": args.steps}))


def run_e2e(args, w, b, pl, idx_h, wt_h, x_h, y, stream, dev, flush):
    """Throughput through the public API with the inputs in pinned host
    memory: every step copies x, topk_idx and topk_weights to the device,
    runs the four stages and copies the output back.  Copies of neighbouring
    steps overlap with compute (an H2D stream, the compute stream and a D2H
    stream; inputs and outputs double-buffered), as a caller streaming
    batches would run it."""
    x_p = x_h.pin_memory()
    idx_p = idx_h.pin_memory()
    wt_p = wt_h.pin_memory()
    outs_p = [torch.empty(b.out.shape, dtype=b.out.dtype).pin_memory()
              for _ in range(2)]
    x_d = [torch.empty_like(x_p, device=dev) for _ in range(2)]
    idx_d = [torch.empty_like(idx_p, device=dev) for _ in range(2)]
    wt_d = [torch.empty_like(wt_p, device=dev) for _ in range(2)]
    out_d = [b.out, torch.empty_like(b.out)]
    s_h2d = torch.cuda.Stream(dev)
    s_d2h = torch.cuda.Stream(dev)
    steps = max(3, min(args.steps, args.e2e_steps))
    n_warm = max(3, args.warmup)
    # per buffer slot: inputs consumed by compute / output drained by D2H
    consumed = [torch.cuda.Event() for _ in range(2)]
    drained = [torch.cuda.Event() for _ in range(2)]

    def one(i, compute=True):
        j = i % 2
        with torch.cuda.stream(s_h2d):
            if i >= 2:
                s_h2d.wait_event(consumed[j])
            x_d[j].copy_(x_p, non_blocking=True)
            idx_d[j].copy_(idx_p, non_blocking=True)
            wt_d[j].copy_(wt_p, non_blocking=True)
            loaded = torch.cuda.Event()
            loaded.record(s_h2d)
        stream.wait_event(loaded)
        if i >= 2:
            stream.wait_event(drained[j])
        b.out = out_d[j]
        if compute:
            pl.run_pipeline(b, x_d[j], idx_d[j], wt_d[j], y, stream)
        consumed[j].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(consumed[j])
            outs_p[j].copy_(out_d[j], non_blocking=True)
            drained[j].record(s_d2h)

    def run(compute):
        for i in range(n_warm):
            one(i, compute)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s_h2d)
        for i in range(steps):
            one(n_warm + i, compute)
        e1.record(s_d2h)      # after the last D2H copy, which waited for compute
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    # Trials, each the ceiling first (the same copies, streams and buffers, no
    # kernels) and then the full loop; the medians are reported and every
    # trial is listed (the host link is shared with the node's other GPUs,
    # so a single trial can catch a neighbour's transfer).
    trials = []
    for _ in range(E2E_TRIALS):
        link_ms = run(False)
        ms = run(True)
        trials.append({"link_ms_per_step": link_ms, "ms_per_step": ms})
    b.out = out_d[0]
    if b.status() != 0:
        raise RuntimeError("device status %d in e2e" % b.status())
    h2d = (x_p.numel() * x_p.element_size() + idx_p.numel() * 4
           + wt_p.numel() * 4)
    d2h = outs_p[0].numel() * outs_p[0].element_size()
    return {"ms_per_step": statistics.median(t["ms_per_step"] for t in trials),
            "link_ms_per_step": statistics.median(t["link_ms_per_step"] for t in trials),
            "trials": trials, "h2d": h2d, "d2h": d2h, "steps": steps}


# ---------------------------------------------------------------------------
# the oracle on the host (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

class OracleHost:
    """The CPU oracle on the host cores, as it stands.  Layout and notify run
    on one thread over the whole batch (the oracle's definitions walk the
    pairs in order); dispatch and combine are split by contiguous token
    ranges over ``threads`` threads, each calling the unchanged
    single-threaded oracle on its range (ctypes releases the GIL during the
    C call).  Outputs go to arrays allocated once here, so the timed calls
    do not include allocation."""

    def __init__(self, w, idx_h, wt_h, x_h, y_h, threads):
        import oracle as o
        from concurrent.futures import ThreadPoolExecutor
        self.o, self.w = o, w
        self.idx, self.wt = idx_h.numpy(), wt_h.numpy()
        self.x, self.y = W.bits(x_h), W.bits(y_h)
        S = o.row_bytes(w.H, w.quant)
        self.images = np.empty((w.T, w.k, S), np.uint8)
        self.row_ids = np.empty((w.T, w.k), np.int64)
        self.out = np.empty((w.T, w.H), np.uint16)
        self.tokens = np.arange(w.T, dtype=np.int64)
        cuts = np.linspace(0, w.T, max(1, threads) + 1).astype(np.int64)
        self.parts = [(int(a), int(c)) for a, c in zip(cuts[:-1], cuts[1:]) if c > a]
        self.threads = max(1, len(self.parts))
        self.pool = ThreadPoolExecutor(self.threads)
        self.L = self.N = None

    def close(self):
        self.pool.shutdown()

    def layout_notify(self):
        w, o = self.w, self.o
        t0 = time.perf_counter()
        self.L = o.layout(self.idx, w.R, w.epr)
        t1 = time.perf_counter()
        self.N = o.notify(self.L["count"], w.R, w.bs, w.epr)
        t2 = time.perf_counter()
        assert self.L["status"] == 0 and self.N["status"] == 0
        return t1 - t0, t2 - t1

    def dispatch(self, toks, images, row_ids):
        w, L, N = self.w, self.L, self.N
        _, _, st = self.o.dispatch_tokens(
            self.x, self.idx, L["send_idx"], N["put_offset"], N["rank_recv_base"],
            w.R, w.epr, w.dtype, w.quant, toks, images=images, row_ids=row_ids)
        return st

    def combine(self, toks, out):
        w, L, N = self.w, self.L, self.N
        _, st = self.o.combine(self.y, self.idx, self.wt, L["send_idx"],
                               N["put_offset"], N["rank_recv_base"], w.R, w.epr,
                               w.dtype, tokens=toks, out=out)
        return st

    def _over_parts(self, fn):
        futs = [self.pool.submit(fn, a, c) for a, c in self.parts]
        sts = [f.result() for f in futs]
        assert all(st == 0 for st in sts), sts

    def step(self):
        """One whole step on all tokens; seconds per stage."""
        t_lay, t_not = self.layout_notify()
        t0 = time.perf_counter()
        self._over_parts(lambda a, c: self.dispatch(self.tokens[a:c], self.images[a:c],
                                                    self.row_ids[a:c]))
        t1 = time.perf_counter()
        self._over_parts(lambda a, c: self.combine(self.tokens[a:c], self.out[a:c]))
        t2 = time.perf_counter()
        return {"layout": t_lay, "notify": t_not, "dispatch": t1 - t0,
                "combine": t2 - t1}

    def one_thread(self, toks):
        """Dispatch and combine of the listed tokens on this thread alone;
        returns (seconds per stage, images, row_ids, out)."""
        images = np.empty((toks.size,) + self.images.shape[1:], np.uint8)
        row_ids = np.empty((toks.size, self.w.k), np.int64)
        out = np.empty((toks.size, self.w.H), np.uint16)
        t0 = time.perf_counter()
        assert self.dispatch(toks, images, row_ids) == 0
        t1 = time.perf_counter()
        assert self.combine(toks, out) == 0
        t2 = time.perf_counter()
        return {"dispatch": t1 - t0, "combine": t2 - t1}, images, row_ids, out


def host_cpu():
    """The host CPU's model string and usable core count (for the CPU baseline)."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    if not model:                       # Arm hosts: /proc/cpuinfo names no model
        try:
            out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
            for line in out.splitlines():
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except (OSError, subprocess.SubprocessError):
            pass
    model = model or platform.processor() or platform.machine()
    try:
        avail = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        avail = os.cpu_count() or 1
    return model, avail


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline(w, idx_h, wt_h, x_h, y_h, seconds, threads=None):
    """The oracle timed on the host: a whole step on every host core (layout
    and notify on one thread, dispatch and combine split by token ranges),
    and dispatch + combine on one thread over a random token sample that
    takes about ``seconds``, scaled to the batch.  The sample's outputs must
    equal the all-core run's for the same tokens byte for byte."""
    threads = threads or host_threads()
    oh = OracleHost(w, idx_h, wt_h, x_h, y_h, threads)
    try:
        oh.step()                                  # first touch of the outputs
        runs = [oh.step() for _ in range(2)]
        stages = {k: float(np.median([r[k] for r in runs])) for k in runs[0]}
        all_s = sum(stages.values())
        rng = np.random.default_rng(0)
        probe = np.sort(rng.choice(w.T, size=min(w.T, 16), replace=False))
        t1, _, _, _ = oh.one_thread(probe)
        per_tok = (t1["dispatch"] + t1["combine"]) / probe.size
        n = int(min(w.T, max(16, seconds / max(per_tok, 1e-9))))
        sample = np.sort(rng.choice(w.T, size=n, replace=False))
        t1, images, row_ids, out = oh.one_thread(sample)
        identical = (np.array_equal(images, oh.images[sample])
                     and np.array_equal(row_ids, oh.row_ids[sample])
                     and np.array_equal(out, oh.out[sample]))
        if not identical:
            raise RuntimeError("%s: the all-core oracle differs from the one-thread "
                               "oracle on the sample" % w.name)
        one_s = (stages["layout"] + stages["notify"]
                 + (t1["dispatch"] + t1["combine"]) * w.T / n)
        model, avail = host_cpu()
        return {
            "value": w.T / all_s, "unit": "tokens/s", "cores": oh.threads,
            "kind": "oracle", "cpu": model, "host_cores_available": avail,
            "stages_ms": {k: v * 1e3 for k, v in stages.items()},
            "sample": "whole batch of %d tokens per step (median of 2 steps after "
                      "one untimed): layout+notify on 1 thread, dispatch+combine "
                      "split by token ranges over %d threads" % (w.T, oh.threads),
            "one_core": {
                "value": w.T / one_s, "cores": 1,
                "stages_ms": {"dispatch": t1["dispatch"] * 1e3 * w.T / n,
                              "combine": t1["combine"] * 1e3 * w.T / n},
                "sample": "dispatch+combine of %s on one thread (%.2f s), scaled "
                          "to the batch; layout+notify as above"
                          % ("all %d tokens" % n if n == w.T else "%d random tokens" % n,
                             t1["dispatch"] + t1["combine"])},
            "identical_to_one_thread": identical,
        }
    finally:
        oh.close()


def run_reference(args, w):
    """The reference arm: the CPU oracle, as it stands, on the host cores.
    Each step is the whole pipeline on the whole batch (see OracleHost)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None                       # rank 0 alone runs the oracle
    idx_h, wt_h = W.routing(w)
    x_h = W.tokens(w)
    y_h = W.expert_outputs(w)
    oh = OracleHost(w, idx_h, wt_h, x_h, y_h, host_threads())
    try:
        for i in range(args.warmup):
            oh.step()
        runs = []
        t0 = time.perf_counter()
        for i in range(args.steps):
            runs.append(oh.step())
        wall = time.perf_counter() - t0
    finally:
        oh.close()
    step_s = wall / args.steps
    value = w.T / step_s
    model, avail = host_cpu()
    stages = {k: float(np.mean([r[k] for r in runs])) * 1e3 for k in runs[0]}
    return {
        "impl": "reference",
        "metric": "dispatch+combine tokens/s",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_s * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": step_config(w, world),
        "arm": "the CPU oracle on the host cores: the same step on the same inputs, "
               "in host memory",
        "stages_ms": stages,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oh.threads,
                         "kind": "oracle", "cpu": model,
                         "host_cores_available": avail,
                         "sample": "every step: the whole batch of %d tokens; "
                                   "layout+notify on 1 thread, dispatch+combine "
                                   "split by token ranges over %d threads"
                                   % (w.T, oh.threads)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
        "wall_s_timed_region": wall,
    }


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--workload", default="dsv3", choices=W.ORDER)
    p.add_argument("--impl", default="moe_ep", choices=["moe_ep", "reference"])
    p.add_argument("--e2e-steps", type=int, default=30)
    p.add_argument("--clocks-csv", default=None,
                   help="where the nvidia-smi clock samples of the timed steps go "
                        "(default: a file in /tmp)")
    p.add_argument("--cpu-seconds", type=float, default=2.0,
                   help="one-thread oracle sample per workload (seconds)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-per-config", action="store_true",
                   help="time the named workload only")
    p.add_argument("--per-config-steps", type=int, default=20,
                   help="timed steps of each non-headline workload")
    p.add_argument("--no-deep-moe", action="store_true",
                   help="skip the fused deep MoE section")
    p.add_argument("--gemm", default=None, metavar="G,ROWS,N,K",
                   help="time the grouped GEMM alone and exit")
    p.add_argument("--gemm-epilogue", default="int32", choices=["int32", "dequant", "swiglu"],
                   help="epilogue of the --gemm benchmark")
    p.add_argument("--bs", type=int, default=None,
                   help="override tokens per rank (small profiling cases)")
    p.add_argument("--hidden", type=int, default=None,
                   help="override the hidden size (profiling the index stages "
                        "at full pair count with small rows)")
    return p.parse_args(argv)


def main(argv=None):
    args = parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.gemm:
        run_gemm_only(args)
        return
    w = W.WORKLOADS[args.workload]
    if args.bs is not None:
        w = w.with_(bs=args.bs)
    if args.hidden is not None:
        w = w.with_(H=args.hidden)
    world, rank, _ = dist_env()
    if world != args.gpus and not (world == 1 and args.gpus == 1):
        raise SystemExit("--gpus %d but WORLD_SIZE=%d; launch N>1 with torchrun"
                         % (args.gpus, world))
    rec = run_reference(args, w) if args.impl == "reference" else run_gpu(args, w)
    if rec is not None and rank == 0:
        print(json.dumps(rec), flush=True)
    if args.impl != "reference" and torch.distributed.is_initialized():
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
