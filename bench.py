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


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        ent = d[kernel][workload]
        if ent["source_sha256_16"] != _file_hash(KERNEL_SOURCES[kernel]):
            return None
        return float(ent["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


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

def run_gpu(args, w):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    init_dist(world, "nccl")
    import combine_moe_dispatch_layout_gb300 as ep  # noqa: F401 (loads the .so)
    from combine_moe_dispatch_layout_gb300 import pipeline as pl
    dev = torch.device("cuda", local)

    idx_h, wt_h = W.routing(w)
    x_h = W.tokens(w)
    y_h = W.expert_outputs(w)
    idx, wt, x = idx_h.to(dev), wt_h.to(dev), x_h.to(dev)
    y = y_h.to(dev)
    b = pl.PipelineBuffers(w.R, w.bs, w.k, w.epr, w.H, w.dtype, w.quant,
                           device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(evs=None, st=None):
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
        pl.run_combine(b, y, idx, wt, st)
        if evs:
            evs[4].record(st)

    for i in range(args.warmup):
        flush.fill_(i & 0xff)
        step()
    torch.cuda.synchronize()
    if b.status() != 0:
        raise RuntimeError("device status %d after warm-up" % b.status())

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)]
           for _ in range(args.steps)]
    clocks = ClockSampler(local, args.clocks_csv)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xff)        # between steps, outside the events
        step(evs[i])
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    clk = clocks.stop()
    if b.status() != 0:
        raise RuntimeError("device status %d after timed steps" % b.status())

    stage_ms = np.array([[evs[i][j].elapsed_time(evs[i][j + 1])
                          for j in range(4)] for i in range(args.steps)])
    step_ms = stage_ms.sum(axis=1)
    mean_step_ms = float(step_ms.mean())
    max_step_ms = reduce_max(mean_step_ms, world, dev)
    value = aggregate_tokens_per_s(w.T, world, max_step_ms / 1e3)
    stage_mean = stage_ms.mean(axis=0)
    ab = alg_bytes(w)
    names = ["layout", "notify", "dispatch", "combine"]
    peak, peak_kind = measured_peaks()
    gbs = {n: ab[n] / (stage_mean[j] * 1e-3) / 1e9 for j, n in enumerate(names)}

    # ---- combine over INT8 expert outputs (moe_combine_quant) -------------
    cq = None
    if w.quant:
        yq = W.expert_outputs_int8(w).to(dev)
        for i in range(3):
            pl.run_combine_quant(b, yq, idx, wt, stream)
        cq_ms = []
        for i in range(min(args.steps, EXTRA_STEPS)):
            flush.fill_(i & 0xff)
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            pl.run_combine_quant(b, yq, idx, wt, stream)
            c1.record(stream)
            cq_ms.append((c0, c1))
        torch.cuda.synchronize()
        if b.status() != 0:
            raise RuntimeError("device status %d in combine_quant" % b.status())
        cq_us = float(np.mean([a.elapsed_time(c) for a, c in cq_ms])) * 1e3
        cq_bytes = alg_bytes(w)["combine_quant"]
        cq = {"us": cq_us, "achieved_gbs": cq_bytes / (cq_us * 1e-6) / 1e9,
              "algorithmic_bytes": cq_bytes,
              "traffic": recorded_traffic("combine_quant", w.name),
              "frac": cq_bytes / (cq_us * 1e-6) / 1e9 / peak,
              "tokens_per_s": w.T / (cq_us * 1e-6)}
        del yq

    # ---- the same step replayed as a CUDA graph (no host enqueue cost) ------
    gs = torch.cuda.Stream(dev)
    gs.wait_stream(stream)
    with torch.cuda.stream(gs):
        step_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(step_graph, stream=gs):
            step(st=gs)
    stream.wait_stream(gs)
    graph_ev = []
    for i in range(min(args.steps, EXTRA_STEPS)):
        flush.fill_(i & 0xff)
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        step_graph.replay()
        g1.record(stream)
        graph_ev.append((g0, g1))
    torch.cuda.synchronize()
    if b.status() != 0:
        raise RuntimeError("device status %d in graph replay" % b.status())
    graph_us = float(np.mean([a.elapsed_time(c) for a, c in graph_ev])) * 1e3
    del step_graph

    # ---- one-launch low-latency dispatch vs the three separate launches ------
    def timed(fn, n):
        evs = []
        for i in range(n):
            flush.fill_(i & 0xff)
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            fn()
            a1.record(stream)
            evs.append((a0, a1))
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(c) for a, c in evs])) * 1e3
    for i in range(3):
        pl.run_dispatch_fused(b, x, idx, stream)
    fused_us = timed(lambda: pl.run_dispatch_fused(b, x, idx, stream),
                     min(args.steps, EXTRA_STEPS))
    if b.status() != 0:
        raise RuntimeError("device status %d in fused dispatch" % b.status())
    separate_us = float(stage_mean[0] + stage_mean[1] + stage_mean[2]) * 1e3

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
                                                  b.dev_status, stream),
                      min(args.steps, EXTRA_STEPS))
        sw_bytes = w.P * (8 * I + (I + 31) // 32 * 32 + 32 + 4) + 8 * I
        sw = {"us": sw_us, "rows": w.P, "I": I, "algorithmic_bytes": sw_bytes,
              "traffic": recorded_traffic("swiglu_quant", w.name),
              "achieved_gbs": sw_bytes / (sw_us * 1e-6) / 1e9,
              "frac": sw_bytes / (sw_us * 1e-6) / 1e9 / peak}
        del acc_d, sw_out

    # ---- token-level layout (moe_token_layout) ------------------------------
    tpr = torch.empty((w.R, w.R), dtype=torch.int32, device=dev)
    inr = torch.empty((w.T, w.R), dtype=torch.uint8, device=dev)
    for i in range(3):
        ep.moe_token_layout(b.shape, idx, tpr, inr, b.dev_status, stream)
    tl_ev = []
    for i in range(min(args.steps, EXTRA_STEPS)):
        flush.fill_(i & 0xff)
        t0e = torch.cuda.Event(enable_timing=True)
        t1e = torch.cuda.Event(enable_timing=True)
        t0e.record(stream)
        ep.moe_token_layout(b.shape, idx, tpr, inr, b.dev_status, stream)
        t1e.record(stream)
        tl_ev.append((t0e, t1e))
    torch.cuda.synchronize()
    if b.status() != 0:
        raise RuntimeError("device status %d in token_layout" % b.status())
    tl_us = float(np.mean([a.elapsed_time(c) for a, c in tl_ev])) * 1e3
    del tpr, inr

    # ---- fused deep MoE (dispatch -> GMM1 -> DeqSwigluQuant -> GMM2 ->
    #      DeqCombine) on the same routing and tokens ------------------------
    deep = None
    if w.quant and w.E <= 256 and not args.no_deep_moe:   # weights: E x 44 M codes
        deep = run_deep_moe_bench(args, w, ep, pl, x, idx, wt, stream, dev, flush)

    # ---- end to end through the public API with host buffers --------------
    e2e = run_e2e(args, w, b, pl, idx_h, wt_h, x_h, y, stream, dev, flush)
    e2e_max_ms = reduce_max(e2e["ms_per_step"], world, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, idx_h, wt_h, x_h, y_h, args.cpu_seconds)

    if rank != 0:
        return None
    comb_ms = float(stage_mean[3])
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
        "data": "synthetic",
        "config": {
            "workload": workload_desc(w),
            "step": "layout+notify+dispatch+combine, inputs resident in HBM",
            "l2": "flushed between steps (256 MiB write outside the step events)",
            "parallelism": "replicas" if world > 1 else "single GPU",
            "io_dtype": "bf16" if w.dtype == W.BF16 else "fp16",
            "recv_rows": "int8 + fp32 1/scale" if w.quant else "verbatim",
        },
        "roofline": {
            "kernel": "combine",
            "bound": "hbm",
            "achieved": gbs["combine"],
            "peak": peak,
            "peak_source": peak_kind,
            "unit": "GB/s",
            "frac": gbs["combine"] / peak,
            "traffic": recorded_traffic("combine", w.name),
            "algorithmic_bytes": ab["combine"],
            "avg_launch_ms": comb_ms,
        },
        "roofline_dispatch": {
            "bound": "hbm", "achieved": gbs["dispatch"], "peak": peak,
            "unit": "GB/s", "frac": gbs["dispatch"] / peak,
            "traffic": recorded_traffic("dispatch", w.name),
            "algorithmic_bytes": ab["dispatch"],
            "avg_launch_ms": float(stage_mean[2]),
        },
        "combine_quant": cq,
        "token_layout_us": tl_us,
        "graph_step_us": graph_us,
        "swiglu_quant": sw,
        "deep_moe": deep,
        "dispatch_fused": {"us": fused_us, "separate_us": separate_us,
                           "note": "layout+notify+dispatch in one cooperative "
                                   "launch vs three launches"},
        "stages_us": {n: float(stage_mean[j] * 1e3) for j, n in enumerate(names)},
        "stages_gbs": gbs,
        "dispatch_combine_tokens_per_s": w.T / ((stage_mean[2] + stage_mean[3]) * 1e-3),
        "e2e": {"value": aggregate_tokens_per_s(w.T, world, e2e_max_ms / 1e3),
                "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": e2e_max_ms, "steps": e2e["steps"],
                "note": "every step copies x, topk_idx, topk_weights from pinned "
                        "host memory and out back inside the timed region; copies "
                        "of neighbouring steps overlap compute (3 streams); expert "
                        "outputs y stay on the device (they are produced there)"},
        "gpu_launches": 4 * args.steps,
        "clocks": clk,
        "wall_s_timed_region": wall,
        "cpu_baseline": cpu,
    }
    return rec


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

    def one(i):
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
        pl.run_pipeline(b, x_d[j], idx_d[j], wt_d[j], y, stream)
        consumed[j].record(stream)
        with torch.cuda.stream(s_d2h):
            s_d2h.wait_event(consumed[j])
            outs_p[j].copy_(out_d[j], non_blocking=True)
            drained[j].record(s_d2h)

    for i in range(n_warm):
        one(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s_h2d)
    for i in range(steps):
        one(n_warm + i)
    s_d2h.wait_event(consumed[(n_warm + steps - 1) % 2])
    e1.record(s_d2h)
    torch.cuda.synchronize()
    b.out = out_d[0]
    if b.status() != 0:
        raise RuntimeError("device status %d in e2e" % b.status())
    h2d = (x_p.numel() * x_p.element_size() + idx_p.numel() * 4
           + wt_p.numel() * 4)
    d2h = outs_p[0].numel() * outs_p[0].element_size()
    return {"ms_per_step": e0.elapsed_time(e1) / steps, "h2d": h2d, "d2h": d2h,
            "steps": steps}


# ---------------------------------------------------------------------------
# the oracle on the host (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------

def _oracle_step(o, w, idx_np, wt_np, x_bits, y_bits, tokens):
    """One bounded sample: layout + notify over the whole batch, then
    dispatch and combine of the sampled tokens.  Returns seconds per phase."""
    t0 = time.perf_counter()
    L = o.layout(idx_np, w.R, w.epr)
    N = o.notify(L["count"], w.R, w.bs, w.epr)
    t1 = time.perf_counter()
    o.dispatch_tokens(x_bits, idx_np, L["send_idx"], N["put_offset"],
                      N["rank_recv_base"], w.R, w.epr, w.dtype, w.quant, tokens)
    o.combine(y_bits, idx_np, wt_np, L["send_idx"], N["put_offset"],
              N["rank_recv_base"], w.R, w.epr, w.dtype, tokens=tokens)
    t2 = time.perf_counter()
    return t1 - t0, t2 - t1


def _oracle_tokens_per_s(w, t_ln, t_dc, n):
    """Full-batch tokens/s extrapolated from the sample: layout+notify ran on
    all T tokens, dispatch+combine on n of them."""
    return w.T / (t_ln + t_dc * w.T / n)


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


def cpu_baseline(w, idx_h, wt_h, x_h, y_h, seconds):
    import oracle as o
    idx_np, wt_np = idx_h.numpy(), wt_h.numpy()
    x_bits, y_bits = W.bits(x_h), W.bits(y_h)
    rng = np.random.default_rng(0)
    probe = np.sort(rng.choice(w.T, size=min(w.T, 64), replace=False))
    t_ln, t_dc = _oracle_step(o, w, idx_np, wt_np, x_bits, y_bits, probe)
    per_tok = t_dc / len(probe)
    n = int(min(w.T, max(64, (seconds - t_ln) / max(per_tok, 1e-9))))
    tokens = np.sort(rng.choice(w.T, size=n, replace=False))
    t_ln, t_dc = _oracle_step(o, w, idx_np, wt_np, x_bits, y_bits, tokens)
    model, avail = host_cpu()
    return {"value": _oracle_tokens_per_s(w, t_ln, t_dc, n), "unit": "tokens/s",
            "cores": 1, "kind": "oracle", "cpu": model, "host_cores_available": avail,
            "sample": "layout+notify on all %d tokens (%.2f ms), dispatch+combine on %s "
                      "(%.2f s)%s"
                      % (w.T, t_ln * 1e3,
                         "all %d tokens" % n if n == w.T else "%d random tokens" % n, t_dc,
                         "" if n == w.T else ", scaled to the full batch")}


def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return None                       # rank 0 alone runs the oracle
    import oracle as o
    idx_h, wt_h = W.routing(w)
    x_h = W.tokens(w)
    y_h = W.expert_outputs(w)
    idx_np, wt_np = idx_h.numpy(), wt_h.numpy()
    x_bits, y_bits = W.bits(x_h), W.bits(y_h)
    rng = np.random.default_rng(1)
    n = min(w.T, args.ref_tokens)
    samples = [np.sort(rng.choice(w.T, size=n, replace=False))
               for _ in range(args.warmup + args.steps)]
    for i in range(args.warmup):
        _oracle_step(o, w, idx_np, wt_np, x_bits, y_bits, samples[i])
    secs = []
    t0 = time.perf_counter()
    for i in range(args.steps):
        t_ln, t_dc = _oracle_step(o, w, idx_np, wt_np, x_bits, y_bits,
                                  samples[args.warmup + i])
        secs.append(t_ln + t_dc * w.T / n)
    wall = time.perf_counter() - t0
    step_s = float(np.mean(secs))
    value = w.T / step_s
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
        "config": {"workload": workload_desc(w),
                   "step": "layout+notify+dispatch+combine (CPU oracle)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1,
                         "kind": "oracle", "cpu": host_cpu()[0],
                         "host_cores_available": host_cpu()[1],
                         "sample": "each step: layout+notify on all %d tokens, "
                                   "dispatch+combine on %d random tokens, "
                                   "scaled to the full batch" % (w.T, n)},
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
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-deep-moe", action="store_true",
                   help="skip the fused deep MoE section")
    p.add_argument("--gemm", default=None, metavar="G,ROWS,N,K",
                   help="time the grouped GEMM alone and exit")
    p.add_argument("--gemm-epilogue", default="int32", choices=["int32", "dequant", "swiglu"],
                   help="epilogue of the --gemm benchmark")
    p.add_argument("--ref-tokens", type=int, default=32)
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
