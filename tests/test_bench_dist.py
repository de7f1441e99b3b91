"""bench.py's multi-rank host logic on CPU with gloo, world size 2.

With N GPUs the benchmark runs N independent replicas of the pipeline (one
per rank, no data-path collective); ranks only meet in a barrier and a
max-reduction of the step time, and rank 0 reports the whole-job
throughput.  These tests run that host logic with two gloo ranks, and the
reference arm (the CPU oracle) under torchrun with two ranks.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    w, r, _ = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    step_ms = [1.5, 2.5][rank]            # rank 1 is the slow one
    mx = bench.reduce_max(step_ms, w)
    tps = bench.aggregate_tokens_per_s(32768, w, mx / 1e3)
    out.put((rank, mx, tps))
    torch.distributed.destroy_process_group()


def test_reduce_max_and_aggregate_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]          # both see the max
    # whole job: 2 replicas x 32768 tokens over the slowest rank's 2.5 ms
    assert res[0][2] == pytest.approx(2 * 32768 / 2.5e-3)


def test_single_rank_helpers():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.0, 1) == 3.0
    assert bench.aggregate_tokens_per_s(100, 1, 0.5) == 200.0
    b = bench.alg_bytes(__import__("workloads").WORKLOADS["dsv3"])
    assert b["combine"] == 4231004160          # P*H*2 + P*12 + T*H*2
    assert b["dispatch"] == (32768 * 7168 * 2 + 262144 * 7200 + 262144 * 8
                             + 256 * 8 * 4 + 9 * 8)


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           "--nproc-per-node=2", "--master-addr=127.0.0.1",
           "--master-port=%d" % port, os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "tiny",
           "--steps", "3", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1                     # rank 0 alone prints
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    assert rec["value"] > 0 and rec["e2e"]["h2d_bytes_per_step"] == 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
    # the same metric, unit, direction and config object as the GPU arm
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    assert rec["config"] == bench.step_config(W.WORKLOADS["tiny"], 2)
    assert rec["metric"] == "dispatch+combine tokens/s" and rec["unit"] == "tokens/s"
    assert rec["higher_is_better"] is True and rec["e2e"]["value"] == rec["value"]


def test_cpu_baseline_leg_on_the_host():
    """The cpu_baseline object the GPU arm adds: the oracle timed on the host
    cores over the whole batch (dispatch and combine split over threads),
    with the one-thread figure beside it and the keys the JSON line needs."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    w = W.WORKLOADS["tiny"]
    idx, wt = W.routing(w)
    cb = bench.cpu_baseline(w, idx, wt, W.tokens(w), W.expert_outputs(w), 0.5,
                            threads=3)
    assert cb["kind"] == "oracle" and cb["cores"] == 3 and cb["unit"] == "tokens/s"
    assert cb["value"] > 0 and cb["host_cores_available"] >= 1
    assert cb["identical_to_one_thread"] is True
    assert cb["one_core"]["cores"] == 1 and cb["one_core"]["value"] > 0
    assert "all %d tokens" % w.T in cb["one_core"]["sample"]
    assert set(cb["stages_ms"]) == {"layout", "notify", "dispatch", "combine"}


@pytest.mark.parametrize("threads", [1, 4, 7])
def test_threaded_oracle_equals_the_whole_batch_oracle(threads):
    """The all-core timing runs the oracle's dispatch and combine over token
    ranges on several threads; the assembled outputs must be byte-identical
    to one call over the whole batch (a ragged split: T not a multiple of
    the thread count)."""
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    import oracle
    import workloads as W
    w = W.Workload("small", R=3, epr=5, bs=37, H=96, k=4, seed=77)
    idx, wt = W.routing(w)
    x, y = W.tokens(w), W.expert_outputs(w)
    oh = bench.OracleHost(w, idx, wt, x, y, threads)
    try:
        oh.step()
    finally:
        oh.close()
    L = oracle.layout(idx.numpy(), w.R, w.epr)
    N = oracle.notify(L["count"], w.R, w.bs, w.epr)
    images, rows, st = oracle.dispatch_tokens(
        W.bits(x), idx.numpy(), L["send_idx"], N["put_offset"], N["rank_recv_base"],
        w.R, w.epr, w.dtype, w.quant, np.arange(w.T))
    out, st2 = oracle.combine(W.bits(y), idx.numpy(), wt.numpy(), L["send_idx"],
                              N["put_offset"], N["rank_recv_base"], w.R, w.epr, w.dtype)
    assert st == 0 and st2 == 0
    assert np.array_equal(images, oh.images)
    assert np.array_equal(rows, oh.row_ids)
    assert np.array_equal(out, oh.out)


@pytest.mark.parametrize("name,dispatch_gb,combine_gb", [
    ("dsv3", 2.359, 4.231), ("skew", 1.082, 1.881), ("fp16", 1.210, 1.211),
    ("maxrank", 3.540, 6.347)])
def test_algorithmic_bytes_all_workloads(name, dispatch_gb, combine_gb):
    """The roofline numerators: dispatch moves x once, k row images and the
    pair indices (plus the count matrix and bases); combine moves k expert
    rows, the pair indices and weights, and the output once.  Stated to
    1 MB per workload."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads as W
    b = bench.alg_bytes(W.WORKLOADS[name])
    assert b["dispatch"] / 1e9 == pytest.approx(dispatch_gb, abs=1e-3)
    assert b["combine"] / 1e9 == pytest.approx(combine_gb, abs=1e-3)


def test_clock_record_parsing(tmp_path):
    """The clocks object of the JSON line from nvidia-smi's CSV rows: median SM
    clock under load, the maximum, and every throttle reason seen Active (a
    run with a slowdown reason is rejected, so the parse must see it)."""
    sys.path.insert(0, ROOT)
    import bench

    class Done:                            # stands in for the finished nvidia-smi
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    rows = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1980, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 2070, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 1500, 2070, 1400.0, 0x8, Active, Not Active, Not Active, Not Active"]
    s = bench.ClockSampler(0, path=str(tmp_path / "clocks.csv"))
    s.f = open(s.path, "w")
    s.f.write("\n".join(rows) + "\n")
    s.proc = Done()
    rec = s.stop()
    assert rec["samples"] == 4 and rec["sm_max_mhz"] == 2070.0
    assert rec["sm_mhz"] == 2025.0                     # median of 1500, 1980, 2070, 2070
    assert rec["reasons"] == ["hw_slowdown", "sw_power_cap"]
