"""Concurrent use: two host threads, each with its own stream and buffers,
run the four-stage pipeline on different shapes at the same time, many times
over (the one-launch dispatch, a cooperative launch sized to the whole GPU,
is left out: two of those must not share the GPU).  The library's only process-wide state
is the per-device launch-fact cache (behind a mutex) and the allocation-free
entry point's scratch array (not used here); everything else lives in the
caller's buffers.  Every result must equal its oracle bit for bit, whatever
the interleaving of the two threads' host calls and of their kernels on the
GPU."""
import threading

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pl():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from combine_moe_dispatch_layout_gb300 import pipeline
    return pipeline


def _reference(oracle, w, idx, wt, x, y):
    L = oracle.layout(idx.numpy(), w.R, w.epr)
    N = oracle.notify(L["count"], w.R, w.bs, w.epr)
    recv, _ = oracle.dispatch(W.bits(x), idx.numpy(), L["send_idx"], N["put_offset"],
                              N["rank_recv_base"], w.R, w.epr, w.dtype, w.quant)
    out, _ = oracle.combine(W.bits(y), idx.numpy(), wt.numpy(), L["send_idx"],
                            N["put_offset"], N["rank_recv_base"], w.R, w.epr, w.dtype)
    return L, N, recv, out


def test_two_threads_two_streams(oracle_mod, pl):
    shapes = [W.Workload("cc_a", R=3, epr=5, bs=700, k=7, H=1000, seed=81),
              W.Workload("cc_b", R=4, epr=6, bs=500, k=5, H=520, quant=False,
                         dtype=W.FP16, x_dist="uniform", x_scale=4.0, seed=82)]
    jobs = []
    for w in shapes:
        idx, wt = W.routing(w)
        x, y = W.tokens(w), W.expert_outputs(w)
        ref = _reference(oracle_mod, w, idx, wt, x, y)
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            b = pl.PipelineBuffers(w.R, w.bs, w.k, w.epr, w.H, w.dtype, w.quant)
            dev = (idx.cuda(), wt.cuda(), x.cuda(), y.cuda())
        torch.cuda.synchronize()
        jobs.append(dict(w=w, ref=ref, st=st, b=b, dev=dev, errors=[]))

    def work(job, rounds):
        try:
            with torch.cuda.stream(job["st"]):
                idx_d, wt_d, x_d, y_d = job["dev"]
                for _ in range(rounds):
                    pl.run_pipeline(job["b"], x_d, idx_d, wt_d, y_d, job["st"])
            job["st"].synchronize()
        except Exception as e:       # reported by the main thread
            job["errors"].append(repr(e))

    for _ in range(3):
        threads = [threading.Thread(target=work, args=(j, 20)) for j in jobs]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        torch.cuda.synchronize()
        for j in jobs:
            assert not j["errors"], j["errors"]
            b = j["b"]
            L, N, recv, out = j["ref"]
            assert b.status() == 0
            assert np.array_equal(b.send_idx.cpu().numpy(), L["send_idx"])
            assert np.array_equal(b.put_offset.cpu().numpy(), N["put_offset"])
            assert np.array_equal(b.rank_recv_base.cpu().numpy(), N["rank_recv_base"])
            assert np.array_equal(b.recv.cpu().numpy(), recv)
            got = b.out.view(torch.int16).cpu().numpy().view(np.uint16)
            assert np.array_equal(got.reshape(out.shape), out)
