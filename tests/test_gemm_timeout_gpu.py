"""The grouped GEMM's timeout path on the GPU, without a fault or a hang.

The kernel bounds every mbarrier wait; a main-loop wait that runs out sets
MOE_ERR_TIMEOUT, stops the CTA issuing work and drains what it already
issued (TMA fills, MMAs, their commits, tile stores) under the full bound
before TMEM is released.  The library exports a test hook,
moe_test_grouped_gemm_i8_polls (not part of the public header), that runs
moe_grouped_gemm_i8 with the main-loop waits limited to a given number of
polls.  With 0 polls the first wait of every working CTA gives up; with a
few polls the waits give up wherever the pipeline happens to be.  Checks:
the status is MOE_ERR_TIMEOUT (or 0, when a few polls sufficed), nothing is
written outside c, every value written inside c is the exact result (a
chunk cut short never reaches the epilogue), and a normal call on the same
buffers right after gives the exact int32 GEMM.  The step-by-step model of
the same protocol is tests/test_gemm_pipeline_model.py."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

SENTINEL = -0x5A5A5A5B


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import combine_moe_dispatch_layout_gb300 as ep
    fn = ep.lib().moe_test_grouped_gemm_i8_polls
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                   ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
                   ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return ep


def _case(ep, sizes, N, K, seed):
    rng = np.random.default_rng(seed)
    M = sum(sizes)
    G = len(sizes)
    a = rng.integers(-127, 128, (M, K)).astype(np.int8)
    w = rng.integers(-127, 128, (G, N, K)).astype(np.int8)
    dev = torch.device("cuda")
    a_bf = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    w_bf = torch.empty((G, N, K), dtype=torch.bfloat16, device=dev)
    ep.moe_codes_to_bf16(torch.from_numpy(a.view(np.uint8)).to(dev), M, K, K, a_bf)
    ep.moe_codes_to_bf16(torch.from_numpy(w.view(np.uint8)).to(dev), G * N, K, K, w_bf)
    gr = torch.tensor(sizes, dtype=torch.int32, device=dev)
    # c sits between two guard regions of 64 int32 (256 bytes: c stays 16-byte aligned)
    buf = torch.full((64 + M * N + 64,), SENTINEL, dtype=torch.int32, device=dev)
    c = buf[64:64 + M * N].view(M, N)
    ref = np.zeros((M, N), np.int64)
    off = np.concatenate([[0], np.cumsum(sizes)])
    for g in range(G):
        ref[off[g]:off[g + 1]] = a[off[g]:off[g + 1]].astype(np.int64) @ w[g].T.astype(np.int64)
    return a_bf, w_bf, gr, buf, c, ref.astype(np.int32)


def _hook(ep, a_bf, w_bf, gr, c, polls, st):
    M, K = a_bf.shape
    G, N, _ = w_bf.shape
    return ep.lib().moe_test_grouped_gemm_i8_polls(
        a_bf.data_ptr(), M, K, w_bf.data_ptr(), G, N, gr.data_ptr(), c.data_ptr(), polls,
        st.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("sizes,N,K,polls", [
    ((100,), 256, 512, 0),           # one group, one tile: every wait gives up at once
    ((100,), 256, 512, 1),           # ... or after one poll
    ((130, 0, 300), 512, 2048, 0),   # several tiles, two K chunks
    ((130, 0, 300), 512, 2048, 1),
    ((130, 0, 300), 512, 2048, 4),
    ((700, 45), 264, 1104, 2),       # a ragged column tile and a ragged K chunk
], ids=lambda v: str(v).replace(" ", ""))
def test_main_loop_timeout_then_a_normal_call(ep, sizes, N, K, polls):
    a_bf, w_bf, gr, buf, c, ref = _case(ep, sizes, N, K, seed=sum(sizes) + N + K + polls)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _hook(ep, a_bf, w_bf, gr, c, polls, st)
    torch.cuda.synchronize()
    assert rc == 0, ep.status_string(rc)
    status = int(st.item())
    if polls == 0:
        assert status == ep.MOE_ERR_TIMEOUT
    else:
        assert status in (0, ep.MOE_ERR_TIMEOUT)
    host = buf.cpu().numpy()
    assert (host[:64] == SENTINEL).all() and (host[-64:] == SENTINEL).all(), \
        "a write outside c"
    got = host[64:-64].reshape(ref.shape)
    written = got != SENTINEL
    assert np.array_equal(got[written], ref[written]), "a partial result was stored"
    if polls == 0:
        assert not written.any()           # no wait passed: nothing was computed
    if status == 0:
        assert np.array_equal(got, ref)
    # the same buffers, a normal call: the exact int32 GEMM
    st.zero_()
    c.fill_(SENTINEL)
    ep.moe_grouped_gemm_i8(a_bf, w_bf, gr, c, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    host = buf.cpu().numpy()
    assert (host[:64] == SENTINEL).all() and (host[-64:] == SENTINEL).all()
    assert np.array_equal(host[64:-64].reshape(ref.shape), ref)
