"""moe_dispatch_layout_static: the layout entry point that allocates nothing.

It exists for callers that cannot allocate device memory (a plugin handed
only its input and output buffers, or a serving loop whose memory is all
reserved up front).  These tests call it through the C ABI and compare its
outputs with the regular entry point's (which takes a caller-allocated
workspace) and with the CPU oracle's layout, bit for bit, on two calls in a
row with different routings, so that the second call cannot pass on what
the first left in the shared scratch array.  The file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import combine_moe_dispatch_layout_gb300 as ep
    L = ep.lib()
    fn = L.moe_dispatch_layout_static
    fn.argtypes = [ctypes.POINTER(ep.moe_shape)] + [ctypes.c_void_p] * 6
    fn.restype = ctypes.c_int
    return ep, L


def _run_both(ep, L, w, seed, stream=None):
    w = w.with_(seed=seed)
    idx_h, _ = W.routing(w)
    idx = idx_h.cuda()
    shape = ep.make_shape(w.R, w.bs, w.k, w.epr, w.H)
    E, T = w.E, w.T

    def outs():
        return (torch.full((w.R, E), -7, dtype=torch.int32, device="cuda"),
                torch.full((w.R, w.R), -7, dtype=torch.int32, device="cuda"),
                torch.full((T, w.k), -7, dtype=torch.int32, device="cuda"),
                torch.zeros(1, dtype=torch.int32, device="cuda"))

    # the existing entry point, with a caller-allocated zeroed workspace
    c1, r1, s1, st1 = outs()
    ws = torch.zeros(max(16, ep.layout_workspace_bytes(shape)),
                     dtype=torch.uint8, device="cuda")
    ep.moe_dispatch_layout(shape, idx, c1, r1, s1, ws, st1)
    # the allocation-free entry point, through the C ABI
    c2, r2, s2, st2 = outs()
    st = torch.cuda.current_stream() if stream is None else stream
    st.wait_stream(torch.cuda.current_stream())
    rc = L.moe_dispatch_layout_static(
        ctypes.byref(shape), ctypes.c_void_p(idx.data_ptr()),
        ctypes.c_void_p(c2.data_ptr()), ctypes.c_void_p(r2.data_ptr()),
        ctypes.c_void_p(s2.data_ptr()), ctypes.c_void_p(st2.data_ptr()),
        ctypes.c_void_p(st.cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0, ep.status_string(rc)
    assert int(st1.item()) == 0 and int(st2.item()) == 0
    # integer outputs: the tolerance is zero
    assert torch.equal(c1, c2)
    assert torch.equal(r1, r2)
    assert torch.equal(s1, s2)
    # and the oracle's layout of the same routing
    ref = oracle.layout(idx_h.numpy(), w.R, w.epr)
    assert ref["status"] == 0
    np.testing.assert_array_equal(c2.cpu().numpy(), ref["count"])
    np.testing.assert_array_equal(r2.cpu().numpy(), ref["rank_send"])
    np.testing.assert_array_equal(s2.cpu().numpy(), ref["send_idx"])


@pytest.mark.parametrize("w", [
    W.WORKLOADS["dsv3"],                       # 8 tiles per rank (look-back)
    W.WORKLOADS["maxrank"],                    # 384 ranks, one tile each
    W.Workload("ragged", R=3, epr=5, bs=1500, k=7, H=64),
], ids=lambda w: w.name)
def test_static_matches_workspace_entry_two_calls(lib, w):
    ep, L = lib
    _run_both(ep, L, w, seed=101)
    _run_both(ep, L, w, seed=202)


def test_static_on_a_side_stream(lib):
    """Two calls in a row on a stream other than torch's current one."""
    ep, L = lib
    side = torch.cuda.Stream()
    w = W.Workload("ragged", R=5, epr=3, bs=700, k=4, H=64)
    _run_both(ep, L, w, seed=303, stream=side)
    _run_both(ep, L, w, seed=404, stream=side)


def test_static_rejects_shapes_beyond_the_array(lib):
    ep, L = lib
    # E = 4096 with 32 tiles per rank needs ~8.4 MB of scratch (> 4 MiB)
    shape = ep.make_shape(8, 8192, 8, 512, 64)
    assert ep.layout_workspace_bytes(shape) > (4 << 20)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = L.moe_dispatch_layout_static(ctypes.byref(shape), p, p, p, p, p,
                                      ctypes.c_void_p(0))
    assert rc == ep.MOE_ERR_INVALID_ARG
    assert int(dummy.abs().sum().item()) == 0       # nothing was enqueued
