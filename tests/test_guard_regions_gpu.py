"""Out-of-bounds and coverage checks on the GPU without a sanitizer.

Every output and scratch buffer of a stage is a view into a larger
allocation whose margins (4 KB on each side) hold a sentinel byte; the
buffer itself is pre-filled with a second sentinel.  After the stage runs:
the margins are unchanged (no write landed outside a buffer), and the
outputs equal the oracle bit for bit (so every element the stage owns was
written: a leftover sentinel would differ).  Covers the four stages, the
one-launch dispatch, the INT8 combine, the token-level layout, the GMM1
epilogue and the whole deep MoE, on shapes with ragged tiles and tails, and
on the two-kernel notify path (R > 64)."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 4096            # bytes of margin on each side (keeps views 4 KB aligned)
OUTSIDE = 0xA5          # margin sentinel
INSIDE = 0x5A           # pre-fill of the buffer itself


@pytest.fixture(scope="module")
def ep():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    import combine_moe_dispatch_layout_gb300 as ep
    return ep


@pytest.fixture(scope="module")
def pl(ep):
    from combine_moe_dispatch_layout_gb300 import pipeline
    return pipeline


class Guarded:
    """Allocates views with sentinel margins and checks the margins later."""

    def __init__(self):
        self.full = []

    def __call__(self, shape, dtype, inside=INSIDE):
        shape = tuple(shape)
        n = int(np.prod(shape)) if shape else 1
        es = torch.empty((), dtype=dtype).element_size()
        g = GUARD // es
        full = torch.empty(n + 2 * g, dtype=dtype, device="cuda")
        full.view(torch.uint8).fill_(OUTSIDE)
        view = full[g:g + n]
        if inside is not None:
            view.view(torch.uint8).fill_(inside)
        self.full.append((full, g, n))
        return view.view(shape)

    def assert_margins(self):
        torch.cuda.synchronize()
        for i, (full, g, n) in enumerate(self.full):
            b = full.view(torch.uint8)
            es = full.element_size()
            lo, hi = b[:g * es], b[(g + n) * es:]
            assert bool((lo == OUTSIDE).all()) and bool((hi == OUTSIDE).all()), \
                "buffer %d: a write landed outside it" % i


def _guarded_buffers(pl, w, G):
    b = pl.PipelineBuffers(w.R, w.bs, w.k, w.epr, w.H, w.dtype, w.quant)
    E, T, P = w.E, w.T, w.P
    b.count = G((w.R, E), torch.int32)
    b.rank_send = G((w.R, w.R), torch.int32)
    b.send_idx = G((T, w.k), torch.int32)
    b.workspace = G(tuple(b.workspace.shape), torch.uint8, inside=0)
    b.put_offset = G((E * w.R,), torch.int32)
    b.total_recv = G((w.R,), torch.int32)
    b.rank_recv_base = G((w.R + 1,), torch.int64)
    b.recv_per_expert = G((E,), torch.int32)
    b.max_bs = G((1,), torch.int32)
    b.dev_status = G((1,), torch.int32, inside=0)
    b.recv = G((P, b.row_bytes), torch.uint8)
    b.out = G((T, w.H), b.torch_dtype)
    b._fused_ws = G((max(16, pl.fused_workspace_bytes(b.shape)),), torch.uint8, inside=0)
    return b


def _eq(name, got, want):
    g = got.detach().cpu().numpy().reshape(want.shape)
    assert np.array_equal(g, want), name


def _check(oracle, b, w, idx, x, wt, y, full_pipeline=True):
    L = oracle.layout(idx.numpy(), w.R, w.epr)
    N = oracle.notify(L["count"], w.R, w.bs, w.epr)
    assert b.status() == 0
    _eq("count", b.count, L["count"])
    _eq("rank_send", b.rank_send, L["rank_send"])
    _eq("send_idx", b.send_idx, L["send_idx"])
    _eq("put_offset", b.put_offset, N["put_offset"])
    _eq("total_recv", b.total_recv, N["total_recv"])
    _eq("rank_recv_base", b.rank_recv_base, N["rank_recv_base"])
    _eq("recv_per_expert", b.recv_per_expert, N["recv_per_expert"])
    assert int(b.max_bs.item()) == N["max_bs"]
    recv, st = oracle.dispatch(W.bits(x), idx.numpy(), L["send_idx"], N["put_offset"],
                               N["rank_recv_base"], w.R, w.epr, w.dtype, w.quant)
    assert st == 0
    _eq("recv", b.recv, recv)
    if full_pipeline:
        out, st = oracle.combine(W.bits(y), idx.numpy(), wt.numpy(), L["send_idx"],
                                 N["put_offset"], N["rank_recv_base"], w.R, w.epr, w.dtype)
        assert st == 0
        got = b.out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got.reshape(out.shape), out), "out"
    return L, N


CASES = [
    W.Workload("g_ragged", R=3, epr=5, bs=1500, k=7, H=1000, seed=71),
    W.Workload("g_verbatim", R=4, epr=6, bs=1111, k=5, H=520, quant=False, seed=72),
    W.Workload("g_fp16", R=5, epr=3, bs=600, k=4, H=136, dtype=W.FP16, seed=73),
    W.Workload("g_r384", R=384, epr=2, bs=4, k=8, H=64, seed=74),        # two-kernel notify
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_pipeline_stays_inside_its_buffers(oracle_mod, pl, w):
    G = Guarded()
    b = _guarded_buffers(pl, w, G)
    idx, wt = W.routing(w)
    x, y = W.tokens(w), W.expert_outputs(w)
    xd, yd = G(tuple(x.shape), x.dtype), G(tuple(y.shape), y.dtype)
    xd.copy_(x.cuda())
    yd.copy_(y.cuda())
    idxd, wtd = G(tuple(idx.shape), torch.int32), G(tuple(wt.shape), torch.float32)
    idxd.copy_(idx.cuda())
    wtd.copy_(wt.cuda())
    pl.run_pipeline(b, xd, idxd, wtd, yd)
    G.assert_margins()
    _check(oracle_mod, b, w, idx, x, wt, y)
    # the one-launch dispatch on fresh (sentinel-filled) outputs
    G2 = Guarded()
    b2 = _guarded_buffers(pl, w, G2)
    pl.run_dispatch_fused(b2, xd, idxd)
    G2.assert_margins()
    _check(oracle_mod, b2, w, idx, x, wt, y, full_pipeline=False)


@pytest.mark.parametrize("w", CASES[:1] + CASES[2:3], ids=lambda w: w.name)
def test_int8_combine_and_token_layout_stay_inside(oracle_mod, ep, pl, w):
    G = Guarded()
    b = _guarded_buffers(pl, w, G)
    idx, wt = W.routing(w)
    yq = W.expert_outputs_int8(w)
    yqd = G(tuple(yq.shape), torch.uint8)
    yqd.copy_(yq.cuda())
    idxd = idx.cuda()
    pl.run_layout_notify(b, idxd)
    pl.run_combine_quant(b, yqd, idxd, wt.cuda())
    tpr = G((w.R, w.R), torch.int32)
    inr = G((w.T, w.R), torch.uint8)
    st = G((1,), torch.int32, inside=0)
    ep.moe_token_layout(b.shape, idxd, tpr, inr, st)
    G.assert_margins()
    assert b.status() == 0 and int(st.item()) == 0
    L = oracle_mod.layout(idx.numpy(), w.R, w.epr)
    N = oracle_mod.notify(L["count"], w.R, w.bs, w.epr)
    ref, s = oracle_mod.combine_quant(yq.numpy(), idx.numpy(), wt.numpy(), L["send_idx"],
                                      N["put_offset"], N["rank_recv_base"], w.R, w.epr,
                                      w.dtype, w.H)
    assert s == 0
    got = b.out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got.reshape(ref.shape), ref), "INT8 combine"
    tl = oracle_mod.token_layout(idx.numpy(), w.R, w.epr)
    _eq("tokens_per_rank", tpr, tl["tokens_per_rank"])
    _eq("in_rank", inr, tl["in_rank"])


@pytest.mark.parametrize("M,I", [(300, 2048), (77, 4104), (5, 40)])
def test_gmm1_epilogue_stays_inside(oracle_mod, ep, M, I):
    acc_h, ws_h, ts_h = W.gmm1_accumulators(M, I)
    G = Guarded()
    acc, ws, ts = G(tuple(acc_h.shape), torch.int32), G(tuple(ws_h.shape), torch.float32), \
        G(tuple(ts_h.shape), torch.float32)
    acc.copy_(acc_h.cuda())
    ws.copy_(ws_h.cuda())
    ts.copy_(ts_h.cuda())
    row_bytes = (I + 31) // 32 * 32 + 32
    out = G((M, row_bytes), torch.uint8)
    st = G((1,), torch.int32, inside=0)
    ep.moe_swiglu_quant(acc, ws, ts, out, st)
    G.assert_margins()
    assert int(st.item()) == 0
    ref = oracle_mod.swiglu_quant(acc_h.numpy(), ws_h.numpy(), ts_h.numpy())
    ref = ref[0] if isinstance(ref, tuple) else ref
    assert np.array_equal(out.cpu().numpy().reshape(ref.shape), ref), "GMM1 epilogue"


@pytest.mark.parametrize("fused", [False, True], ids=["int32_gmm1", "swiglu_in_gmm1"])
def test_deep_moe_stays_inside_its_buffers(oracle_mod, pl, fused):
    """The fused deep MoE (dispatch_expand, group offsets, the grouped GEMMs
    with their int32 / SwiGLU / dequantising epilogues, the requantisation
    and the fp32 combine) on a ragged Zipf-routed shape, every intermediate
    in a guarded view."""
    w = W.Workload("g_deep", R=3, epr=3, bs=70, H=1096, k=3, routing="zipf",
                   weights="sigmoid", x_scale=2.0, seed=75)
    I = 264
    idx, wt = W.routing(w)
    x = W.tokens(w)
    w1, ws1, w2, ws2 = W.moe_weights(w.E, w.H, I, seed=7)
    ref = oracle_mod.deep_moe(W.bits(x), idx.numpy(), wt.numpy(), w.R, w.epr, w.dtype,
                              w1.numpy(), ws1.numpy(), w2.numpy(), ws2.numpy())
    G = Guarded()
    b = pl.DeepMoeBuffers(w.R, w.bs, w.k, w.epr, w.H, I, w.dtype)
    base = _guarded_buffers(pl, w.with_(quant=True), G)
    for name in ("count", "rank_send", "send_idx", "workspace", "put_offset", "total_recv",
                 "rank_recv_base", "recv_per_expert", "max_bs", "dev_status", "out"):
        setattr(b, name, getattr(base, name))
    P = w.P
    b.group_off = G((w.E + 1,), torch.int64)
    b.a1 = G((P, w.H), torch.bfloat16)
    b.ts1 = G((P,), torch.float32)
    b.acc1 = G((P, 2 * I), torch.int32)
    b.h = G((P, I), torch.float32)
    b.a2 = G((P, I), torch.bfloat16)
    b.ts2 = G((P,), torch.float32)
    b.y2 = G((P, w.H), torch.float32)
    dev = torch.device("cuda")
    wts = pl.DeepMoeWeights(w1.to(dev), ws1.to(dev), w2.to(dev), ws2.to(dev))
    idx_d, wt_d, x_d = idx.to(dev), wt.to(dev), x.to(dev)
    pl.run_layout_notify(b, idx_d)
    pl.run_dispatch_expand(b, x_d, idx_d)
    pl.run_deep_moe_experts(b, wts, fused_swiglu=fused)
    pl.run_deep_combine(b, idx_d, wt_d)
    G.assert_margins()
    assert b.status() == 0
    got = b.out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got.reshape(ref["out"].shape), ref["out"]), "deep MoE out"
