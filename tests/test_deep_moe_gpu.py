"""GPU parity of the fused deep MoE path (grouped INT8 GEMM on the tensor
cores, per-expert GMM1 epilogue, DeqCombine, and the whole pipeline) against
the CPU oracle, through the C ABI.  Integer results (the GEMMs' int32
accumulators, INT8 row images) and the bf16 outputs are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


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


def _eq(name, got, want):
    g = got.detach().cpu().numpy() if isinstance(got, torch.Tensor) else got
    g = g.reshape(want.shape)
    if not np.array_equal(g, want):
        bad = np.argwhere(g != want)
        raise AssertionError("%s: %d mismatches, first at %s: got %s want %s"
                             % (name, len(bad), bad[0].tolist(), g[tuple(bad[0])],
                                want[tuple(bad[0])]))


def _gemm_gpu(ep, a_i8, w_i8, sizes, a_rows=None, fill=-7):
    """Runs codes_to_bf16 + grouped GEMM; returns (c int32 numpy, status)."""
    dev = torch.device("cuda")
    M, K = a_i8.shape
    G, N, _ = w_i8.shape
    rows = M if a_rows is None else a_rows
    a_d = torch.from_numpy(a_i8.view(np.uint8)).to(dev)
    w_d = torch.from_numpy(w_i8.view(np.uint8)).to(dev)
    a_bf = torch.empty((rows, K), dtype=torch.bfloat16, device=dev)
    a_bf.zero_()
    w_bf = torch.empty((G, N, K), dtype=torch.bfloat16, device=dev)
    ep.moe_codes_to_bf16(a_d, M, K, K, a_bf)
    ep.moe_codes_to_bf16(w_d, G * N, K, K, w_bf)
    gr = torch.tensor(sizes, dtype=torch.int32, device=dev)
    c = torch.full((rows, N), fill, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ep.moe_grouped_gemm_i8(a_bf, w_bf, gr, c, st)
    torch.cuda.synchronize()
    return c.cpu().numpy(), int(st.item())


GEMM_CASES = [
    # (G, N, K, group sizes): ragged row tiles, empty groups, one K block,
    # a ragged K block, several exact 1024-wide chunks
    (3, 128, 64, (5, 0, 130)),
    (4, 256, 200, (128, 1, 0, 257)),
    (2, 128, 1096, (300, 45)),
    (5, 384, 2056, (64, 129, 0, 200, 3)),
    (3, 136, 520, (70, 0, 200)),          # a ragged last column tile
    (2, 8, 32, (3, 140)),                 # N and K below one tile
    (3000, 136, 72, tuple((7 * i) % 5 for i in range(3000))),   # many groups: 3 stages
    # large groups: odd row-tile counts, ragged tails, an empty group, a
    # partial third K chunk
    (7, 136, 2112, (700, 1030, 128, 513, 900, 0, 2049)),
    (2, 512, 1024, (1, 1100)),
    (1, 256, 64, (640,)),
]


@pytest.mark.parametrize("case", GEMM_CASES, ids=lambda c: "G%d_N%d_K%d" % c[:3])
def test_grouped_gemm_exact(oracle_mod, ep, case):
    G, N, K, sizes = case
    rng = np.random.default_rng(sum(sizes) + K)
    M = sum(sizes)
    a = rng.integers(-127, 128, (M, K)).astype(np.int8)
    w = rng.integers(-127, 128, (G, N, K)).astype(np.int8)
    c, st = _gemm_gpu(ep, a, w, sizes)
    assert st == 0
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    _eq("c", c, oracle_mod.grouped_gemm(a.view(np.uint8), off, w))


def test_grouped_gemm_extreme_sums(oracle_mod, ep):
    """Codes of one sign make every 1024-wide chunk sum reach 1024*127*127
    (just under 2^24), and the whole row 7168*127*127; alternating rows
    flip the sign; a row of -128 codes reaches exactly 2^24 per chunk."""
    K, N = 7168, 128
    a = np.full((6, K), 127, np.int8)
    a[1] = -127
    a[2, ::2] = -127
    a[3] = -128
    a[4] = np.arange(K) % 255 - 127
    a[5] = 1
    w = np.full((1, N, K), 127, np.int8)
    w[0, 1::2] = -128
    c, st = _gemm_gpu(ep, a, w, (6,))
    assert st == 0
    want = oracle_mod.grouped_gemm(a.view(np.uint8), np.array([0, 6], np.int64), w)
    _eq("c", c, want)
    assert want[0, 0] == 127 * 127 * K and want[3, 1] == 128 * 128 * K


def test_grouped_gemm_rows_beyond_groups_untouched_and_capacity(ep):
    rng = np.random.default_rng(5)
    K, N = 64, 128
    a = rng.integers(-127, 128, (40, K)).astype(np.int8)
    w = rng.integers(-127, 128, (2, N, K)).astype(np.int8)
    c, st = _gemm_gpu(ep, a, w, (10, 20), fill=-7)       # 30 of 40 rows used
    assert st == 0 and (c[30:] == -7).all()
    c, st = _gemm_gpu(ep, a, w, (30, 20), fill=-7)       # 50 rows > 40
    assert st == ep.MOE_ERR_CAPACITY and (c == -7).all()


def test_grouped_gemm_rejects_bad_shapes(ep):
    dev = torch.device("cuda")
    a = torch.zeros((16, 64), dtype=torch.bfloat16, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    gr = torch.tensor([16], dtype=torch.int32, device=dev)
    for N, K in ((100, 64), (128, 60)):   # N % 8, K % 8
        w = torch.zeros((1, N, K), dtype=torch.bfloat16, device=dev)
        aa = torch.zeros((16, K), dtype=torch.bfloat16, device=dev)
        c = torch.zeros((16, N), dtype=torch.int32, device=dev)
        with pytest.raises(ep.MoeError):
            ep.moe_grouped_gemm_i8(aa, w, gr, c, st)
    del a


def _dequant_bits(oracle, ref, ws2, I):
    """GMM2's dequantised rows, (fp32(acc2) * ws2[e]) * 1/scale of the
    requantised row, as int32 bit patterns (numpy float32: one rounding per
    product)."""
    grp = np.searchsorted(ref["group_off"], ref["rows"], side="right") - 1
    ts = oracle.row_inv_scale(ref["x2"], I)
    y = (ref["acc2"].astype(np.float32) * ws2[grp]) * ts[:, None]
    return y.astype(np.float32).view(np.int32)


@pytest.mark.parametrize("case", [(3, 264, 200, (130, 0, 70)),
                                  (3, 264, 1104, (600, 0, 1000))],   # two K chunks
                         ids=lambda c: "G%d_N%d_K%d" % c[:3])
def test_grouped_gemm_dequant_epilogue(oracle_mod, ep, case):
    rng = np.random.default_rng(9)
    G, N, K, sizes = case
    M = sum(sizes)
    dev = torch.device("cuda")
    a = rng.integers(-127, 128, (M, K)).astype(np.int8)
    w = rng.integers(-127, 128, (G, N, K)).astype(np.int8)
    cs = rng.uniform(0.5, 1.5, (G, N)).astype(np.float32) * 1e-3
    rs_rows = np.zeros((M, 48), np.uint8)                   # scale at byte 20 of 48-byte rows
    rs = rng.uniform(0.01, 0.1, M).astype(np.float32)
    rs_rows[:, 20:24] = rs.view(np.uint8).reshape(M, 4)
    a_bf = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    w_bf = torch.empty((G, N, K), dtype=torch.bfloat16, device=dev)
    ep.moe_codes_to_bf16(torch.from_numpy(a.view(np.uint8)).to(dev), M, K, K, a_bf)
    ep.moe_codes_to_bf16(torch.from_numpy(w.view(np.uint8)).to(dev), G * N, K, K, w_bf)
    y = torch.full((M, N), -1.0, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ep.moe_grouped_gemm_i8_dequant(a_bf, w_bf, torch.tensor(sizes, dtype=torch.int32, device=dev),
                                   torch.from_numpy(cs).to(dev),
                                   (torch.from_numpy(rs_rows).to(dev), 20, 48), y, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    c = oracle_mod.grouped_gemm(a.view(np.uint8), off, w)
    grp = np.searchsorted(off, np.arange(M), side="right") - 1
    want = ((c.astype(np.float32) * cs[grp]) * rs[:, None]).astype(np.float32)
    _eq("y", y.view(torch.int32), want.view(np.int32))


def _deep_inputs(w, I, seed, device="cpu"):
    idx, wt = W.routing(w)
    x = W.tokens(w)
    w1, ws1, w2, ws2 = W.moe_weights(w.E, w.H, I, seed=seed, device=device)
    return idx, wt, x, (w1, ws1, w2, ws2)


DEEP_CASES = [
    W.Workload("deep_small", R=2, epr=4, bs=96, H=256, k=4, seed=21),
    W.Workload("deep_fp16", R=2, epr=3, bs=50, H=264, k=2, dtype=W.FP16, x_dist="uniform",
               x_scale=4.0, seed=23),
    W.Workload("deep_ragged", R=3, epr=3, bs=70, H=1096, k=3, routing="zipf",
               weights="sigmoid", x_scale=2.0, seed=22),
]


def _swiglu_bits(oracle, acc1, group_off, rows, ws1, ts, I):
    """h of the GMM1 epilogue as int32 bit patterns, restated with numpy
    float32 operations (one rounding each) and the oracle's exp."""
    grp = np.searchsorted(group_off, rows, side="right") - 1
    v = (acc1.astype(np.float32) * ws1[grp]) * ts[:, None].astype(np.float32)
    gate, up = v[:, :I], v[:, I:]
    e = oracle.exp_f32(-gate)
    h = (gate / (e + np.float32(1.0))) * up
    return h.astype(np.float32).view(np.int32)


def _codes_bf16(images, K):
    """bf16 bit patterns of the INT8 codes of row images (exact)."""
    q = images[:, :K].view(np.int8).astype(np.float32)
    return (q.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("w", DEEP_CASES, ids=lambda w: w.name)
def test_deep_moe_pipeline(oracle_mod, ep, pl, w):
    I = 136 if w.H > 512 else 128
    idx, wt, x, (w1, ws1, w2, ws2) = _deep_inputs(w, I, w.seed)
    ref = oracle_mod.deep_moe(W.bits(x), idx.numpy(), wt.numpy(), w.R, w.epr, w.dtype,
                              w1.numpy(), ws1.numpy(), w2.numpy(), ws2.numpy())
    dev = torch.device("cuda")
    b = pl.DeepMoeBuffers(w.R, w.bs, w.k, w.epr, w.H, I, w.dtype)
    wts = pl.DeepMoeWeights(w1.to(dev), ws1.to(dev), w2.to(dev), ws2.to(dev))
    idx_d, wt_d, x_d = idx.to(dev), wt.to(dev), x.to(dev)
    pl.run_layout_notify(b, idx_d)
    pl.run_dispatch_expand(b, x_d, idx_d)
    assert b.status() == 0, "dispatch"
    L = oracle_mod.layout(idx.numpy(), w.R, w.epr)
    N = oracle_mod.notify(L["count"], w.R, w.bs, w.epr)
    recv, _ = oracle_mod.dispatch(W.bits(x), idx.numpy(), L["send_idx"], N["put_offset"],
                                  N["rank_recv_base"], w.R, w.epr, w.dtype, True)
    _eq("expand_x", b.a1.view(torch.int16).cpu().numpy().view(np.uint16),
        _codes_bf16(recv, w.H))
    _eq("dynamic_scale", b.ts1.view(torch.int32), oracle_mod.row_inv_scale(recv, w.H).view(np.int32))
    for fused in (True, False):      # SwiGLU in GMM1's epilogue, or the standalone kernel
        for t in (b.a2, b.ts2, b.y2, b.out):
            t.zero_()
        pl.run_deep_moe_experts(b, wts, fused_swiglu=fused)
        assert b.status() == 0, "experts"
        pl.run_deep_combine(b, idx_d, wt_d)
        assert b.status() == 0, "combine"
        tag = "(fused)" if fused else "(int32 + epilogue kernel)"
        _eq("group_off", b.group_off, ref["group_off"])
        if fused:
            _eq("h" + tag, b.h.view(torch.int32),
                _swiglu_bits(oracle_mod, ref["acc1"], ref["group_off"], ref["rows"],
                             ws1.numpy(), oracle_mod.row_inv_scale(recv, w.H), I))
        else:
            _eq("acc1" + tag, b.acc1, ref["acc1"])
        _eq("a2 codes" + tag, b.a2.view(torch.int16).cpu().numpy().view(np.uint16),
            _codes_bf16(ref["x2"], I))
        _eq("a2 1/scale" + tag, b.ts2.view(torch.int32),
            oracle_mod.row_inv_scale(ref["x2"], I).view(np.int32))
        _eq("y2" + tag, b.y2.view(torch.int32), _dequant_bits(oracle_mod, ref, ws2.numpy(), I))
        _eq("out" + tag, b.out.view(torch.int16).cpu().numpy().view(np.uint16), ref["out"])

    # the INT8-row-image route gives the same intermediates and output
    pl.run_dispatch(b, x_d, idx_d)                                 # b.recv: INT8 rows
    _eq("recv", b.recv, recv)
    a1 = torch.empty_like(b.a1)
    ep.moe_codes_to_bf16(b.recv, b.capacity, b.row_bytes, w.H, a1)
    _eq("codes_to_bf16(recv)", a1.view(torch.int16), b.a1.view(torch.int16).cpu().numpy())
    row2 = (I + 31) // 32 * 32 + 32
    x2 = torch.zeros((b.capacity, row2), dtype=torch.uint8, device=dev)
    ep.moe_swiglu_quant_grouped(b.acc1, wts.ws1, b.group_off,
                                (b.recv, (w.H + 31) // 32 * 32, b.row_bytes), x2, b.dev_status)
    _eq("x2 images", x2, ref["x2"])
    acc2 = torch.empty((b.capacity, w.H), dtype=torch.int32, device=dev)
    ep.moe_grouped_gemm_i8(b.a2, wts.w2, b.recv_per_expert, acc2, b.dev_status)
    _eq("acc2", acc2, ref["acc2"])
    b.out.zero_()
    ep.moe_deq_combine(b.shape, acc2, wts.ws2, (x2, (I + 31) // 32 * 32, row2), idx_d, wt_d,
                       b.send_idx, b.put_offset, b.rank_recv_base, b.out, b.dev_status)
    assert b.status() == 0
    _eq("out(int32 DeqCombine)", b.out.view(torch.int16).cpu().numpy().view(np.uint16),
        ref["out"])


@pytest.mark.parametrize("w", DEEP_CASES, ids=lambda w: w.name)
def test_deep_moe_swiglu_vs_plain_exp(oracle_mod, pl, w):
    """Both GMM1 epilogue routes (SwiGLU in the GEMM's epilogue + the
    requantisation pass, and the int32 GEMM + the grouped epilogue kernel)
    against the oracle whose Exp is the float nearest to e^x, within the
    bound that one exp ulp allows."""
    from conftest import assert_near_plain_exp
    I = 136 if w.H > 512 else 128
    idx, wt, x, (w1, ws1, w2, ws2) = _deep_inputs(w, I, w.seed)
    ref = oracle_mod.deep_moe(W.bits(x), idx.numpy(), wt.numpy(), w.R, w.epr, w.dtype,
                              w1.numpy(), ws1.numpy(), w2.numpy(), ws2.numpy())
    ts1 = oracle_mod.row_inv_scale(
        oracle_mod.dispatch(W.bits(x), idx.numpy(), *_layout_notify_args(oracle_mod, idx, w),
                            w.R, w.epr, w.dtype, True)[0], w.H)
    grp = np.searchsorted(ref["group_off"], ref["rows"], side="right") - 1
    x2 = np.zeros_like(ref["x2"])
    for e in np.unique(grp):
        sel = np.nonzero(grp == e)[0]
        x2[sel] = oracle_mod.swiglu_quant(ref["acc1"][sel], ws1.numpy()[e], ts1[sel],
                                          exp="libm")
    dev = torch.device("cuda")
    b = pl.DeepMoeBuffers(w.R, w.bs, w.k, w.epr, w.H, I, w.dtype)
    wts = pl.DeepMoeWeights(w1.to(dev), ws1.to(dev), w2.to(dev), ws2.to(dev))
    idx_d, x_d = idx.to(dev), x.to(dev)
    pl.run_layout_notify(b, idx_d)
    pl.run_dispatch_expand(b, x_d, idx_d)
    for fused in (True, False):
        b.a2.zero_()
        b.ts2.zero_()
        pl.run_deep_moe_experts(b, wts, fused_swiglu=fused)
        assert b.status() == 0
        n = ref["rows"].size
        codes = b.a2[:n].float().cpu().numpy().astype(np.int64)
        assert_near_plain_exp("a2 (%s)" % ("fused" if fused else "kernel"), codes,
                              b.ts2[:n].cpu().numpy(), x2, I)


def _layout_notify_args(oracle_mod, idx, w):
    L = oracle_mod.layout(idx.numpy(), w.R, w.epr)
    N = oracle_mod.notify(L["count"], w.R, w.bs, w.epr)
    return L["send_idx"], N["put_offset"], N["rank_recv_base"]


def test_deep_moe_dsv3_size_sampled(oracle_mod, pl):
    """DeepSeek-V3 shape (R = 8, E = 256, bs = 4096, k = 8, H = 7168,
    I = 2048), weights drawn on the device; sampled tokens are checked
    against the oracle run on their rows only (the needed experts' weights
    copied back)."""
    w = W.WORKLOADS["dsv3"]
    I = 2048
    dev = torch.device("cuda")
    idx, wt = W.routing(w)
    x = W.tokens(w)
    w1, ws1, w2, ws2 = W.moe_weights(w.E, w.H, I, seed=31, device=dev)
    b = pl.DeepMoeBuffers(w.R, w.bs, w.k, w.epr, w.H, I, w.dtype)
    wts = pl.DeepMoeWeights(w1, ws1, w2, ws2)
    pl.run_deep_moe(b, wts, x.to(dev), idx.to(dev), wt.to(dev))
    torch.cuda.synchronize()
    assert b.status() == 0
    toks = np.array([0, 12345, w.T - 1], np.int64)
    idx_n, wt_n = idx.numpy(), wt.numpy()
    L = oracle_mod.layout(idx_n, w.R, w.epr)
    N = oracle_mod.notify(L["count"], w.R, w.bs, w.epr)
    images, row_ids, st = oracle_mod.dispatch_tokens(
        W.bits(x), idx_n, L["send_idx"], N["put_offset"], N["rank_recv_base"], w.R,
        w.epr, w.dtype, True, toks)
    assert st == 0
    n = toks.size * w.k
    acc2 = np.zeros((n, w.H), np.int32)
    ws2_h = ws2.cpu().numpy()
    x2 = np.zeros((n, (I + 31) // 32 * 32 + 32), np.uint8)
    one = np.array([0, 1], np.int64)
    for i in range(n):
        t, kk = divmod(i, w.k)
        e = int(idx_n[toks[t], kk])
        img = images[t, kk][None]
        a1 = oracle_mod.grouped_gemm(img, one, w1[e].cpu().numpy()[None])
        _eq("acc1 row", b.acc1[int(row_ids[t, kk])], a1[0])
        ts = oracle_mod.row_inv_scale(img, w.H)
        x2[i] = oracle_mod.swiglu_quant(a1, ws1[e].cpu().numpy(), ts)[0]
        r = int(row_ids[t, kk])
        _eq("a2 row", b.a2[r].view(torch.int16).cpu().numpy().view(np.uint16),
            _codes_bf16(x2[i:i + 1], I)[0])
        _eq("ts2 row", b.ts2[r:r + 1].view(torch.int32),
            oracle_mod.row_inv_scale(x2[i:i + 1], I).view(np.int32))
        acc2[i] = oracle_mod.grouped_gemm(x2[i:i + 1], one, w2[e].cpu().numpy()[None])[0]
        y = (acc2[i].astype(np.float32) * ws2_h[e]) * oracle_mod.row_inv_scale(x2[i:i + 1], I)[0]
        _eq("y2 row", b.y2[int(row_ids[t, kk])].view(torch.int32),
            y.astype(np.float32).view(np.int32))
    out, st = oracle_mod.deq_combine(acc2, ws2.cpu().numpy(), oracle_mod.row_inv_scale(x2, I),
                                     idx_n, wt_n, L["send_idx"], N["put_offset"],
                                     N["rank_recv_base"], w.R, w.epr, w.dtype, tokens=toks)
    assert st == 0
    _eq("out rows", b.out[torch.from_numpy(toks).to(dev)].view(torch.int16).cpu().numpy()
        .view(np.uint16), out)


def test_deep_moe_graph_replay(oracle_mod, pl):
    """The deep MoE's calls enqueue only kernels on the caller's stream (tensor
    maps are encoded on the host into the launch), so the whole pipeline can
    be captured once and replayed on new inputs."""
    w = W.Workload("deep_graph", R=2, epr=4, bs=80, H=384, k=3, seed=41)
    I = 192
    dev = torch.device("cuda")
    _, _, _, (w1, ws1, w2, ws2) = _deep_inputs(w, I, w.seed)
    b = pl.DeepMoeBuffers(w.R, w.bs, w.k, w.epr, w.H, I, w.dtype)
    wts = pl.DeepMoeWeights(w1.to(dev), ws1.to(dev), w2.to(dev), ws2.to(dev))
    idx_d = torch.zeros((w.T, w.k), dtype=torch.int32, device=dev)
    idx_d[:, 1] = 1
    idx_d[:, 2] = 2
    wt_d = torch.zeros((w.T, w.k), dtype=torch.float32, device=dev)
    x_d = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pl.run_deep_moe(b, wts, x_d, idx_d, wt_d, s)      # warm-up outside the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pl.run_deep_moe(b, wts, x_d, idx_d, wt_d, s)
    for seed in (42, 43):
        ww = w.with_(seed=seed)
        idx, wt = W.routing(ww)
        x = W.tokens(ww)
        idx_d.copy_(idx)
        wt_d.copy_(wt)
        x_d.copy_(x)
        b.dev_status.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert b.status() == 0
        ref = oracle_mod.deep_moe(W.bits(x), idx.numpy(), wt.numpy(), w.R, w.epr, w.dtype,
                                  w1.numpy(), ws1.numpy(), w2.numpy(), ws2.numpy())
        _eq("out(graph)", b.out.view(torch.int16).cpu().numpy().view(np.uint16), ref["out"])


def test_deep_moe_empty_batch(pl):
    w = W.Workload("deep_empty", R=2, epr=2, bs=0, H=128, k=2)
    dev = torch.device("cuda")
    _, _, _, (w1, ws1, w2, ws2) = _deep_inputs(w, 64, 3)
    b = pl.DeepMoeBuffers(w.R, w.bs, w.k, w.epr, w.H, 64, w.dtype)
    wts = pl.DeepMoeWeights(w1.to(dev), ws1.to(dev), w2.to(dev), ws2.to(dev))
    e = torch.zeros((0, w.k), device=dev)
    pl.run_deep_moe(b, wts, torch.zeros((0, w.H), dtype=torch.bfloat16, device=dev),
                    e.to(torch.int32), e)
    torch.cuda.synchronize()
    assert b.status() == 0
    assert int(b.group_off[-1].item()) == 0
