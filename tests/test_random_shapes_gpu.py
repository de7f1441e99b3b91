"""Randomised shapes: 120 seeded random problems (ranks, experts per rank,
tokens per rank including 0, top-k, hidden size down to 8, both token
dtypes, INT8 or verbatim rows, uniform or Zipf routing) through the four
stages, the one-launch dispatch and, for INT8 rows, the INT8 combine, each
compared with the oracle bit for bit; then random GMM1-epilogue shapes and
random grouped GEMMs and random small deep MoE problems, also bit-exact.  The fixed cases elsewhere pin the
known edges; this sweep crosses the kernels' internal size decisions (tile
geometry, parts per token, one-CTA or cooperative one-launch form, chunks
per thread) at combinations nobody chose by hand."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _shapes(n, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < n:
        R = int(rng.choice([1, 2, 3, 5, 8, 13, 24, 40, 70]))
        epr = int(rng.integers(1, 9))
        E = R * epr
        if E > 4096:
            continue
        bs = int(rng.choice([0, 1, 7, 33, 64, 129, 300, 517],
                            p=[0.04, 0.12, 0.14, 0.14, 0.14, 0.14, 0.14, 0.14]))
        k = int(rng.integers(1, min(E, 12) + 1))
        H = int(8 * rng.integers(1, 151))
        dtype = W.BF16 if rng.random() < 0.6 else W.FP16
        quant = bool(rng.random() < 0.7)
        routing = "zipf" if (rng.random() < 0.25 and k < E) else "uniform"
        out.append(W.Workload("rand%d" % len(out), R=R, epr=epr, bs=bs, H=H, k=k,
                              dtype=dtype, quant=quant, routing=routing,
                              seed=3000 + len(out)))
    return out


SHAPES = _shapes(120)


@pytest.fixture(scope="module")
def pl():
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    from combine_moe_dispatch_layout_gb300 import pipeline
    return pipeline


def _u16(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("w", SHAPES, ids=lambda w: "R%d-epr%d-bs%d-k%d-H%d-%s-%s%s" % (
    w.R, w.epr, w.bs, w.k, w.H, "fp16" if w.dtype == W.FP16 else "bf16",
    "q" if w.quant else "v", "-zipf" if w.routing == "zipf" else ""))
def test_random_shape(oracle_mod, pl, w):
    idx, wt = W.routing(w)
    x, y = W.tokens(w), W.expert_outputs(w)
    L = oracle_mod.layout(idx.numpy(), w.R, w.epr)
    N = oracle_mod.notify(L["count"], w.R, w.bs, w.epr)
    recv, st = oracle_mod.dispatch(W.bits(x), idx.numpy(), L["send_idx"], N["put_offset"],
                                   N["rank_recv_base"], w.R, w.epr, w.dtype, w.quant)
    out, st2 = oracle_mod.combine(W.bits(y), idx.numpy(), wt.numpy(), L["send_idx"],
                                  N["put_offset"], N["rank_recv_base"], w.R, w.epr, w.dtype)
    assert st == 0 and st2 == 0
    dev = torch.device("cuda")
    idx_d, wt_d, x_d, y_d = idx.to(dev), wt.to(dev), x.to(dev), y.to(dev)

    def check(b, with_out):
        assert b.status() == 0
        np.testing.assert_array_equal(b.count.cpu().numpy(), L["count"])
        np.testing.assert_array_equal(b.rank_send.cpu().numpy(), L["rank_send"])
        np.testing.assert_array_equal(b.send_idx.cpu().numpy(), L["send_idx"])
        np.testing.assert_array_equal(b.put_offset.cpu().numpy(), N["put_offset"])
        np.testing.assert_array_equal(b.rank_recv_base.cpu().numpy(), N["rank_recv_base"])
        np.testing.assert_array_equal(b.recv_per_expert.cpu().numpy(), N["recv_per_expert"])
        np.testing.assert_array_equal(b.recv.cpu().numpy(), recv)
        if with_out:
            np.testing.assert_array_equal(_u16(b.out).reshape(out.shape), out)

    b = pl.PipelineBuffers(w.R, w.bs, w.k, w.epr, w.H, w.dtype, w.quant)
    b.recv.fill_(0xCD)
    pl.run_pipeline(b, x_d, idx_d, wt_d, y_d)
    torch.cuda.synchronize()
    check(b, True)

    b2 = pl.PipelineBuffers(w.R, w.bs, w.k, w.epr, w.H, w.dtype, w.quant)
    b2.recv.fill_(0xCD)
    pl.run_dispatch_fused(b2, x_d, idx_d)
    torch.cuda.synchronize()
    check(b2, False)

    if w.quant and w.T > 0:
        yq = W.expert_outputs_int8(w)
        ref, s = oracle_mod.combine_quant(yq.numpy(), idx.numpy(), wt.numpy(), L["send_idx"],
                                          N["put_offset"], N["rank_recv_base"], w.R, w.epr,
                                          w.dtype, w.H)
        assert s == 0
        pl.run_combine_quant(b, yq.to(dev), idx_d, wt_d)
        torch.cuda.synchronize()
        assert b.status() == 0
        np.testing.assert_array_equal(_u16(b.out).reshape(ref.shape), ref)


# ---- the GMM1 epilogue and the grouped GEMM over random shapes ----------------

def _epilogue_shapes(n, seed=2025):
    rng = np.random.default_rng(seed)
    return [(int(rng.choice([1, 2, 17, 64, 300, 1000])),
             int(8 * rng.choice([1, 3, 5, 32, 100, 255, 256, 257, 512, 513, 700, 1024]))
             ) for _ in range(n)]


@pytest.fixture(scope="module")
def ep(pl):
    import combine_moe_dispatch_layout_gb300 as ep
    return ep


@pytest.mark.parametrize("M,I", _epilogue_shapes(30), ids=lambda v: str(v))
def test_random_gmm1_epilogue(oracle_mod, ep, M, I):
    """Row widths from 8 to 8192 outputs: the warp form (I <= 4096) and the
    CTA form (larger I), bit-exact against the oracle's exp reading."""
    acc, ws, ts = W.gmm1_accumulators(M, I, seed=M * 7 + I)
    rb = (I + 31) // 32 * 32 + 32
    out = torch.full((M, rb), 0xAB, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ep.moe_swiglu_quant(acc.cuda(), ws.cuda(), ts.cuda(), out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle_mod.swiglu_quant(acc.numpy(), ws.numpy(), ts.numpy())
    np.testing.assert_array_equal(out.cpu().numpy(), ref)


def _gemm_shapes(n, seed=2026):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        G = int(rng.choice([1, 2, 3, 7, 16, 40]))
        sizes = tuple(int(v) for v in rng.choice([0, 1, 5, 63, 128, 129, 200, 333], G))
        if sum(sizes) == 0:
            sizes = (1,) + sizes[1:]
        N = int(8 * rng.choice([1, 2, 17, 32, 33, 64, 96]))
        K = int(8 * rng.choice([1, 8, 9, 127, 128, 129, 260]))
        out.append((G, N, K, sizes))
    return out


@pytest.mark.parametrize("case", _gemm_shapes(20), ids=lambda c: "G%d_N%d_K%d" % c[:3])
def test_random_grouped_gemm(oracle_mod, ep, case):
    """Exact int32 sums for random group sizes (empty groups included),
    output widths down to 8 and K from 8 to 2080 (one to three 1024-wide
    exact chunks, ragged K blocks)."""
    G, N, K, sizes = case
    rng = np.random.default_rng(sum(sizes) * 31 + N + K)
    M = sum(sizes)
    a = rng.integers(-128, 128, (M, K)).astype(np.int8)
    w = rng.integers(-128, 128, (G, N, K)).astype(np.int8)
    dev = torch.device("cuda")
    a_bf = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    w_bf = torch.empty((G, N, K), dtype=torch.bfloat16, device=dev)
    ep.moe_codes_to_bf16(torch.from_numpy(a.view(np.uint8)).to(dev), M, K, K, a_bf)
    ep.moe_codes_to_bf16(torch.from_numpy(w.view(np.uint8)).to(dev), G * N, K, K, w_bf)
    gr = torch.tensor(sizes, dtype=torch.int32, device=dev)
    c = torch.full((M, N), -7, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ep.moe_grouped_gemm_i8(a_bf, w_bf, gr, c, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    np.testing.assert_array_equal(c.cpu().numpy(), oracle_mod.grouped_gemm(a.view(np.uint8),
                                                                           off, w))


def _deep_shapes(n, seed=2027):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        R = int(rng.choice([1, 2, 3, 5]))
        epr = int(rng.integers(1, 5))
        k = int(rng.integers(1, min(R * epr, 4) + 1))
        bs = int(rng.choice([1, 9, 40, 77]))
        H = int(8 * rng.choice([16, 33, 64, 130]))
        I = int(8 * rng.choice([2, 8, 33, 64]))
        dtype = W.BF16 if rng.random() < 0.6 else W.FP16
        out.append((W.Workload("rdeep%d" % i, R=R, epr=epr, bs=bs, H=H, k=k, dtype=dtype,
                               x_dist="uniform" if dtype == W.FP16 else "normal",
                               seed=5000 + i), I))
    return out


@pytest.mark.parametrize("w,I", _deep_shapes(8), ids=lambda v: getattr(v, "name", str(v)))
def test_random_deep_moe(oracle_mod, pl, w, I):
    """The fused deep MoE (both GMM1 routes) on random small shapes, bit-exact."""
    idx, wt = W.routing(w)
    x = W.tokens(w)
    w1, ws1, w2, ws2 = W.moe_weights(w.E, w.H, I, seed=w.seed)
    ref = oracle_mod.deep_moe(W.bits(x), idx.numpy(), wt.numpy(), w.R, w.epr, w.dtype,
                              w1.numpy(), ws1.numpy(), w2.numpy(), ws2.numpy())
    dev = torch.device("cuda")
    wts = pl.DeepMoeWeights(w1.to(dev), ws1.to(dev), w2.to(dev), ws2.to(dev))
    for fused in (False, True):
        b = pl.DeepMoeBuffers(w.R, w.bs, w.k, w.epr, w.H, I, w.dtype)
        idx_d, wt_d, x_d = idx.to(dev), wt.to(dev), x.to(dev)
        pl.run_layout_notify(b, idx_d)
        pl.run_dispatch_expand(b, x_d, idx_d)
        pl.run_deep_moe_experts(b, wts, fused_swiglu=fused)
        pl.run_deep_combine(b, idx_d, wt_d)
        torch.cuda.synchronize()
        assert b.status() == 0
        np.testing.assert_array_equal(_u16(b.out).reshape(ref["out"].shape), ref["out"])
