"""Property tests of the oracle over random shapes (hypothesis): the layout,
notify and receive-row invariants, the quantisation bounds, the combine
(one-hot weights give the token back; general weights within the rounding
bound of the fp64 sum), the INT8 combine and DeqCombine where they reduce
exactly to the combine, verbatim dispatch and a short receive buffer, the
token-level layout against Python sets, the grouped GEMM against numpy int64
matmuls and the GMM1 epilogue against a float64 restatement, on shapes the
fixed-seed pins do not reach (empty batches and groups, one rank, k = E,
repeated experts in a token).  CPU only; skipped where hypothesis is not
installed."""
import numpy as np
import pytest
import torch

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings, strategies as st  # noqa: E402

import test_oracle_pins as P  # noqa: E402  (the pins' helpers and closed forms)

# derandomize: the same examples on every run (a wider random search with
# 1500 examples per test found no counterexample)
SETTINGS = dict(max_examples=80, deadline=None, derandomize=True,
                suppress_health_check=[HealthCheck.function_scoped_fixture])


@st.composite
def routings(draw):
    R = draw(st.integers(1, 6))
    epr = draw(st.integers(1, 5))
    E = R * epr
    bs = draw(st.integers(0, 30))
    distinct = draw(st.booleans())
    k = draw(st.integers(1, min(E, 8) if distinct else 8))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    rng = np.random.default_rng(seed)
    idx = P._random_routing(rng, R, epr, bs, k, distinct=distinct)
    return R, epr, bs, k, idx


@settings(**SETTINGS)
@given(case=routings())
def test_layout_notify_rows_any_shape(oracle_mod, case):
    """Counts sum to bs*k per source rank; each (rank, expert) numbers its pairs
    0, 1, 2, ... in (token, k) order; putOffset is the exclusive prefix over
    (local expert, source rank) per destination rank; the receive rows equal
    the closed-form order (expert, token, k) and are a bijection onto
    [0, T*k) that keeps every row inside its destination rank's partition."""
    R, epr, bs, k, idx = case
    E = R * epr
    L = oracle_mod.layout(idx, R, epr)
    assert L["status"] == 0
    cnt = L["count"].astype(np.int64)
    assert (cnt.sum(axis=1) == bs * k).all()
    np.testing.assert_array_equal(L["rank_send"],
                                  cnt.reshape(R, R, epr).sum(axis=2))
    for s in range(R):
        sub_idx = idx[s * bs:(s + 1) * bs].reshape(-1)
        sub_send = L["send_idx"][s * bs:(s + 1) * bs].reshape(-1)
        for e in range(E):
            np.testing.assert_array_equal(sub_send[sub_idx == e], np.arange(cnt[s, e]))
    N = oracle_mod.notify(L["count"], R, bs, epr)
    po = N["put_offset"].reshape(E, R).astype(np.int64)
    for r in range(R):
        walk = [(e, s) for e in range(r * epr, (r + 1) * epr) for s in range(R)]
        offs = np.array([po[e, s] for (e, s) in walk])
        vals = np.array([cnt[s, e] for (e, s) in walk])
        assert offs[0] == 0
        np.testing.assert_array_equal(offs[1:], offs[:-1] + vals[:-1])
        assert offs[-1] + vals[-1] == N["total_recv"][r]
    np.testing.assert_array_equal(N["recv_per_expert"], cnt.sum(axis=0))
    np.testing.assert_array_equal(
        N["rank_recv_base"], np.concatenate([[0], np.cumsum(N["total_recv"])]))
    rows = oracle_mod.dst_rows(idx, L["send_idx"], N["put_offset"],
                               N["rank_recv_base"], R, epr)
    np.testing.assert_array_equal(rows, P.rows_by_sort(idx))
    assert sorted(rows.reshape(-1).tolist()) == list(range(R * bs * k))
    base = N["rank_recv_base"]
    dst = idx // epr
    assert ((rows >= base[dst]) & (rows < base[dst + 1])).all()


@settings(**SETTINGS)
@given(H8=st.integers(1, 96), dtype=st.sampled_from([0, 1]),
       scale=st.sampled_from([1e-3, 0.5, 1.0, 8.0, 200.0]),
       zeros=st.floats(0.0, 1.0), seed=st.integers(0, 2 ** 31 - 1))
def test_quant_row_any_shape(oracle_mod, H8, dtype, scale, zeros, seed):
    """Codes in [-127, 127] reaching 127 on the largest element; pads zero;
    1/scale = (amax + 1e-12)/127 to fp32 rounding; each code is the exact
    round-half-even of x*127/(amax + 1e-12) away from rounding boundaries; the
    dequantised row is within amax/254 of x (fp32 slack only)."""
    H = 8 * H8
    rng = np.random.default_rng(seed)
    v = (rng.standard_normal(H) * scale).astype(np.float32)
    v[rng.random(H) < zeros * 0.5] = 0.0
    xb = P._bf16_bits(v) if dtype == 0 else P._f16_bits(v)
    x = (torch.from_numpy(xb.view(np.int16))
         .view(torch.bfloat16 if dtype == 0 else torch.float16)
         .to(torch.float64).numpy())
    img = oracle_mod.quant_row(xb, dtype)
    ha = (H + 31) // 32 * 32
    assert img.size == ha + 32
    q = img[:H].view(np.int8).astype(np.int64)
    inv = float(img[ha:ha + 4].view(np.float32)[0])
    assert not img[H:ha].any() and not img[ha + 4:].any()
    amax = np.abs(x).max()
    assert np.abs(q).max() <= 127
    if amax > 0:
        assert np.abs(q).max() == 127
    assert abs(inv / ((amax + 1e-12) / 127) - 1) < 1e-6
    qe, margin = P.exact_q(x, amax)
    ok = margin > 1e-4
    np.testing.assert_array_equal(q[ok], qe[ok])
    assert (np.abs(q * inv - x) <= (amax + 1e-12) / 254 * (1 + 2.0 ** -14)).all()


@settings(**SETTINGS)
@given(R=st.integers(1, 4), epr=st.integers(1, 4), bs=st.integers(1, 12),
       kfrac=st.floats(0.0, 1.0), H8=st.integers(1, 12), dtype=st.sampled_from([0, 1]),
       seed=st.integers(0, 10 ** 6))
def test_combine_any_shape(oracle_mod, R, epr, bs, kfrac, H8, dtype, seed):
    """Combine over the dispatched rows: all the weight on one k gives the token
    back exactly; general weights stay within the bf16/fp16 rounding of the
    fp64 sum plus k fp32 roundings."""
    E = R * epr
    k = 1 + int(kfrac * (min(E, 6) - 1))
    H = 8 * H8
    wl = P.W.Workload("prop", R=R, epr=epr, bs=bs, H=H, k=k, dtype=dtype, quant=False,
                      seed=seed)
    idx, wt = P.W.routing(wl)
    idx, wt = idx.numpy(), wt.numpy()
    x = P.W.tokens(wl)
    L = oracle_mod.layout(idx, R, epr)
    N = oracle_mod.notify(L["count"], R, bs, epr)
    recv, stt = oracle_mod.dispatch(P.W.bits(x), idx, L["send_idx"], N["put_offset"],
                                    N["rank_recv_base"], R, epr, dtype, 0)
    assert stt == 0
    y = recv.view(np.uint16)
    rng = np.random.default_rng(seed)
    w1 = np.zeros_like(wt)
    w1[np.arange(wl.T), rng.integers(0, k, size=wl.T)] = 1.0
    out, stt = oracle_mod.combine(y, idx, w1, L["send_idx"], N["put_offset"],
                                  N["rank_recv_base"], R, epr, dtype)
    assert stt == 0
    np.testing.assert_array_equal(oracle_mod.to_f32(out, dtype), x.float().numpy())
    out, stt = oracle_mod.combine(y, idx, wt, L["send_idx"], N["put_offset"],
                                  N["rank_recv_base"], R, epr, dtype)
    rows = oracle_mod.dst_rows(idx, L["send_idx"], N["put_offset"],
                               N["rank_recv_base"], R, epr)
    yf = oracle_mod.to_f32(y, dtype).astype(np.float64)
    terms = yf[rows] * wt[..., None].astype(np.float64)
    ref = terms.sum(axis=1)
    got = oracle_mod.to_f32(out, dtype).astype(np.float64)
    rel = 2.0 ** -8 if dtype == 0 else 2.0 ** -10
    tol = rel * np.abs(ref) + (k + 1) * 2.0 ** -23 * np.abs(terms).sum(axis=1) + 2.0 ** -24
    assert (np.abs(got - ref) <= tol).all()


@settings(**SETTINGS)
@given(R=st.integers(1, 4), epr=st.integers(1, 4), bs=st.integers(1, 10),
       kfrac=st.floats(0.0, 1.0), H8=st.integers(1, 16),
       inv_exp=st.integers(-12, 6), seed=st.integers(0, 10 ** 6))
def test_combine_quant_exact_scales_any_shape(oracle_mod, R, epr, bs, kfrac, H8, inv_exp,
                                              seed):
    """With 1/scale an exact power of two the dequantised value q * 1/scale is
    exact, so the INT8 combine equals the combine of those values as bf16 rows
    (exact in bf16: |q| <= 127 has 7 significant bits), bit for bit; H % 32 != 0
    also checks where 1/scale is read."""
    E = R * epr
    k = 1 + int(kfrac * (min(E, 6) - 1))
    H = 8 * H8
    wl = P.W.Workload("propq", R=R, epr=epr, bs=bs, H=H, k=k, seed=seed)
    idx, wt = P.W.routing(wl)
    idx, wt = idx.numpy(), wt.numpy()
    L = oracle_mod.layout(idx, R, epr)
    N = oracle_mod.notify(L["count"], R, bs, epr)
    args = (idx, wt, L["send_idx"], N["put_offset"], N["rank_recv_base"], R, epr, 0)
    rng = np.random.default_rng(seed)
    codes = rng.integers(-127, 128, size=(wl.P, H))
    inv = 2.0 ** inv_exp
    img = P._int8_images(codes, np.full(wl.P, inv), H)
    got, stt = oracle_mod.combine_quant(img, *args, H=H)
    assert stt == 0
    ref, _ = oracle_mod.combine(P._bf16_bits((codes * inv).astype(np.float32)), *args)
    np.testing.assert_array_equal(got, ref)


@settings(**SETTINGS)
@given(case=routings(), H8=st.integers(1, 12), dtype=st.sampled_from([0, 1]),
       capfrac=st.floats(0.0, 1.0))
def test_dispatch_verbatim_and_capacity_any_shape(oracle_mod, case, H8, dtype, capfrac):
    """Verbatim dispatch puts the bytes of x[g] in each of g's k rows (the
    receive rows being the closed-form order); with a shorter receive buffer
    the rows inside it are unchanged and status 3 is set exactly when some
    row falls outside."""
    R, epr, bs, k, idx = case
    H = 8 * H8
    T = R * bs
    rng = np.random.default_rng(H8 * 7919 + T)
    xb = rng.integers(0, 1 << 16, size=(T, H), dtype=np.uint16)
    L = oracle_mod.layout(idx, R, epr)
    N = oracle_mod.notify(L["count"], R, bs, epr)
    args = (xb, idx, L["send_idx"], N["put_offset"], N["rank_recv_base"], R, epr, dtype, 0)
    recv, stt = oracle_mod.dispatch(*args)
    assert stt == 0
    rows = P.rows_by_sort(idx)
    y = recv.view(np.uint16).reshape(-1, H)
    for g in range(T):
        for kk in range(k):
            np.testing.assert_array_equal(y[rows[g, kk]], xb[g])
    cap = int(capfrac * T * k)
    short, stt = oracle_mod.dispatch(*args, capacity_rows=cap)
    assert stt == (3 if cap < T * k else 0)
    np.testing.assert_array_equal(short[:cap], recv[:cap])


@settings(**SETTINGS)
@given(case=routings())
def test_token_layout_any_shape(oracle_mod, case):
    """Membership = the set of destination ranks of a token's experts (Python
    sets); tokens per rank = membership summed over the source rank's tokens,
    never more than the pair counts."""
    R, epr, bs, k, idx = case
    TL = oracle_mod.token_layout(idx, R, epr)
    assert TL["status"] == 0
    exp_in = np.zeros((R * bs, R), np.uint8)
    for g in range(R * bs):
        for r in {int(e) // epr for e in idx[g]}:
            exp_in[g, r] = 1
    np.testing.assert_array_equal(TL["in_rank"], exp_in)
    np.testing.assert_array_equal(TL["tokens_per_rank"], exp_in.reshape(R, bs, R).sum(axis=1))
    assert (TL["tokens_per_rank"] <= oracle_mod.layout(idx, R, epr)["rank_send"]).all()


@st.composite
def gemm_problems(draw):
    G = draw(st.integers(1, 6))
    sizes = draw(st.lists(st.integers(0, 20), min_size=G, max_size=G))
    K = draw(st.integers(1, 300))
    N = draw(st.integers(1, 24))
    pad = draw(st.integers(0, 16))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return G, sizes, K, N, pad, seed


@settings(**SETTINGS)
@given(prob=gemm_problems())
def test_grouped_gemm_any_shape(oracle_mod, prob):
    """Each group's rows times that group's weights, as numpy int64 matmuls,
    over random group sizes (empty groups included), K, N and row strides;
    a random subset of listed rows gives the same rows."""
    G, sizes, K, N, pad, seed = prob
    rng = np.random.default_rng(seed)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    M = int(off[-1])
    a = rng.integers(-128, 128, (M, K + pad)).astype(np.int8)
    b = rng.integers(-128, 128, (G, N, K)).astype(np.int8)
    c = oracle_mod.grouped_gemm(a.view(np.uint8), off, b)
    assert c.shape == (M, N)
    for g in range(G):
        ref = a[off[g]:off[g + 1], :K].astype(np.int64) @ b[g].T.astype(np.int64)
        np.testing.assert_array_equal(c[off[g]:off[g + 1]], ref)
    if M:
        rows = rng.choice(M, size=min(M, 5), replace=False).astype(np.int64)
        np.testing.assert_array_equal(
            oracle_mod.grouped_gemm(a[rows].view(np.uint8), off, b, rows=rows), c[rows])


@settings(**SETTINGS)
@given(R=st.integers(1, 4), epr=st.integers(1, 4), bs=st.integers(1, 10),
       kfrac=st.floats(0.0, 1.0), H8=st.integers(1, 8), dtype=st.sampled_from([0, 1]),
       seed=st.integers(0, 10 ** 6))
def test_deq_combine_unit_scales_any_shape(oracle_mod, R, epr, bs, kfrac, H8, dtype, seed):
    """With unit weight and row scales and accumulators exact in the token
    dtype (|acc| <= 256), DeqCombine is the combine of those values, bit for
    bit, in bf16 and fp16."""
    E = R * epr
    k = 1 + int(kfrac * (min(E, 6) - 1))
    H = 8 * H8
    wl = P.W.Workload("propdq", R=R, epr=epr, bs=bs, H=H, k=k, seed=seed)
    idx, wt = P.W.routing(wl)
    idx, wt = idx.numpy(), wt.numpy()
    L = oracle_mod.layout(idx, R, epr)
    N = oracle_mod.notify(L["count"], R, bs, epr)
    rng = np.random.default_rng(seed)
    acc2 = rng.integers(-256, 257, (wl.P, H)).astype(np.int32)
    args = (idx, wt, L["send_idx"], N["put_offset"], N["rank_recv_base"], R, epr, dtype)
    out, stt = oracle_mod.deq_combine(acc2, np.ones((E, H), np.float32),
                                      np.ones(wl.P, np.float32), *args)
    assert stt == 0
    ref, _ = oracle_mod.combine(oracle_mod.from_f32(acc2.astype(np.float32), dtype), *args)
    np.testing.assert_array_equal(out, ref)


@settings(**SETTINGS)
@given(M=st.integers(1, 12), I8=st.integers(1, 40), seed=st.integers(0, 2 ** 31 - 1))
def test_swiglu_quant_any_shape(oracle_mod, M, I8, seed):
    """GMM1 epilogue against a float64 restatement of dequant -> SwiGLU: the
    stored 1/scale, the dequantisation error bound, codes equal to the
    round-half-even of the float64 value away from ties, and zero pads."""
    I = 8 * I8
    rng = np.random.default_rng(seed)
    acc = np.round(rng.standard_normal((M, 2 * I)) * 2.0 ** 17).astype(np.int32)
    ws = (rng.uniform(0.5, 1.5, 2 * I) * 4e-4).astype(np.float32)
    ts = rng.uniform(0.005, 0.03, M).astype(np.float32)
    img = oracle_mod.swiglu_quant(acc, ws, ts)
    ia = (I + 31) // 32 * 32
    assert img.shape == (M, ia + 32)
    assert not img[:, I:ia].any() and not img[:, ia + 4:].any()
    q = img[:, :I].view(np.int8).astype(np.int64)
    inv = img[:, ia:ia + 4].copy().view(np.float32)[:, 0].astype(np.float64)
    v = acc.astype(np.float64) * ws.astype(np.float64) * ts.astype(np.float64)[:, None]
    gate, up = v[:, :I], v[:, I:]
    h = gate / (1.0 + np.exp(-gate)) * up
    amax = np.abs(h).max(axis=1)
    np.testing.assert_allclose(inv, (amax + 1e-12) / 127, rtol=1e-5)
    err = np.abs(q * inv[:, None] - h)
    assert (err <= (amax[:, None] + 1e-12) / 254 * (1 + 2.0 ** -10) + 1e-6 * np.abs(h)).all()
    t = h * (127.0 / (amax + 1e-12))[:, None]
    ok = np.abs(np.abs(t - np.floor(t)) - 0.5) > 1e-3
    np.testing.assert_array_equal(q[ok], np.rint(t)[ok].astype(np.int64))


@settings(**SETTINGS)
@given(case=routings(), frac=st.floats(0.0, 0.5), seed=st.integers(0, 2 ** 31 - 1))
def test_invalid_ids_any_shape(oracle_mod, case, frac, seed):
    """Pairs with an expert id outside [0, E) (-1, E, or far out of range) are
    not counted, get send index -1 and status 2; the valid pairs keep the
    stable numbering and their receive rows are a bijection onto
    [0, valid pairs) in the closed-form order of the valid pairs alone."""
    R, epr, bs, k, idx = case
    E = R * epr
    rng = np.random.default_rng(seed)
    idx = idx.copy()
    bad = rng.random(idx.shape) < frac
    idx[bad] = rng.choice(np.array([-1, E, E + 7, -(2 ** 31)], dtype=np.int64),
                          size=int(bad.sum())).astype(np.int32)
    L = oracle_mod.layout(idx, R, epr)
    assert L["status"] == (2 if bad.any() else 0)
    assert (L["send_idx"][bad] == -1).all()
    valid = ~bad
    cnt = L["count"].astype(np.int64)
    assert cnt.sum() == int(valid.sum())
    for s in range(R):
        sub_idx = idx[s * bs:(s + 1) * bs].reshape(-1)
        sub_send = L["send_idx"][s * bs:(s + 1) * bs].reshape(-1)
        for e in range(E):
            np.testing.assert_array_equal(sub_send[sub_idx == e], np.arange(cnt[s, e]))
    N = oracle_mod.notify(L["count"], R, bs, epr)
    rows = oracle_mod.dst_rows(idx, L["send_idx"], N["put_offset"], N["rank_recv_base"],
                               R, epr)
    assert (rows[bad] == -1).all()
    assert sorted(rows[valid].tolist()) == list(range(int(valid.sum())))
    # closed form over the valid pairs: ordered by (expert, token, k)
    g, kk = np.nonzero(valid)
    order = np.lexsort((kk, g, idx[valid]))
    np.testing.assert_array_equal(rows[g[order], kk[order]], np.arange(len(order)))
