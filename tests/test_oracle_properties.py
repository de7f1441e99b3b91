"""Property tests of the oracle over random shapes (hypothesis): the layout,
notify and receive-row invariants, the quantisation bounds and the combine
(one-hot weights give the token back; general weights within the rounding
bound of the fp64 sum), on shapes the fixed-seed pins do not reach (empty
batches, one rank, k = E, repeated experts in a token).  CPU only; skipped
where hypothesis is not installed."""
import numpy as np
import pytest
import torch

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import HealthCheck, given, settings, strategies as st  # noqa: E402

import test_oracle_pins as P  # noqa: E402  (the pins' helpers and closed forms)

SETTINGS = dict(max_examples=80, deadline=None,
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
