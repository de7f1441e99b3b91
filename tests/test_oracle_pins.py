"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each check below ties the oracle to a fact fixed by the UMDK/CAM deep-analysis
page (v2, section 2) or by mathematics: brute force on tiny inputs, invariants
of the count matrix, the closed form of the receive-row order, hand-worked
fixtures under ``tests/golden/``, exact-rational evaluation of the quantisation
formula, error bounds, and special cases that reduce to a library routine
(numpy / torch rounding).  ``test_mutants_are_caught`` then compiles broken
copies of the oracle (one plausible mistake each) and shows that some pin
fails for every one of them.
"""
import json
import os
import shutil
import subprocess
import tempfile
from fractions import Fraction

import numpy as np
import pytest
import torch

import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16_bits(vals):
    return W.bits(torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16))


def _f16_bits(vals):
    return W.bits(torch.tensor(vals, dtype=torch.float32).to(torch.float16))


def _random_routing(rng, R, epr, bs, k, distinct=True):
    E = R * epr
    T = R * bs
    if distinct:
        out = np.zeros((T, k), np.int32)
        for g in range(T):
            out[g] = rng.permutation(E)[:k]
        return out
    return rng.integers(0, E, size=(T, k), dtype=np.int32)


# ---------------------------------------------------------------------------
# Independent restatements used as pins (not the oracle's own code paths)
# ---------------------------------------------------------------------------

def brute_layout(idx, R, epr):
    """O(P^2): send index = number of EARLIER pairs of the same source rank
    routed to the same expert (section 2.3's 'send index' in stable order)."""
    T, k = idx.shape
    bs = T // R
    E = R * epr
    pairs = [(g, kk) for g in range(T) for kk in range(k)]
    send = np.full((T, k), -1, np.int64)
    count = np.zeros((R, E), np.int64)
    for (g, kk) in pairs:
        e = int(idx[g, kk])
        if not 0 <= e < E:
            continue
        s = g // bs
        count[s, e] += 1
        send[g, kk] = sum(1 for (g2, k2) in pairs
                          if g2 // bs == s and int(idx[g2, k2]) == e
                          and (g2, k2) < (g, kk))
    rank_send = count.reshape(R, R, epr).sum(axis=2)
    return send, count, rank_send


def rows_by_sort(idx):
    """Closed form of the receive-row order: ranks' rows are packed back to
    back, a rank's rows go expert by expert, an expert's rows source rank by
    source rank (putOffset, section 2.4), a source rank's rows in send-index
    order (2.3).  Since dst = e // epr is monotone in e and g = s*bs + t,
    that is the lexicographic order of (e, g, k) over all pairs."""
    T, k = idx.shape
    g = np.repeat(np.arange(T), k)
    kk = np.tile(np.arange(k), T)
    e = idx.reshape(-1).astype(np.int64)
    order = np.lexsort((kk, g, e))
    rows = np.empty(T * k, np.int64)
    rows[order] = np.arange(T * k)
    return rows.reshape(T, k)


def exact_q(x_vals, amax):
    """q = RINT(x * 127/(amax + 1e-12f)) in exact rational arithmetic (the
    page's formula without any fp32 rounding), with the distance of x*scale
    to the nearest rounding boundary."""
    eps = Fraction(float(np.float32(1e-12)))
    scale = Fraction(127) / (Fraction(float(amax)) + eps)
    q, margin = [], []
    for v in x_vals:
        t = Fraction(float(v)) * scale
        fl = t.numerator // t.denominator
        frac = t - fl
        q.append(fl + 1 if frac > Fraction(1, 2) else
                 fl if frac < Fraction(1, 2) else fl + (fl & 1))
        margin.append(abs(float(frac) - 0.5))
    return np.array(q, np.int64), np.array(margin)


# ---------------------------------------------------------------------------
# Checks (each raises AssertionError; reused by the mutant test)
# ---------------------------------------------------------------------------

def check_handworked_layout_notify(oracle):
    f = _load("handworked_layout_notify.json")
    R, epr, bs = f["R"], f["epr"], f["bs"]
    idx = np.array(f["topk_idx"], np.int32)
    L = oracle.layout(idx, R, epr)
    assert L["status"] == 0
    np.testing.assert_array_equal(L["send_idx"], f["send_idx"])
    np.testing.assert_array_equal(L["count"], f["count"])
    np.testing.assert_array_equal(L["rank_send"], f["rank_send"])
    N = oracle.notify(L["count"], R, bs, epr)
    np.testing.assert_array_equal(N["put_offset"], f["put_offset"])
    np.testing.assert_array_equal(N["total_recv"], f["total_recv"])
    np.testing.assert_array_equal(N["rank_recv_base"], f["rank_recv_base"])
    np.testing.assert_array_equal(N["recv_per_expert"], f["recv_per_expert"])
    assert N["max_bs"] == f["max_bs"]
    rows = oracle.dst_rows(idx, L["send_idx"], N["put_offset"],
                           N["rank_recv_base"], R, epr)
    np.testing.assert_array_equal(rows, f["rows"])


def check_layout_brute_force(oracle, seed=0, n_cases=12):
    rng = np.random.default_rng(seed)
    for c in range(n_cases):
        R = int(rng.integers(1, 5))
        epr = int(rng.integers(1, 4))
        bs = int(rng.integers(0, 9))
        E = R * epr
        k = int(rng.integers(1, E + 1))
        idx = _random_routing(rng, R, epr, bs, k, distinct=(c % 2 == 0))
        send, count, rank_send = brute_layout(idx, R, epr)
        L = oracle.layout(idx, R, epr)
        assert L["status"] == 0
        np.testing.assert_array_equal(L["send_idx"], send)
        np.testing.assert_array_equal(L["count"], count)
        np.testing.assert_array_equal(L["rank_send"], rank_send)


def check_layout_invariants(oracle, R=5, epr=7, bs=300, k=6, seed=1):
    rng = np.random.default_rng(seed)
    idx = _random_routing(rng, R, epr, bs, k)
    L = oracle.layout(idx, R, epr)
    E = R * epr
    # counts of a rank sum to bs*k (each (token,k) pair is one row)
    assert (L["count"].sum(axis=1) == bs * k).all()
    assert (L["rank_send"].sum(axis=1) == bs * k).all()
    # send indices of each (s, e) are 0,1,2,... in (t, k) order
    for s in range(R):
        sub_idx = idx[s * bs:(s + 1) * bs].reshape(-1)
        sub_send = L["send_idx"][s * bs:(s + 1) * bs].reshape(-1)
        for e in range(E):
            got = sub_send[sub_idx == e]
            np.testing.assert_array_equal(got, np.arange(L["count"][s, e]))


def check_notify_closed_form(oracle, R=6, epr=5, bs=200, k=4, seed=2):
    rng = np.random.default_rng(seed)
    idx = _random_routing(rng, R, epr, bs, k)
    L = oracle.layout(idx, R, epr)
    N = oracle.notify(L["count"], R, bs, epr)
    E = R * epr
    cnt = L["count"].astype(np.int64)
    po = N["put_offset"].reshape(E, R).astype(np.int64)
    for r in range(R):
        es = range(r * epr, (r + 1) * epr)
        walk = [(e, s) for e in es for s in range(R)]
        offs = np.array([po[e, s] for (e, s) in walk])
        vals = np.array([cnt[s, e] for (e, s) in walk])
        assert offs[0] == 0                        # exclusive: starts at 0
        np.testing.assert_array_equal(offs[1:], offs[:-1] + vals[:-1])
        assert offs[-1] + vals[-1] == N["total_recv"][r]
    assert N["total_recv"].sum() == R * bs * k
    np.testing.assert_array_equal(N["recv_per_expert"], cnt.sum(axis=0))
    np.testing.assert_array_equal(
        N["rank_recv_base"], np.concatenate([[0], np.cumsum(N["total_recv"])]))
    assert N["max_bs"] == bs


def check_rows_closed_form(oracle, R=4, epr=3, bs=50, k=5, seed=3):
    rng = np.random.default_rng(seed)
    idx = _random_routing(rng, R, epr, bs, k)
    L = oracle.layout(idx, R, epr)
    N = oracle.notify(L["count"], R, bs, epr)
    rows = oracle.dst_rows(idx, L["send_idx"], N["put_offset"],
                           N["rank_recv_base"], R, epr)
    np.testing.assert_array_equal(rows, rows_by_sort(idx))
    # a bijection onto [0, T*k); rank r's rows inside its partition
    assert sorted(rows.reshape(-1).tolist()) == list(range(R * bs * k))
    base = N["rank_recv_base"]
    dst = idx // epr
    assert ((rows >= base[dst]) & (rows < base[dst + 1])).all()


def check_invalid_ids(oracle):
    idx = np.array([[0, 5], [3, -1], [2, 1], [1, 0]], np.int32)  # E = 4
    L = oracle.layout(idx, 2, 2)
    assert L["status"] == 2
    assert L["send_idx"][0, 1] == -1 and L["send_idx"][1, 1] == -1
    assert L["count"].sum() == 6
    np.testing.assert_array_equal(L["count"], [[1, 0, 0, 1], [1, 2, 1, 0]])


def check_handworked_quant(oracle):
    f = _load("handworked_quant_rows.json")
    r0 = f["rows"][0]
    img = oracle.quant_row(_bf16_bits(r0["x"]), 0)
    assert img.size == r0["row_bytes"]
    np.testing.assert_array_equal(img[:8].view(np.int8), r0["q"])
    assert not img[8:32].any()
    assert img[32:36].view(np.uint32)[0] == int(r0["inv_scale_hex"], 16)
    assert not img[36:].any()
    r1 = f["rows"][1]
    xs = [0.0 if s == "0" else (-1.0 if s.startswith("-") else 1.0)
          * 2.0 ** int(s.lstrip("-").split("^")[1]) for s in r1["x_exact"]]
    img = oracle.quant_row(_bf16_bits(xs), 0)
    np.testing.assert_array_equal(img[:8].view(np.int8), r1["q"])
    q, margin = exact_q(xs, max(abs(v) for v in xs))
    np.testing.assert_array_equal(q, r1["q"])      # fixture vs exact formula
    assert margin.min() > 1e-3


def check_quant_properties(oracle, seed=4):
    rng = np.random.default_rng(seed)
    for H, dtype in [(8, 0), (40, 0), (136, 1), (1000, 0), (7168, 0),
                     (2048, 1)]:
        for trial in range(3):
            v = rng.standard_normal(H).astype(np.float32) * [1, 2, 1e-3][trial]
            if trial == 0:
                v[rng.integers(0, H, size=max(1, H // 100))] *= 20
            xb = _bf16_bits(v) if dtype == 0 else _f16_bits(v)
            x = (torch.from_numpy(xb.view(np.int16)).view(
                torch.bfloat16 if dtype == 0 else torch.float16)
                 .to(torch.float64).numpy())
            img = oracle.quant_row(xb, dtype)
            ha = (H + 31) // 32 * 32
            assert img.size == ha + 32
            q = img[:H].view(np.int8).astype(np.int64)
            inv = float(img[ha:ha + 4].view(np.float32)[0])
            assert not img[H:ha].any() and not img[ha + 4:].any()
            amax = np.abs(x).max()
            assert np.abs(q).max() == 127
            # 1/scale ~ (amax + 1e-12)/127
            assert abs(inv / ((amax + 1e-12) / 127) - 1) < 1e-6
            # exact formula, away from rounding boundaries
            sel = rng.choice(H, size=min(H, 64), replace=False)
            qe, margin = exact_q(x[sel], amax)
            ok = margin > 1e-4
            np.testing.assert_array_equal(q[sel][ok], qe[ok])
            # dequant error bound: amax/254 per element (plus fp32 slack)
            err = np.abs(q * inv - x)
            # slack: the fp32 product x*scale is off by <= 127*2^-24 of a step,
            # i.e. 2^-16 relative to the half step; truncation would be 2x
            assert (err <= (amax + 1e-12) / 254 * (1 + 2.0 ** -14)).all()


def check_quant_zero_row(oracle):
    img = oracle.quant_row(np.zeros(64, np.uint16), 0)
    assert not img[:64].any()
    inv = float(img[64:68].view(np.float32)[0])
    assert abs(inv / (float(np.float32(1e-12)) / 127) - 1) < 1e-6


def check_conversions(oracle, seed=5):
    rng = np.random.default_rng(seed)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 3,
        rng.standard_normal(2000).astype(np.float32) * 1e-6,
        np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 65504.0,
                  65520.0, 3e38, -3e38, 2 ** -24, 3 * 2 ** -26, 2 ** -25,
                  1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11], np.float32)])
    ref_bf = W.bits(torch.from_numpy(vals).to(torch.bfloat16))
    np.testing.assert_array_equal(oracle.from_f32(vals, 0), ref_bf)
    with np.errstate(over="ignore"):   # 65520 and 3e38 overflow to inf
        ref_h = vals.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(oracle.from_f32(vals, 1), ref_h)
    b = rng.integers(0, 1 << 16, size=5000, dtype=np.uint16)
    b = b[(b & 0x7F80) != 0x7F80]     # finite bf16 patterns
    np.testing.assert_array_equal(
        oracle.to_f32(b, 0),
        torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float().numpy())
    h = rng.integers(0, 1 << 16, size=5000, dtype=np.uint16)
    h = h[(h & 0x7C00) != 0x7C00]
    np.testing.assert_array_equal(oracle.to_f32(h, 1),
                                  h.view(np.float16).astype(np.float32))


def _one_token_combine(oracle, y_vals, w_vals, dtype=0):
    """Combine of a single token whose k pairs go to rows 0..k-1 (R=1,
    experts 0..k-1 on the one rank, so row(kk) = kk)."""
    k = len(y_vals)
    idx = np.arange(k, dtype=np.int32).reshape(1, k)
    L = oracle.layout(idx, 1, k)
    N = oracle.notify(L["count"], 1, 1, k)
    yb = (_bf16_bits if dtype == 0 else _f16_bits)(
        np.array(y_vals, np.float32).reshape(k, 1))
    out, st = oracle.combine(yb, idx, np.array([w_vals], np.float32),
                             L["send_idx"], N["put_offset"],
                             N["rank_recv_base"], 1, k, dtype)
    assert st == 0
    return float(oracle.to_f32(out, dtype)[0, 0])


def check_combine_special_cases(oracle):
    # k order: ((2^24 + 1) - 2^24) in fp32, left to right, is 0, not 1
    assert _one_token_combine(oracle, [2.0 ** 24, 1.0, -2.0 ** 24],
                              [1.0, 1.0, 1.0]) == 0.0
    # Muls then Add (two roundings), not a fused multiply-add
    y, w = 1.0 + 2 ** -7, 1.0 + 2 ** -20
    assert _one_token_combine(oracle, [-y, y], [w, w]) == 0.0
    # CAST_RINT to bf16: ties go to even
    assert _one_token_combine(oracle, [1.0], [1.0 + 2 ** -8]) == 1.0
    assert _one_token_combine(oracle, [1.0], [1.0 + 3 * 2 ** -8]) == \
        1.0 + 2 ** -6
    # fp16: ties to even, subnormal output
    assert _one_token_combine(oracle, [1.0], [1.0 + 2 ** -11], 1) == 1.0
    assert _one_token_combine(oracle, [2.0 ** -10], [3 * 2.0 ** -16], 1) == \
        2.0 ** -24


def check_combine_one_hot_and_bound(oracle, seed=6):
    rng = np.random.default_rng(seed)
    for dtype, quant_rows in [(0, False), (1, False)]:
        wl = W.Workload("pin", R=3, epr=2, bs=20, H=48, k=3, dtype=dtype,
                        quant=quant_rows, seed=99)
        idx, wt = W.routing(wl)
        idx, wt = idx.numpy(), wt.numpy()
        x = W.tokens(wl)
        L = oracle.layout(idx, wl.R, wl.epr)
        N = oracle.notify(L["count"], wl.R, wl.bs, wl.epr)
        recv, st = oracle.dispatch(W.bits(x), idx, L["send_idx"],
                                   N["put_offset"], N["rank_recv_base"],
                                   wl.R, wl.epr, dtype, 0)
        assert st == 0
        y = recv.view(np.uint16)                  # y = dispatched x
        # all the weight on one k: the output is x again
        hot = rng.integers(0, wl.k, size=wl.T)
        w1 = np.zeros_like(wt)
        w1[np.arange(wl.T), hot] = 1.0
        out, st = oracle.combine(y, idx, w1, L["send_idx"], N["put_offset"],
                                 N["rank_recv_base"], wl.R, wl.epr, dtype)
        np.testing.assert_array_equal(oracle.to_f32(out, dtype),
                                      x.float().numpy())
        # k = 1 reduces to RNE(float(y) * w), computed with torch
        tok = np.arange(wl.T)
        rows = oracle.dst_rows(idx, L["send_idx"], N["put_offset"],
                               N["rank_recv_base"], wl.R, wl.epr)
        # general weights: error bound against the fp64 sum
        out, st = oracle.combine(y, idx, wt, L["send_idx"], N["put_offset"],
                                 N["rank_recv_base"], wl.R, wl.epr, dtype)
        yf = oracle.to_f32(y, dtype).astype(np.float64)
        terms = yf[rows] * wt[..., None].astype(np.float64)   # [T, k, H]
        ref = terms.sum(axis=1)
        got = oracle.to_f32(out, dtype).astype(np.float64)
        rel = 2.0 ** -8 if dtype == 0 else 2.0 ** -10
        tol = rel * np.abs(ref) + (wl.k + 1) * 2.0 ** -23 * \
            np.abs(terms).sum(axis=1) + 2.0 ** -24
        assert (np.abs(got - ref) <= tol).all()
        del tok


def check_combine_k1(oracle):
    wl = W.Workload("pin", R=2, epr=3, bs=16, H=32, k=1, seed=7)
    idx, wt = W.routing(wl)
    y = W.expert_outputs(wl)
    L = oracle.layout(idx.numpy(), wl.R, wl.epr)
    N = oracle.notify(L["count"], wl.R, wl.bs, wl.epr)
    out, st = oracle.combine(W.bits(y), idx.numpy(), wt.numpy(),
                             L["send_idx"], N["put_offset"],
                             N["rank_recv_base"], wl.R, wl.epr, 0)
    rows = torch.from_numpy(rows_by_sort(idx.numpy())[:, 0])
    ref = (y.float()[rows] * wt[:, :1]).to(torch.bfloat16)
    np.testing.assert_array_equal(out, W.bits(ref))


def check_dispatch_capacity(oracle):
    wl = W.WORKLOADS["tiny"]
    idx, _ = W.routing(wl)
    x = W.tokens(wl)
    L = oracle.layout(idx.numpy(), wl.R, wl.epr)
    N = oracle.notify(L["count"], wl.R, wl.bs, wl.epr)
    cap = wl.P - 5
    recv, st = oracle.dispatch(W.bits(x), idx.numpy(), L["send_idx"],
                               N["put_offset"], N["rank_recv_base"], wl.R,
                               wl.epr, 0, 1, capacity_rows=cap)
    assert st == 3 and recv.shape[0] == cap
    full, st = oracle.dispatch(W.bits(x), idx.numpy(), L["send_idx"],
                               N["put_offset"], N["rank_recv_base"], wl.R,
                               wl.epr, 0, 1)
    assert st == 0
    np.testing.assert_array_equal(recv, full[:cap])


def _int8_images(codes, inv, H):
    """Row images: codes int8 [n, H], inv float32 [n]."""
    ha = (H + 31) // 32 * 32
    n = codes.shape[0]
    img = np.zeros((n, ha + 32), np.uint8)
    img[:, :H] = codes.astype(np.int8).view(np.uint8)
    img[:, ha:ha + 4] = np.asarray(inv, np.float32).reshape(n, 1).view(np.uint8)
    return img


def check_combine_quant(oracle, seed=8):
    rng = np.random.default_rng(seed)
    for H in (40, 96):       # H % 32 != 0 checks where 1/scale is read from
        wl = W.Workload("pinq", R=3, epr=2, bs=12, H=H, k=3, seed=5)
        idx, wt = W.routing(wl)
        idx, wt = idx.numpy(), wt.numpy()
        L = oracle.layout(idx, wl.R, wl.epr)
        N = oracle.notify(L["count"], wl.R, wl.bs, wl.epr)
        args = (idx, wt, L["send_idx"], N["put_offset"], N["rank_recv_base"],
                wl.R, wl.epr, 0)
        codes = rng.integers(-127, 128, size=(wl.P, H))
        # 1/scale = 1 or an exact power of two: float(q) * inv is exact, so
        # the result is the (pinned) combine of the exactly dequantised rows
        for inv in (1.0, 2.0 ** -7, 2.0 ** 5):
            img = _int8_images(codes, np.full(wl.P, inv), H)
            got, st = oracle.combine_quant(img, *args, H=H)
            assert st == 0
            y = _bf16_bits((codes * inv).astype(np.float32))
            ref, _ = oracle.combine(y, *args)
            np.testing.assert_array_equal(got, ref)
        # general 1/scale: error bound against the fp64 value
        inv = rng.uniform(1e-3, 3e-2, size=wl.P).astype(np.float32)
        img = _int8_images(codes, inv, H)
        got, _ = oracle.combine_quant(img, *args, H=H)
        rows = rows_by_sort(idx)
        terms = (codes[rows] * inv[rows][..., None].astype(np.float64)
                 * wt[..., None].astype(np.float64))
        ref = terms.sum(axis=1)
        g = oracle.to_f32(got, 0).astype(np.float64)
        tol = 2.0 ** -8 * np.abs(ref) + (wl.k + 2) * 2.0 ** -23 * \
            np.abs(terms).sum(axis=1) + 1e-30
        assert (np.abs(g - ref) <= tol).all()


def check_token_layout(oracle, seed=9):
    rng = np.random.default_rng(seed)
    for c in range(6):
        R = int(rng.integers(1, 6))
        epr = int(rng.integers(1, 4))
        bs = int(rng.integers(0, 30))
        E = R * epr
        k = int(rng.integers(1, E + 1))
        idx = _random_routing(rng, R, epr, bs, k, distinct=(c % 2 == 0))
        TL = oracle.token_layout(idx, R, epr)
        L = oracle.layout(idx, R, epr)
        assert TL["status"] == 0
        # brute force: a Python set of destination ranks per token
        exp_in = np.zeros((R * bs, R), np.uint8)
        for g in range(R * bs):
            for r in {int(e) // epr for e in idx[g]}:
                exp_in[g, r] = 1
        np.testing.assert_array_equal(TL["in_rank"], exp_in)
        np.testing.assert_array_equal(
            TL["tokens_per_rank"], exp_in.reshape(R, bs, R).sum(axis=1))
        # never more tokens than pairs; equal when a rank owns one expert and
        # experts are distinct per token
        assert (TL["tokens_per_rank"] <= L["rank_send"]).all()
        if epr == 1 and c % 2 == 0:
            np.testing.assert_array_equal(TL["tokens_per_rank"], L["rank_send"])


def check_exp(oracle):
    x = np.linspace(-87.0, 88.0, 400001, dtype=np.float32)
    y = oracle.exp_f32(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.abs(y - ref) / np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert ulp.max() <= 1.0                    # textbook method, fp32 FMA Horner
    assert float(oracle.exp_f32(np.array([0.0], np.float32))[0]) == 1.0
    assert (np.diff(y) >= 0).all()             # monotone on the sweep


def _swiglu_inputs(rng, M, I, big=False):
    acc = np.round(rng.standard_normal((M, 2 * I)) * 2.0 ** 17).astype(np.int64)
    if big:                                    # beyond 2^24: the cast rounds
        acc[:, ::37] = acc[:, ::37] * 64 + 1
    acc = acc.astype(np.int32)
    ws = (rng.uniform(0.5, 1.5, 2 * I) * 4e-4).astype(np.float32)
    ts = rng.uniform(0.005, 0.03, M).astype(np.float32)
    return acc, ws, ts


def check_swiglu_quant(oracle, seed=10):
    for exp in ("cw", "libm"):
        _check_swiglu_quant(oracle, seed, exp)
    # the two readings of Exp agree up to the exp's last bit: codes move by
    # at most one step, and only where the value sits next to a rounding tie
    rng = np.random.default_rng(seed + 1)
    acc, ws, ts = _swiglu_inputs(rng, 400, 256, True)
    a = oracle.swiglu_quant(acc, ws, ts, exp="cw")
    b = oracle.swiglu_quant(acc, ws, ts, exp="libm")
    qa = a[:, :256].view(np.int8).astype(np.int64)
    qb = b[:, :256].view(np.int8).astype(np.int64)
    assert np.abs(qa - qb).max() <= 1 and (qa != qb).mean() < 1e-3
    ia = a[:, 256:260].copy().view(np.int32)[:, 0].astype(np.int64)
    ib = b[:, 256:260].copy().view(np.int32)[:, 0].astype(np.int64)
    assert np.abs(ia - ib).max() <= 8
    np.testing.assert_array_equal(a[:, 260:], b[:, 260:])


def _check_swiglu_quant(oracle, seed, exp):
    rng = np.random.default_rng(seed)
    for I, big in ((40, False), (256, True)):
        M = 24
        acc, ws, ts = _swiglu_inputs(rng, M, I, big)
        img = oracle.swiglu_quant(acc, ws, ts, exp=exp)
        ia = (I + 31) // 32 * 32
        assert img.shape == (M, ia + 32)
        q = img[:, :I].view(np.int8).astype(np.int64)
        inv = img[:, ia:ia + 4].copy().view(np.float32)[:, 0].astype(np.float64)
        assert not img[:, I:ia].any() and not img[:, ia + 4:].any()
        # fp64 restatement of dequant -> SwiGLU (independent arithmetic)
        v = acc.astype(np.float64) * ws.astype(np.float64) * ts.astype(np.float64)[:, None]
        gate, up = v[:, :I], v[:, I:]
        h = gate / (1.0 + np.exp(-gate)) * up
        amax = np.abs(h).max(axis=1)
        np.testing.assert_allclose(inv, (amax + 1e-12) / 127, rtol=1e-5)
        # dequantised values within the quantisation step (+ fp32 slack)
        err = np.abs(q * inv[:, None] - h)
        assert (err <= (amax[:, None] + 1e-12) / 254 * (1 + 2.0 ** -10)
                + 1e-6 * np.abs(h)).all()
        # codes equal round-half-even of the fp64 value away from ties
        t = h * (127.0 / (amax + 1e-12))[:, None]
        margin = np.abs(np.abs(t - np.floor(t)) - 0.5)
        ok = margin > 1e-3
        np.testing.assert_array_equal(q[ok], np.rint(t)[ok].astype(np.int64))
        # a listed-rows call gives the same images
        rows = np.array([3, 0, M - 1], np.int64)
        np.testing.assert_array_equal(oracle.swiglu_quant(acc, ws, ts, rows=rows, exp=exp),
                                      img[rows])
    # gate = 0 everywhere: silu(0) = 0, the row is all zero codes
    acc = np.zeros((2, 64), np.int32)
    acc[:, 32:] = 12345
    img = oracle.swiglu_quant(acc, np.ones(64, np.float32), np.ones(2, np.float32),
                              exp=exp)
    assert not img[:, :32].any()
    assert abs(float(img[0, 32:36].copy().view(np.float32)[0]) /
               (float(np.float32(1e-12)) / 127) - 1) < 1e-6


def check_grouped_gemm(oracle, seed=11):
    rng = np.random.default_rng(seed)
    # numpy int64 matmul per group, with an empty group and a ragged K
    for G, N, K, sizes in ((3, 5, 37, (3, 0, 7)), (4, 16, 130, (1, 9, 0, 20))):
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
        M = int(off[-1])
        lda = K + 11                            # codes at byte 0 of wider rows
        a = rng.integers(-127, 128, (M, lda)).astype(np.int8)
        b = rng.integers(-127, 128, (G, N, K)).astype(np.int8)
        c = oracle.grouped_gemm(a.view(np.uint8), off, b)
        for g in range(G):
            ref = a[off[g]:off[g + 1], :K].astype(np.int64) @ b[g].T.astype(np.int64)
            np.testing.assert_array_equal(c[off[g]:off[g + 1]], ref)
        # listed rows (a holds only those rows) give the same results
        rows = np.array([M - 1, 0, 2], np.int64)
        np.testing.assert_array_equal(
            oracle.grouped_gemm(a[rows].view(np.uint8), off, b, rows=rows), c[rows])
    # identity weights return the codes; group g's weights g*I scale by g
    K = 24
    off = np.array([0, 4, 9], np.int64)
    a = rng.integers(-127, 128, (9, K)).astype(np.int8)
    b = np.stack([np.eye(K, dtype=np.int8), 2 * np.eye(K, dtype=np.int8)])
    c = oracle.grouped_gemm(a.view(np.uint8), off, b)
    np.testing.assert_array_equal(c[:4], a[:4].astype(np.int32))
    np.testing.assert_array_equal(c[4:], 2 * a[4:].astype(np.int32))
    # the extreme sum: K = 7168 products of 127 * 127 (and of -127 * 127)
    K = 7168
    a = np.full((2, K), 127, np.int8)
    a[1] = -127
    b = np.full((1, 1, K), 127, np.int8)
    c = oracle.grouped_gemm(a.view(np.uint8), np.array([0, 2], np.int64), b)
    assert c[0, 0] == 127 * 127 * K and c[1, 0] == -127 * 127 * K


def check_deq_combine(oracle, seed=12):
    rng = np.random.default_rng(seed)
    R, epr, bs, k, H = 2, 3, 9, 3, 40
    wl = W.Workload("dq", R=R, epr=epr, bs=bs, H=H, k=k, seed=seed)
    idx, wt = W.routing(wl)
    idx, wt = idx.numpy(), wt.numpy()
    L = oracle.layout(idx, R, epr)
    N = oracle.notify(L["count"], R, bs, epr)
    P = R * bs * k
    args = (idx, wt, L["send_idx"], N["put_offset"], N["rank_recv_base"], R, epr, 0)
    # unit scales and bf16-exact accumulators: the pinned combine of those values
    acc2 = rng.integers(-256, 257, (P, H)).astype(np.int32)
    ones_w = np.ones((R * epr, H), np.float32)
    ones_r = np.ones(P, np.float32)
    out, st = oracle.deq_combine(acc2, ones_w, ones_r, *args)
    assert st == 0
    y_bits = oracle.from_f32(acc2.astype(np.float32), 0)
    ref, _ = oracle.combine(y_bits, idx, wt, L["send_idx"], N["put_offset"],
                            N["rank_recv_base"], R, epr, 0)
    np.testing.assert_array_equal(out, ref)
    # general scales: float64 bound
    acc2 = rng.integers(-2 ** 20, 2 ** 20, (P, H)).astype(np.int32)
    ws = rng.uniform(0.5, 1.5, (R * epr, H)).astype(np.float32) * 1e-4
    rs = rng.uniform(0.001, 0.05, P).astype(np.float32)
    out, st = oracle.deq_combine(acc2, ws, rs, *args)
    assert st == 0
    rows = oracle.dst_rows(idx, L["send_idx"], N["put_offset"], N["rank_recv_base"], R, epr)
    y = (acc2[rows].astype(np.float64) * ws[idx].astype(np.float64)
         * rs[rows].astype(np.float64)[..., None])
    exact = (y * wt[..., None].astype(np.float64)).sum(axis=1)
    got = oracle.to_f32(out, 0).astype(np.float64)
    bound = np.abs(exact) * 2.0 ** -8 + (np.abs(y) * wt[..., None]).sum(axis=1) * 2.0 ** -20
    assert (np.abs(got - exact) <= bound + 1e-30).all()
    # two roundings per term, checked where they show in bf16: (1 + 2^-8)
    # then + 673 * (24929 * 2^-48) = 2^-24 + 2^-48.  Rounded product:
    # 1 + 2^-8 + 2^-24 is an fp32 tie (-> 1 + 2^-8), a bf16 tie (-> 1.0);
    # a fused multiply-add would give 1 + 2^-8 + 2^-23 -> 1 + 2^-7.
    idx2 = np.array([[0, 1]], np.int32)
    wt2 = np.array([[2.0 ** -8, 24929 * 2.0 ** -48]], np.float32)
    L2 = oracle.layout(idx2, 1, 2)
    N2 = oracle.notify(L2["count"], 1, 1, 2)
    r2 = oracle.dst_rows(idx2, L2["send_idx"], N2["put_offset"], N2["rank_recv_base"], 1, 2)
    a2 = np.zeros((2, 8), np.int32)
    a2[r2[0, 0]] = 257
    a2[r2[0, 1]] = 673
    out2, st = oracle.deq_combine(a2, np.ones((2, 8), np.float32), np.ones(2, np.float32),
                                  idx2, wt2, L2["send_idx"], N2["put_offset"],
                                  N2["rank_recv_base"], 1, 2, 0)
    assert st == 0 and (out2 == 0x3F80).all()
    # listed tokens: rows in (token, k) order give the same output rows
    toks = np.array([5, 0, R * bs - 1], np.int64)
    sub, st = oracle.deq_combine(acc2[rows[toks].reshape(-1)], ws,
                                 rs[rows[toks].reshape(-1)], *args, tokens=toks)
    assert st == 0
    np.testing.assert_array_equal(sub, out[toks])


def check_deep_moe(oracle, seed=13):
    R, epr, bs, k, H, I = 2, 2, 12, 2, 64, 32
    wl = W.Workload("deep", R=R, epr=epr, bs=bs, H=H, k=k, seed=seed)
    idx, wt = W.routing(wl)
    idx, wt = idx.numpy(), wt.numpy()
    x = W.tokens(wl)
    w1, ws1, w2, ws2 = (t.numpy() for t in W.moe_weights(R * epr, H, I, seed=seed))
    res = oracle.deep_moe(W.bits(x), idx, wt, R, epr, 0, w1, ws1, w2, ws2)
    # expert groups: the exclusive prefix of the per-expert row counts
    L = oracle.layout(idx, R, epr)
    N = oracle.notify(L["count"], R, bs, epr)
    np.testing.assert_array_equal(
        res["group_off"], np.concatenate([[0], np.cumsum(N["recv_per_expert"])]))
    # float64 MoE without quantisation: agreement within the INT8 noise
    xf = x.float().numpy().astype(np.float64)
    ref = np.zeros_like(xf)
    for t in range(R * bs):
        for kk in range(k):
            e = idx[t, kk]
            v = (w1[e].astype(np.float64) * ws1[e][:, None]) @ xf[t]
            h = v[:I] / (1 + np.exp(-v[:I])) * v[I:]
            y = (w2[e].astype(np.float64) * ws2[e][:, None]) @ h
            ref[t] += wt[t, kk] * y
    got = oracle.to_f32(res["out"], 0).astype(np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 0.03, rel
    # listed tokens give the same rows
    toks = np.array([3, 0, R * bs - 1], np.int64)
    sub = oracle.deep_moe(W.bits(x), idx, wt, R, epr, 0, w1, ws1, w2, ws2, tokens=toks)
    np.testing.assert_array_equal(sub["out"], res["out"][toks])


ALL_CHECKS = [
    check_handworked_layout_notify, check_layout_brute_force,
    check_layout_invariants, check_notify_closed_form, check_rows_closed_form,
    check_invalid_ids, check_handworked_quant, check_quant_properties,
    check_quant_zero_row, check_conversions, check_combine_special_cases,
    check_combine_one_hot_and_bound, check_combine_k1, check_dispatch_capacity,
    check_combine_quant, check_token_layout, check_exp, check_swiglu_quant,
    check_grouped_gemm, check_deq_combine, check_deep_moe,
]


@pytest.mark.parametrize("check", ALL_CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(oracle_mod, check):
    check(oracle_mod)


# ---------------------------------------------------------------------------
# Mutants: each is one plausible mistake; some pin must catch every one.
# ---------------------------------------------------------------------------

MUTANTS = {
    "rint_truncates": ("(int)nearbyintf(v)", "(int)truncf(v)", 0),
    "requant_rint_truncates": ("(int)nearbyintf(v)", "(int)truncf(v)", 1),
    "no_epsilon": ("amax + 1e-12f", "amax + 0.0f", 0),
    "requant_no_epsilon": ("amax + 1e-12f", "amax + 0.0f", 1),
    "stores_scale": ("1.0f / scale", "scale", 0),
    "fused_multiply_add": ("acc[h] = acc[h] + prod;",
                           "acc[h] = fmaf(to_f32(dtype, yrow[h]), w, acc[h]);", 0),
    "combine_reverse_k": ("for (int kk = 0; kk < k; ++kk) {\n"
                          "      const int64_t row",
                          "for (int kk = k - 1; kk >= 0; --kk) {\n"
                          "      const int64_t row", 0),
    "send_idx_inclusive": ("send_idx[p] = cnt[e];\n        cnt[e] += 1;",
                           "cnt[e] += 1;\n        send_idx[p] = cnt[e];"),
    "put_offset_source_major": ("for (int j = 0; j < epr; ++j) {\n"
                                "      const int e = r * epr + j;\n"
                                "      for (int s = 0; s < R; ++s) {",
                                "for (int s = 0; s < R; ++s) {\n"
                                "      for (int j = 0; j < epr; ++j) {\n"
                                "      const int e = r * epr + j;"),
    "put_offset_inclusive": ("put_offset[(int64_t)e * R + s] = run;\n"
                             "        run += count[(int64_t)s * E + e];",
                             "run += count[(int64_t)s * E + e];\n"
                             "        put_offset[(int64_t)e * R + s] = run;"),
    "bf16_round_half_up": ("u += 0x7fffu + lsb;", "u += 0x8000u + 0 * lsb;"),
    "row_uses_dst_rank_index": ("put_offset[(int64_t)e * R + s] +",
                                "put_offset[(int64_t)e * R + dst] +"),
    "amax_signed": ("fabsf(to_f32(dtype, xrow[h]))", "(to_f32(dtype, xrow[h]))"),
    "dequant_ignores_scale": ("const float t = (float)(int8_t)img[h] * inv;",
                              "const float t = (float)(int8_t)img[h] + 0.0f * inv;"),
    "dequant_scale_after_codes": ("memcpy(&inv, img + h_align, 4);",
                                  "memcpy(&inv, img + H, 4);"),
    "token_layout_counts_pairs": ("row[e / epr] = 1;", "row[e / epr] += 1;"),
    "swiglu_halves_swapped": ("float gate = (float)a_row[j];", "float gate = (float)a_row[I + j];"),
    "swiglu_no_token_scale": ("      gate = gate * ts;\n", "      gate = gate * 1.0f;\n"),
    "swiglu_sigmoid_not_silu": ("const float sg = gate / d;", "const float sg = 1.0f / d;"),
    "exp_sign_error": ("const float e = exp_fn(-gate);", "const float e = exp_fn(gate);"),
    "exp_low_part_dropped": ("r = fmaf(-n, -2.12194440e-4f, r);", "r = fmaf(-n, 0.0f, r);"),
    "gemm_always_group_zero": ("b + ((int64_t)g * N + n) * K;", "b + ((int64_t)0 * N + n) * K;"),
    "gemm_listed_rows_by_global_index": ("a + (rows ? i : m) * lda;", "a + m * lda;"),
    "deq_combine_scale_of_expert_zero": ("weight_scale + (int64_t)e * H;",
                                         "weight_scale + (int64_t)0 * H;"),
    "deq_combine_no_row_scale": ("        y = y * ts;\n", "        y = y * 1.0f;\n"),
    "deq_combine_fused_multiply_add": ("acc[h] = acc[h] + prod;",
                                       "acc[h] = fmaf(y, w, acc[h]);", 2),
    "exp_horner_coefficient_order": ("p = fmaf(p, r, 4.16666667e-2f);", "p = fmaf(p, r, 8.33333333e-3f);"),
    "rank_send_strided_experts": ("sum += cnt[r * epr + j];", "sum += cnt[j * R + r];"),
    "invalid_id_send_index_zero": ("send_idx[p] = -1;", "send_idx[p] = 0;"),
    "rank_recv_base_inclusive": ("rank_recv_base[r] = base;\n    base += total_recv[r];",
                                 "base += total_recv[r];\n    rank_recv_base[r] = base;"),
    "recv_per_expert_one_source": ("for (int s = 0; s < R; ++s) sum += count[(int64_t)s * E + e];",
                                   "for (int s = 0; s < 1; ++s) sum += count[(int64_t)s * E + e];"),
    "max_bs_counts_all_ranks": ("max_bs[0] = bs;", "max_bs[0] = bs * R;"),
    "source_rank_by_modulo": ("const int64_t s = g / bs;", "const int64_t s = g % R;"),
    "quant_pads_not_zeroed": ("memset(out, 0, (size_t)Sq);", "memset(out, 0x5a, (size_t)Sq);"),
    "verbatim_drops_last_element": ("memcpy(image, xrow, (size_t)S);",
                                    "memcpy(image, xrow, (size_t)S - 2); memset(image + S - 2, 0, 2);"),
    "combine_weight_of_first_k": ("const float w = topk_weights[g * k + kk];",
                                  "const float w = topk_weights[g * k];", 0),
    "combine_quant_weight_of_first_k": ("const float w = topk_weights[g * k + kk];",
                                        "const float w = topk_weights[g * k];", 1),
    "f16_ties_toward_zero": ("_Float16 h = (_Float16)f;",
                             "_Float16 h = (_Float16)nextafterf(f, 0.0f);"),
    "swiglu_up_uses_gate_scale": ("up = up * weight_scale[I + j];", "up = up * weight_scale[j];"),
    "gemm_drops_last_k": ("for (int kk = 0; kk < K; ++kk) acc +=",
                          "for (int kk = 0; kk < K - 1; ++kk) acc +="),
    "requant_scale_stored": ("const float inv = 1.0f / scale;\n    memcpy(img + i_align",
                             "const float inv = scale;\n    memcpy(img + i_align"),
    "deq_combine_weight_scale_by_row": ("y = y * ws[h];", "y = y * ws[0];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutants_are_caught(oracle_mod, name):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    here = os.path.dirname(os.path.abspath(oracle_mod.__file__))
    src = open(os.path.join(here, "moe_oracle.c")).read()
    old, new = MUTANTS[name][:2]
    occurrence = MUTANTS[name][2] if len(MUTANTS[name]) > 2 else None
    if occurrence is None:
        assert src.count(old) == 1, "mutation anchor not unique: " + name
    else:   # replace only the given occurrence of a repeated anchor
        parts = src.split(old)
        assert len(parts) > occurrence + 1, "mutation anchor not found: " + name
        src = old.join(parts[:occurrence + 1]) + "\x00" + old.join(parts[occurrence + 1:])
        old = "\x00"
    tmp = tempfile.mkdtemp()
    try:
        shutil.copy(os.path.join(here, "moe_oracle.h"), tmp)
        with open(os.path.join(tmp, "moe_oracle.c"), "w") as f:
            f.write(src.replace(old, new))
        so = os.path.join(tmp, "libmutant.so")
        from oracle import build as ob
        subprocess.run(["gcc", *ob.CFLAGS, "-w", os.path.join(tmp, "moe_oracle.c"),
                        "-o", so, "-lm"], check=True)
        prev = oracle_mod.use_library(so)
        caught = []
        try:
            for check in ALL_CHECKS:
                try:
                    check(oracle_mod)
                except AssertionError:
                    caught.append(check.__name__)
        finally:
            oracle_mod.restore_library(prev)
        assert caught, "no pin catches mutant " + name
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
