"""CPU oracle for the MoE expert-parallel token pipeline (numpy front end).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package.  The product library never calls it and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (plain single-threaded C, one IEEE
rounding per fp32 operation); this module only marshals numpy arrays.
Stages follow the "EP Normal" pipeline of the UMDK/CAM deep-analysis page
(v2), section 2: 2.3 dispatch layout, 2.4 notify, 2.5 dispatch with dynamic
INT8 quantisation, 2.6 combine.

Arrays of 16-bit floats (bf16 / fp16) are passed as ``np.uint16`` bit
patterns; ``dtype`` is 0 for bf16 and 1 for fp16.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i8p = ctypes.POINTER(ctypes.c_int8)
_f32p = ctypes.POINTER(ctypes.c_float)


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i, i64 = ctypes.c_int, ctypes.c_int64
        for name in ("oracle_bf16_to_f32", "oracle_f16_to_f32"):
            getattr(L, name).argtypes = [_u16p, _f32p, i64]
        for name in ("oracle_f32_to_bf16", "oracle_f32_to_f16"):
            getattr(L, name).argtypes = [_f32p, _u16p, i64]
        L.oracle_layout.argtypes = [i, i, i, i, _i32p, _i32p, _i32p, _i32p]
        L.oracle_notify.argtypes = [i, i, i, _i32p, _i32p, _i32p, _i64p,
                                    _i32p, _i32p]
        L.oracle_dst_row.argtypes = [i, i, i, i, _i32p, _i32p, _i32p, _i64p,
                                     i64, i]
        L.oracle_dst_row.restype = i64
        L.oracle_dst_rows.argtypes = [i, i, i, i, _i32p, _i32p, _i32p, _i64p,
                                      _i64p]
        L.oracle_row_bytes.argtypes = [i, i]
        L.oracle_row_bytes.restype = i64
        L.oracle_quant_row.argtypes = [i, i, _u16p, _u8p]
        L.oracle_dispatch.argtypes = [i, i, i, i, i, i, i, _u16p, _i32p,
                                      _i32p, _i32p, _i64p, _u8p, i64]
        L.oracle_dispatch_tokens.argtypes = [i, i, i, i, i, i, i, _u16p,
                                             _i32p, _i32p, _i32p, _i64p,
                                             _i64p, i64, _u8p, _i64p]
        L.oracle_combine_tokens.argtypes = [i, i, i, i, i, i, _u16p, i64,
                                            _i32p, _f32p, _i32p, _i32p,
                                            _i64p, _i64p, i64, _u16p]
        L.oracle_token_layout.argtypes = [i, i, i, i, _i32p, _i32p, _u8p]
        L.oracle_exp_f32.argtypes = [_f32p, _f32p, i64]
        for name in ("oracle_swiglu_quant_rows", "oracle_swiglu_quant_rows_libm"):
            getattr(L, name).argtypes = [i64, i, _i32p, _f32p, _f32p, _i64p, i64, _u8p]
        L.oracle_combine_quant_tokens.argtypes = [i, i, i, i, i, i, _u8p, i64,
                                                  _i32p, _f32p, _i32p, _i32p,
                                                  _i64p, _i64p, i64, _u16p]
        L.oracle_grouped_gemm_i8.argtypes = [i, _i64p, i, i, _i8p, i64, _i8p,
                                             _i64p, i64, _i32p]
        L.oracle_deq_combine_tokens.argtypes = [i, i, i, i, i, i, _i32p, i64,
                                                _f32p, _f32p, _i32p, _f32p,
                                                _i32p, _i32p, _i64p, _i64p,
                                                i64, _u16p]
        _lib = L
    return _lib


def use_library(path):
    """Swap in another build of the oracle (tests use this to run the pins
    against deliberately broken copies); returns the previous library."""
    global _lib
    prev = lib()
    _lib = None
    saved = _build.build
    try:
        _build.build = lambda: path
        lib()
    finally:
        _build.build = saved
    return prev


def restore_library(prev):
    global _lib
    _lib = prev


def _p(a, ptype):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ptype)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def row_bytes(H, quant):
    """Receive-row size in bytes: align32(H) + 32 for INT8 rows, else 2H."""
    return int(lib().oracle_row_bytes(int(H), int(bool(quant))))


# ---- number conversions (exported for pinning) ---------------------------

def to_f32(bits, dtype):
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, np.float32)
    fn = lib().oracle_bf16_to_f32 if dtype == 0 else lib().oracle_f16_to_f32
    fn(_p(bits, _u16p), _p(out, _f32p), bits.size)
    return out


def from_f32(vals, dtype):
    vals = _c(vals, np.float32)
    out = np.empty(vals.shape, np.uint16)
    fn = lib().oracle_f32_to_bf16 if dtype == 0 else lib().oracle_f32_to_f16
    fn(_p(vals, _f32p), _p(out, _u16p), vals.size)
    return out


# ---- the four stages -----------------------------------------------------

def layout(topk_idx, R, epr):
    """Stage 1.  topk_idx int32 [T, k] (T = R*bs) -> dict(count [R,E],
    rank_send [R,R], send_idx [T,k], status)."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    bs = T // R
    assert bs * R == T
    E = R * epr
    count = np.zeros((R, E), np.int32)
    rank_send = np.zeros((R, R), np.int32)
    send_idx = np.zeros((T, k), np.int32)
    st = lib().oracle_layout(R, bs, k, epr, _p(idx, _i32p), _p(count, _i32p),
                             _p(rank_send, _i32p), _p(send_idx, _i32p))
    return dict(count=count, rank_send=rank_send, send_idx=send_idx,
                status=st)


def notify(count, R, bs, epr):
    """Stage 2.  count int32 [R, E] -> dict(put_offset [E*R],
    total_recv [R], rank_recv_base [R+1] int64, recv_per_expert [E],
    max_bs, status)."""
    count = _c(count, np.int32)
    E = R * epr
    assert count.shape == (R, E)
    put_offset = np.zeros(E * R, np.int32)
    total_recv = np.zeros(R, np.int32)
    base = np.zeros(R + 1, np.int64)
    rpe = np.zeros(E, np.int32)
    max_bs = np.zeros(1, np.int32)
    st = lib().oracle_notify(R, bs, epr, _p(count, _i32p),
                             _p(put_offset, _i32p), _p(total_recv, _i32p),
                             _p(base, _i64p), _p(rpe, _i32p),
                             _p(max_bs, _i32p))
    return dict(put_offset=put_offset, total_recv=total_recv,
                rank_recv_base=base, recv_per_expert=rpe,
                max_bs=int(max_bs[0]), status=st)


def dst_rows(topk_idx, send_idx, put_offset, rank_recv_base, R, epr):
    """Row id of every pair, int64 [T, k] (-1 for a bad expert id)."""
    idx = _c(topk_idx, np.int32)
    sidx = _c(send_idx, np.int32)
    po = _c(put_offset, np.int32)
    base = _c(rank_recv_base, np.int64)
    T, k = idx.shape
    bs = T // R
    out = np.empty((T, k), np.int64)
    lib().oracle_dst_rows(R, bs, k, epr, _p(idx, _i32p), _p(sidx, _i32p),
                          _p(po, _i32p), _p(base, _i64p), _p(out, _i64p))
    return out


def quant_row(xrow_bits, dtype):
    """One row's INT8 receive image (uint8, align32(H) + 32 bytes)."""
    xrow = _c(xrow_bits, np.uint16)
    H = xrow.size
    out = np.zeros(row_bytes(H, 1), np.uint8)
    lib().oracle_quant_row(H, dtype, _p(xrow, _u16p), _p(out, _u8p))
    return out


def dispatch(x_bits, topk_idx, send_idx, put_offset, rank_recv_base, R, epr,
             dtype, quant, capacity_rows=None):
    """Stage 3 over all tokens.  Returns (recv uint8 [rows, S], status)."""
    x = _c(x_bits, np.uint16)
    idx = _c(topk_idx, np.int32)
    T, H = x.shape
    k = idx.shape[1]
    bs = T // R
    base = _c(rank_recv_base, np.int64)
    rows = int(base[R]) if capacity_rows is None else int(capacity_rows)
    S = row_bytes(H, quant)
    recv = np.zeros((rows, S), np.uint8)
    st = lib().oracle_dispatch(R, bs, k, epr, H, dtype, int(bool(quant)),
                               _p(x, _u16p), _p(idx, _i32p),
                               _p(_c(send_idx, np.int32), _i32p),
                               _p(_c(put_offset, np.int32), _i32p),
                               _p(base, _i64p), _p(recv, _u8p), rows)
    return recv, st


def dispatch_tokens(x_bits, topk_idx, send_idx, put_offset, rank_recv_base,
                    R, epr, dtype, quant, tokens, images=None, row_ids=None):
    """Stage 3 for the listed tokens only.  Returns (images uint8
    [n, k, S], row_ids int64 [n, k], status).  ``images`` / ``row_ids``:
    optional caller-provided C-contiguous output arrays of those shapes
    (every byte is written)."""
    x = _c(x_bits, np.uint16)
    idx = _c(topk_idx, np.int32)
    T, H = x.shape
    k = idx.shape[1]
    bs = T // R
    toks = _c(tokens, np.int64)
    S = row_bytes(H, quant)
    if images is None:
        images = np.zeros((toks.size, k, S), np.uint8)
    if row_ids is None:
        row_ids = np.zeros((toks.size, k), np.int64)
    assert images.shape == (toks.size, k, S) and images.dtype == np.uint8
    assert row_ids.shape == (toks.size, k) and row_ids.dtype == np.int64
    st = lib().oracle_dispatch_tokens(
        R, bs, k, epr, H, dtype, int(bool(quant)), _p(x, _u16p),
        _p(idx, _i32p), _p(_c(send_idx, np.int32), _i32p),
        _p(_c(put_offset, np.int32), _i32p),
        _p(_c(rank_recv_base, np.int64), _i64p), _p(toks, _i64p), toks.size,
        _p(images, _u8p), _p(row_ids, _i64p))
    return images, row_ids, st


def combine(y_bits, topk_idx, topk_weights, send_idx, put_offset,
            rank_recv_base, R, epr, dtype, tokens=None, out=None):
    """Stage 4.  y uint16 [rows, H]; returns (out uint16 [n, H], status),
    n = T when ``tokens`` is None, else len(tokens).  ``out``: optional
    caller-provided C-contiguous uint16 [n, H] output array."""
    y = _c(y_bits, np.uint16)
    idx = _c(topk_idx, np.int32)
    w = _c(topk_weights, np.float32)
    T, k = idx.shape
    H = y.shape[1]
    bs = T // R
    if tokens is None:
        toks = None
        n = T
    else:
        toks = _c(tokens, np.int64)
        n = toks.size
    if out is None:
        out = np.zeros((n, H), np.uint16)
    assert out.shape == (n, H) and out.dtype == np.uint16
    st = lib().oracle_combine_tokens(
        R, bs, k, epr, H, dtype, _p(y, _u16p), y.shape[0], _p(idx, _i32p),
        _p(w, _f32p), _p(_c(send_idx, np.int32), _i32p),
        _p(_c(put_offset, np.int32), _i32p),
        _p(_c(rank_recv_base, np.int64), _i64p),
        None if toks is None else _p(toks, _i64p), n, _p(out, _u16p))
    return out, st


def combine_quant(yq, topk_idx, topk_weights, send_idx, put_offset,
                  rank_recv_base, R, epr, dtype, H, tokens=None):
    """Combine over INT8 expert outputs (uint8 [rows, align32(H)+32] row
    images).  Returns (out uint16 [n, H], status)."""
    yq = _c(yq, np.uint8)
    idx = _c(topk_idx, np.int32)
    w = _c(topk_weights, np.float32)
    T, k = idx.shape
    bs = T // R
    assert yq.ndim == 2 and yq.shape[1] == row_bytes(H, 1)
    if tokens is None:
        toks, n = None, T
    else:
        toks = _c(tokens, np.int64)
        n = toks.size
    out = np.zeros((n, H), np.uint16)
    st = lib().oracle_combine_quant_tokens(
        R, bs, k, epr, H, dtype, _p(yq, _u8p), yq.shape[0], _p(idx, _i32p),
        _p(w, _f32p), _p(_c(send_idx, np.int32), _i32p),
        _p(_c(put_offset, np.int32), _i32p),
        _p(_c(rank_recv_base, np.int64), _i64p),
        None if toks is None else _p(toks, _i64p), n, _p(out, _u16p))
    return out, st


def token_layout(topk_idx, R, epr):
    """Distinct tokens per (source rank, destination rank) and the token x
    rank membership map.  Returns dict(tokens_per_rank [R,R] int32,
    in_rank [T,R] uint8, status)."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    bs = T // R
    tpr = np.zeros((R, R), np.int32)
    inr = np.zeros((T, R), np.uint8)
    st = lib().oracle_token_layout(R, bs, k, epr, _p(idx, _i32p), _p(tpr, _i32p),
                                   _p(inr, _u8p))
    return dict(tokens_per_rank=tpr, in_rank=inr, status=st)


def exp_f32(x):
    """The oracle's fp32 exp (Cody-Waite reduction + Taylor polynomial)."""
    x = _c(x, np.float32)
    out = np.empty_like(x)
    lib().oracle_exp_f32(_p(x, _f32p), _p(out, _f32p), x.size)
    return out


def swiglu_quant(acc, weight_scale, token_scale, rows=None, exp="cw"):
    """GMM1 epilogue: acc int32 [M, 2I] -> INT8 row images uint8
    [n, align32(I) + 32] (n = M, or len(rows)).  exp="cw": Exp is the
    oracle's fp32 evaluation (exp_f32); exp="libm": Exp is the float
    nearest to e^x (libm's double exp rounded once)."""
    fn = {"cw": "oracle_swiglu_quant_rows", "libm": "oracle_swiglu_quant_rows_libm"}[exp]
    acc = _c(acc, np.int32)
    M, N = acc.shape
    I = N // 2
    ws = _c(weight_scale, np.float32)
    ts = _c(token_scale, np.float32)
    assert ws.size == N and ts.size == M
    if rows is None:
        rr, n = None, M
    else:
        rr = _c(rows, np.int64)
        n = rr.size
    out = np.zeros((n, row_bytes(I, 1)), np.uint8)
    getattr(lib(), fn)(M, I, _p(acc, _i32p), _p(ws, _f32p), _p(ts, _f32p),
                       None if rr is None else _p(rr, _i64p), n, _p(out, _u8p))
    return out


# ---- fused deep MoE (section 4.3: GMM1 -> DeqSwigluQuant -> GMM2 ->
#      DeqCombine), on top of the dispatch above ----------------------------

def group_offsets(rank_recv_base, put_offset, R, epr):
    """First receive row of every expert (int64 [E+1]): expert e's rows
    start at rank_recv_base[e // epr] + put_offset[e*R + 0] (its first
    source rank); the last entry is the total row count."""
    base = _c(rank_recv_base, np.int64)
    po = _c(put_offset, np.int32)
    E = R * epr
    off = np.empty(E + 1, np.int64)
    for e in range(E):
        off[e] = int(base[e // epr]) + int(po[e * R])
    off[E] = int(base[R])
    return off


def grouped_gemm(a, group_off, b, rows=None):
    """c[i][n] = sum_k a[i][k] * b[g][n][k] (int32), g the group of the
    row.  a: int8 codes, uint8/int8 [n, lda] (first K = b.shape[2] bytes
    used); b: int8 [G, N, K].  rows: global row of each a row (None: a
    holds all rows in order)."""
    a = _c(a, np.uint8).view(np.int8)
    b = _c(b, np.int8)
    G, N, K = b.shape
    off = _c(group_off, np.int64)
    assert off.size == G + 1 and a.shape[1] >= K
    n = a.shape[0]
    rr = None if rows is None else _c(rows, np.int64)
    if rr is None:
        assert n == int(off[G])
    else:
        assert rr.size == n
    c = np.zeros((n, N), np.int32)
    st = lib().oracle_grouped_gemm_i8(G, _p(off, _i64p), K, N, _p(a, _i8p),
                                      a.shape[1], _p(b, _i8p),
                                      None if rr is None else _p(rr, _i64p), n,
                                      _p(c, _i32p))
    assert st == 0, "grouped_gemm: invalid row or int32 overflow"
    return c


def deq_combine(acc2, weight_scale, row_scale, topk_idx, topk_weights,
                send_idx, put_offset, rank_recv_base, R, epr, dtype,
                tokens=None):
    """DeqCombine.  acc2 int32 [rows, H] (by receive row, or [n*k, H] in
    (token, k) order with ``tokens``), weight_scale fp32 [E, H], row_scale
    fp32 per acc2 row.  Returns (out uint16 [n, H], status)."""
    acc2 = _c(acc2, np.int32)
    ws = _c(weight_scale, np.float32)
    rs = _c(row_scale, np.float32)
    idx = _c(topk_idx, np.int32)
    w = _c(topk_weights, np.float32)
    T, k = idx.shape
    bs = T // R
    H = acc2.shape[1]
    assert ws.shape == (R * epr, H) and rs.size == acc2.shape[0]
    if tokens is None:
        toks, n = None, T
    else:
        toks = _c(tokens, np.int64)
        n = toks.size
        assert acc2.shape[0] == n * k
    out = np.zeros((n, H), np.uint16)
    st = lib().oracle_deq_combine_tokens(
        R, bs, k, epr, H, dtype, _p(acc2, _i32p), acc2.shape[0], _p(ws, _f32p),
        _p(rs, _f32p), _p(idx, _i32p), _p(w, _f32p),
        _p(_c(send_idx, np.int32), _i32p), _p(_c(put_offset, np.int32), _i32p),
        _p(_c(rank_recv_base, np.int64), _i64p),
        None if toks is None else _p(toks, _i64p), n, _p(out, _u16p))
    return out, st


def row_inv_scale(images, K):
    """The fp32 1/scale stored at byte align32(K) of INT8 row images."""
    im = _c(images, np.uint8)
    ka = (K + 31) // 32 * 32
    return im[:, ka:ka + 4].copy().view(np.float32)[:, 0].copy()


def deep_moe(x_bits, topk_idx, topk_weights, R, epr, dtype, w1, ws1, w2, ws2,
             tokens=None):
    """The fused deep MoE's data path (section 4.3) for all tokens, or for
    the listed ones: dispatch with INT8 quantisation; GMM1 = codes x w1[e]
    (int8 [E, 2I, H]); DeqSwigluQuant with weight_scale ws1[e] and the
    dispatch row's 1/scale as per-token scale; GMM2 = codes x w2[e] (int8
    [E, H, I]); DeqCombine with ws2 [E, H] and the requantised row's
    1/scale.  Returns dict(out uint16 [n, H], acc1, x2, acc2, rows)."""
    idx = _c(topk_idx, np.int32)
    T, k = idx.shape
    H = x_bits.shape[1]
    E, N1, K1 = w1.shape
    I = N1 // 2
    assert K1 == H and w2.shape == (E, H, I) and E == R * epr
    L = layout(idx, R, epr)
    Nn = notify(L["count"], R, T // R, epr)
    off = group_offsets(Nn["rank_recv_base"], Nn["put_offset"], R, epr)
    if tokens is None:
        recv, st = dispatch(x_bits, idx, L["send_idx"], Nn["put_offset"],
                            Nn["rank_recv_base"], R, epr, dtype, True)
        rows = np.arange(int(off[E]), dtype=np.int64)
        a1, r1 = recv, None
    else:
        toks = _c(tokens, np.int64)
        images, row_ids, st = dispatch_tokens(
            x_bits, idx, L["send_idx"], Nn["put_offset"], Nn["rank_recv_base"],
            R, epr, dtype, True, toks)
        rows = row_ids.reshape(-1)
        a1, r1 = images.reshape(rows.size, -1), rows
    assert st == 0
    acc1 = grouped_gemm(a1, off, w1, rows=r1)
    ts1 = row_inv_scale(a1, H)
    grp = np.searchsorted(off, rows, side="right") - 1
    x2 = np.zeros((rows.size, row_bytes(I, 1)), np.uint8)
    for e in np.unique(grp):
        sel = np.nonzero(grp == e)[0]
        x2[sel] = swiglu_quant(acc1[sel], ws1[e], ts1[sel])
    acc2 = grouped_gemm(x2, off, w2, rows=r1)
    out, st2 = deq_combine(acc2, ws2, row_inv_scale(x2, I), idx, topk_weights,
                           L["send_idx"], Nn["put_offset"], Nn["rank_recv_base"],
                           R, epr, dtype, tokens=tokens)
    assert st2 == 0
    return dict(out=out, acc1=acc1, x2=x2, acc2=acc2, rows=rows, group_off=off)
