"""Python binding of ``libmoe_ep.so`` (the C ABI in ``include/moe_ep.h``).

Argument marshalling only: every stage runs in the library's sm_103a
kernels.  Tensors must be CUDA tensors of the stated dtype, contiguous, on
the current device; they are passed to the C ABI as raw device pointers
with the current (or given) torch stream.  There is no CPU fallback: if the
shared library has not been built, importing this package raises.

Stages (UMDK/CAM deep analysis v2, section 2 "EP Normal"):
``moe_dispatch_layout`` (2.3), ``moe_notify_dispatch`` (2.4),
``moe_dispatch`` (2.5, optional INT8 quantisation), ``moe_combine`` (2.6).
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_ep.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_EXPERT_ID = 2
MOE_ERR_CAPACITY = 3
MOE_ERR_TIMEOUT = 4
MOE_ERR_CUDA = 5
MOE_ERR_WORKSPACE = 6
MOE_BF16 = 0
MOE_FP16 = 1

_DTYPE = {torch.bfloat16: MOE_BF16, torch.float16: MOE_FP16}


class moe_shape(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int32), ("bs", ctypes.c_int32),
                ("k", ctypes.c_int32), ("experts_per_rank", ctypes.c_int32),
                ("H", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class MoeError(RuntimeError):
    def __init__(self, status, what):
        super().__init__("%s: %s (status %d)" % (what, status_string(status),
                                                 status))
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            "libmoe_ep.so is not built (%s); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first"
            % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    sp = ctypes.POINTER(moe_shape)
    L.moe_status_string.argtypes = [ctypes.c_int]
    L.moe_status_string.restype = ctypes.c_char_p
    L.moe_recv_row_bytes.argtypes = [sp, ctypes.c_int]
    L.moe_recv_row_bytes.restype = i64
    L.moe_layout_workspace_bytes.argtypes = [sp]
    L.moe_layout_workspace_bytes.restype = ctypes.c_size_t
    L.moe_dispatch_layout.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_dispatch_layout_static.argtypes = [sp, vp, vp, vp, vp, vp, vp]
    L.moe_notify_dispatch.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_dispatch.argtypes = [sp, vp, vp, vp, vp, vp, ctypes.c_int, vp, i64,
                               vp, vp]
    L.moe_combine.argtypes = [sp, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_combine_quant.argtypes = [sp, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_token_layout.argtypes = [sp, vp, vp, vp, vp, vp]
    L.moe_swiglu_quant.argtypes = [vp, i64, ctypes.c_int32, vp, vp, vp, vp, vp]
    L.moe_fused_workspace_bytes.argtypes = [sp]
    L.moe_fused_workspace_bytes.restype = ctypes.c_size_t
    L.moe_dispatch_fused.argtypes = [sp, vp, vp, ctypes.c_int] + [vp] * 9 + [i64, vp, vp, vp]
    L.moe_group_offsets.argtypes = [vp, ctypes.c_int32, vp, vp, vp]
    L.moe_codes_to_bf16.argtypes = [vp, i64, i64, ctypes.c_int32, vp, vp]
    L.moe_gmm_block_n.argtypes = []
    L.moe_gmm_block_n.restype = ctypes.c_int32
    L.moe_grouped_gemm_i8.argtypes = [vp, i64, ctypes.c_int32, vp, ctypes.c_int32,
                                      ctypes.c_int32, vp, vp, vp, vp]
    L.moe_swiglu_quant_grouped.argtypes = [vp, i64, ctypes.c_int32, vp, vp,
                                           ctypes.c_int32, vp, i64, vp, vp, vp]
    L.moe_deq_combine.argtypes = [sp, vp, i64, vp, vp, i64, vp, vp, vp, vp, vp,
                                  vp, vp, vp]
    L.moe_grouped_gemm_i8_dequant.argtypes = [vp, i64, ctypes.c_int32, vp, ctypes.c_int32,
                                              ctypes.c_int32, vp, vp, vp, i64, vp, vp, vp]
    L.moe_combine_f32.argtypes = [sp, vp, i64, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_dispatch_expand.argtypes = [sp, vp, vp, vp, vp, vp, vp, vp, i64, vp, vp]
    L.moe_grouped_gemm_i8_swiglu.argtypes = [vp, i64, ctypes.c_int32, vp, ctypes.c_int32,
                                             ctypes.c_int32, vp, vp, vp, i64, vp, vp, vp]
    L.moe_interleave_gate_up.argtypes = [vp, vp, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, vp, vp, vp]
    L.moe_quant_rows_bf16.argtypes = [vp, i64, ctypes.c_int32, vp, ctypes.c_int32, vp, vp,
                                      vp]
    L.moe_swiglu_quant_grouped_bf16.argtypes = [vp, i64, ctypes.c_int32, vp, vp,
                                                ctypes.c_int32, vp, i64, vp, vp, vp, vp]
    for name in ("moe_dispatch_layout", "moe_notify_dispatch", "moe_dispatch",
                 "moe_combine", "moe_combine_quant", "moe_token_layout",
                 "moe_dispatch_fused", "moe_swiglu_quant", "moe_group_offsets",
                 "moe_codes_to_bf16", "moe_grouped_gemm_i8",
                 "moe_swiglu_quant_grouped", "moe_deq_combine",
                 "moe_grouped_gemm_i8_dequant", "moe_combine_f32",
                 "moe_dispatch_expand", "moe_swiglu_quant_grouped_bf16",
                 "moe_grouped_gemm_i8_swiglu", "moe_interleave_gate_up",
                 "moe_quant_rows_bf16", "moe_dispatch_layout_static"):
        getattr(L, name).restype = ctypes.c_int
    return L


_lib = _load()


def lib():
    """The loaded ``ctypes.CDLL`` of libmoe_ep.so."""
    return _lib


def make_shape(R, bs, k, experts_per_rank, H, dtype=MOE_BF16):
    if isinstance(dtype, torch.dtype):
        dtype = _DTYPE[dtype]
    return moe_shape(int(R), int(bs), int(k), int(experts_per_rank), int(H),
                     int(dtype))


def status_string(status):
    return _lib.moe_status_string(int(status)).decode()


def recv_row_bytes(shape, quant):
    return int(_lib.moe_recv_row_bytes(ctypes.byref(shape), int(bool(quant))))


def layout_workspace_bytes(shape):
    return int(_lib.moe_layout_workspace_bytes(ctypes.byref(shape)))


def _ptr(t, dtype=None, numel=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype not in (
            dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError("%s must have dtype %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if numel is not None and t.numel() < numel:
        raise ValueError("%s holds %d elements, needs %d" % (name, t.numel(),
                                                             numel))
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status, what):
    if status != MOE_OK:
        raise MoeError(status, what)
    return status


def moe_dispatch_layout(shape, topk_idx, count, rank_send, send_idx,
                        workspace, dev_status, stream=None):
    """Stage 1: counts per (source rank, expert), per (source, destination)
    rank, and the stable send index of every (token, k) pair."""
    R, E = shape.R, shape.R * shape.experts_per_rank
    P = shape.R * shape.bs * shape.k
    st = _lib.moe_dispatch_layout(
        ctypes.byref(shape), _ptr(topk_idx, torch.int32, P, "topk_idx"),
        _ptr(count, torch.int32, R * E, "count"),
        _ptr(rank_send, torch.int32, R * R, "rank_send"),
        _ptr(send_idx, torch.int32, P, "send_idx"),
        _ptr(workspace, None, None, "workspace"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_dispatch_layout")


def moe_dispatch_layout_static(shape, topk_idx, count, rank_send, send_idx,
                               dev_status, stream=None):
    """Stage 1 without a caller workspace: the library's own scratch array
    (for callers that cannot allocate device memory); calls that overlap on
    the GPU must be serialised by the caller."""
    R, E = shape.R, shape.R * shape.experts_per_rank
    P = shape.R * shape.bs * shape.k
    st = _lib.moe_dispatch_layout_static(
        ctypes.byref(shape), _ptr(topk_idx, torch.int32, P, "topk_idx"),
        _ptr(count, torch.int32, R * E, "count"),
        _ptr(rank_send, torch.int32, R * R, "rank_send"),
        _ptr(send_idx, torch.int32, P, "send_idx"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_dispatch_layout_static")


def moe_notify_dispatch(shape, count, put_offset, total_recv, rank_recv_base,
                        recv_per_expert, max_bs, dev_status, stream=None):
    """Stage 2: putOffset (exclusive prefix per destination rank), receive
    totals, partition bases, rows per expert and maxBs."""
    R, E = shape.R, shape.R * shape.experts_per_rank
    st = _lib.moe_notify_dispatch(
        ctypes.byref(shape), _ptr(count, torch.int32, R * E, "count"),
        _ptr(put_offset, torch.int32, E * R, "put_offset"),
        _ptr(total_recv, torch.int32, R, "total_recv"),
        _ptr(rank_recv_base, torch.int64, R + 1, "rank_recv_base"),
        _ptr(recv_per_expert, torch.int32, E, "recv_per_expert"),
        _ptr(max_bs, torch.int32, 1, "max_bs"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_notify_dispatch")


def moe_dispatch(shape, x, topk_idx, send_idx, put_offset, rank_recv_base,
                 quant, recv, recv_capacity_rows, dev_status, stream=None):
    """Stage 3: scatter token rows (optionally INT8-quantised) into the
    expert-grouped receive buffer."""
    R, E = shape.R, shape.R * shape.experts_per_rank
    T, P = shape.R * shape.bs, shape.R * shape.bs * shape.k
    rb = recv_row_bytes(shape, quant)
    if recv is not None and recv.numel() * recv.element_size() < \
            rb * int(recv_capacity_rows):
        raise ValueError("recv is smaller than recv_capacity_rows rows")
    st = _lib.moe_dispatch(
        ctypes.byref(shape),
        _ptr(x, (torch.bfloat16, torch.float16), T * shape.H, "x"),
        _ptr(topk_idx, torch.int32, P, "topk_idx"),
        _ptr(send_idx, torch.int32, P, "send_idx"),
        _ptr(put_offset, torch.int32, E * R, "put_offset"),
        _ptr(rank_recv_base, torch.int64, R + 1, "rank_recv_base"),
        int(bool(quant)),
        _ptr(recv, None, None, "recv"), int(recv_capacity_rows),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_dispatch")


def moe_combine(shape, expert_out, expert_out_rows, topk_idx, topk_weights,
                send_idx, put_offset, rank_recv_base, out, dev_status,
                stream=None):
    """Stage 4: per token, the fp32 weighted sum of its k expert outputs,
    rounded to the token dtype."""
    R, E = shape.R, shape.R * shape.experts_per_rank
    T, P = shape.R * shape.bs, shape.R * shape.bs * shape.k
    st = _lib.moe_combine(
        ctypes.byref(shape),
        _ptr(expert_out, (torch.bfloat16, torch.float16),
             int(expert_out_rows) * shape.H, "expert_out"),
        int(expert_out_rows),
        _ptr(topk_idx, torch.int32, P, "topk_idx"),
        _ptr(topk_weights, torch.float32, P, "topk_weights"),
        _ptr(send_idx, torch.int32, P, "send_idx"),
        _ptr(put_offset, torch.int32, E * R, "put_offset"),
        _ptr(rank_recv_base, torch.int64, R + 1, "rank_recv_base"),
        _ptr(out, (torch.bfloat16, torch.float16), T * shape.H, "out"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_combine")


def moe_combine_quant(shape, expert_out_q, expert_out_rows, topk_idx,
                      topk_weights, send_idx, put_offset, rank_recv_base, out,
                      dev_status, stream=None):
    """Stage 4 over INT8 expert outputs (row images with 1/scale):
    dequantise, then the same weighted sum as moe_combine."""
    R, E = shape.R, shape.R * shape.experts_per_rank
    T, P = shape.R * shape.bs, shape.R * shape.bs * shape.k
    rb = recv_row_bytes(shape, True)
    if expert_out_q is not None and \
            expert_out_q.numel() * expert_out_q.element_size() < rb * int(expert_out_rows):
        raise ValueError("expert_out_q is smaller than expert_out_rows rows")
    st = _lib.moe_combine_quant(
        ctypes.byref(shape), _ptr(expert_out_q, None, None, "expert_out_q"),
        int(expert_out_rows),
        _ptr(topk_idx, torch.int32, P, "topk_idx"),
        _ptr(topk_weights, torch.float32, P, "topk_weights"),
        _ptr(send_idx, torch.int32, P, "send_idx"),
        _ptr(put_offset, torch.int32, E * R, "put_offset"),
        _ptr(rank_recv_base, torch.int64, R + 1, "rank_recv_base"),
        _ptr(out, (torch.bfloat16, torch.float16), T * shape.H, "out"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_combine_quant")


def moe_token_layout(shape, topk_idx, tokens_per_rank, in_rank, dev_status,
                     stream=None):
    """Distinct tokens per (source rank, destination rank) and the token x
    rank membership map (uint8 [T, R])."""
    R, T = shape.R, shape.R * shape.bs
    P = T * shape.k
    st = _lib.moe_token_layout(
        ctypes.byref(shape), _ptr(topk_idx, torch.int32, P, "topk_idx"),
        _ptr(tokens_per_rank, torch.int32, R * R, "tokens_per_rank"),
        _ptr(in_rank, torch.uint8, T * R, "in_rank"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_token_layout")


def fused_workspace_bytes(shape):
    return int(_lib.moe_fused_workspace_bytes(ctypes.byref(shape)))


def moe_dispatch_fused(shape, x, topk_idx, quant, count, rank_send, send_idx,
                       put_offset, total_recv, rank_recv_base, recv_per_expert,
                       max_bs, recv, recv_capacity_rows, workspace, dev_status,
                       stream=None):
    """Low-latency dispatch: layout + notify + dispatch in one launch, same
    results as the three separate calls."""
    R, E = shape.R, shape.R * shape.experts_per_rank
    T, P = shape.R * shape.bs, shape.R * shape.bs * shape.k
    rb = recv_row_bytes(shape, quant)
    if recv is not None and recv.numel() * recv.element_size() < \
            rb * int(recv_capacity_rows):
        raise ValueError("recv is smaller than recv_capacity_rows rows")
    st = _lib.moe_dispatch_fused(
        ctypes.byref(shape),
        _ptr(x, (torch.bfloat16, torch.float16), T * shape.H, "x"),
        _ptr(topk_idx, torch.int32, P, "topk_idx"), int(bool(quant)),
        _ptr(count, torch.int32, R * E, "count"),
        _ptr(rank_send, torch.int32, R * R, "rank_send"),
        _ptr(send_idx, torch.int32, P, "send_idx"),
        _ptr(put_offset, torch.int32, E * R, "put_offset"),
        _ptr(total_recv, torch.int32, R, "total_recv"),
        _ptr(rank_recv_base, torch.int64, R + 1, "rank_recv_base"),
        _ptr(recv_per_expert, torch.int32, E, "recv_per_expert"),
        _ptr(max_bs, torch.int32, 1, "max_bs"),
        _ptr(recv, None, None, "recv"), int(recv_capacity_rows),
        _ptr(workspace, None, None, "workspace"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_dispatch_fused")


def moe_swiglu_quant(acc, weight_scale, token_scale, out, dev_status,
                     stream=None):
    """GMM1 epilogue: int32 acc [M, 2I] -> INT8 row images out
    [M, align32(I) + 32] (dequant, SwiGLU, dynamic requant)."""
    if acc.dim() != 2 or acc.shape[1] % 2:
        raise ValueError("acc must be [M, 2I]")
    M, I = acc.shape[0], acc.shape[1] // 2
    rb = (I + 31) // 32 * 32 + 32
    if out.numel() * out.element_size() < M * rb:
        raise ValueError("out is smaller than M rows")
    st = _lib.moe_swiglu_quant(
        _ptr(acc, torch.int32, M * 2 * I, "acc"), int(M), int(I),
        _ptr(weight_scale, torch.float32, 2 * I, "weight_scale"),
        _ptr(token_scale, torch.float32, M, "token_scale"),
        _ptr(out, None, None, "out"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_swiglu_quant")


# ---- fused deep MoE ---------------------------------------------------------

def _strided(src, rows, name):
    """(tensor, byte_offset, byte_stride) -> pointer to the fp32 at
    offset + r * stride for r < rows, checked against the tensor's bytes."""
    t, off, stride = src
    if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous():
        raise TypeError("%s must be a contiguous CUDA tensor" % name)
    nbytes = t.numel() * t.element_size()
    if off < 0 or stride < 4 or (rows > 0 and off + (rows - 1) * stride + 4 > nbytes):
        raise ValueError("%s: rows reach past the tensor" % name)
    return ctypes.c_void_p(t.data_ptr() + int(off)), int(stride)


def gmm_block_n():
    """Output-column tile of moe_grouped_gemm_i8."""
    return int(_lib.moe_gmm_block_n())


def moe_group_offsets(group_rows, group_off, dev_status, stream=None):
    """group_off int64 [G+1] = exclusive prefix of group_rows int32 [G]."""
    G = group_rows.numel()
    st = _lib.moe_group_offsets(
        _ptr(group_rows, torch.int32, G, "group_rows"), int(G),
        _ptr(group_off, torch.int64, G + 1, "group_off"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_group_offsets")


def moe_codes_to_bf16(codes, rows, row_stride, K, out, stream=None):
    """INT8 codes at byte 0 of rows ``row_stride`` bytes apart -> bf16
    out [rows, K] (exact)."""
    if codes.numel() * codes.element_size() < rows * row_stride:
        raise ValueError("codes is smaller than rows x row_stride bytes")
    st = _lib.moe_codes_to_bf16(
        _ptr(codes, (torch.uint8, torch.int8), None, "codes"), int(rows),
        int(row_stride), int(K), _ptr(out, torch.bfloat16, rows * K, "out"),
        _stream(stream))
    return _check(st, "moe_codes_to_bf16")


def moe_grouped_gemm_i8(a, w, group_rows, c, dev_status, stream=None):
    """c [a_rows, N] int32 = per-group a [a_rows, K] x w[g] [N, K]^T on the
    tensor cores (int8 values held as bf16; exact)."""
    if a.dim() != 2 or w.dim() != 3 or w.shape[2] != a.shape[1]:
        raise ValueError("a must be [rows, K] and w [G, N, K]")
    rows, K = a.shape
    G, N = w.shape[0], w.shape[1]
    if group_rows.numel() != G:
        raise ValueError("group_rows must have G entries")
    if rows == 0:
        return MOE_OK
    st = _lib.moe_grouped_gemm_i8(
        _ptr(a, torch.bfloat16, rows * K, "a"), int(rows), int(K),
        _ptr(w, torch.bfloat16, G * N * K, "w"), int(G), int(N),
        _ptr(group_rows, torch.int32, G, "group_rows"),
        _ptr(c, torch.int32, rows * N, "c"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_grouped_gemm_i8")


def moe_swiglu_quant_grouped(acc, weight_scale, group_off, token_scale, out,
                             dev_status, stream=None):
    """GMM1 epilogue with per-expert weight scales [G, 2I]; token_scale is
    (tensor, byte_offset, byte_stride) of each row's fp32 scale."""
    if acc.dim() != 2 or acc.shape[1] % 2 or weight_scale.dim() != 2:
        raise ValueError("acc must be [M, 2I] and weight_scale [G, 2I]")
    M, I = acc.shape[0], acc.shape[1] // 2
    G = weight_scale.shape[0]
    if weight_scale.shape[1] != 2 * I or group_off.numel() != G + 1:
        raise ValueError("weight_scale / group_off do not match acc")
    rb = (I + 31) // 32 * 32 + 32
    if out.numel() * out.element_size() < M * rb:
        raise ValueError("out is smaller than M rows")
    tp, tstride = _strided(token_scale, M, "token_scale")
    st = _lib.moe_swiglu_quant_grouped(
        _ptr(acc, torch.int32, M * 2 * I, "acc"), int(M), int(I),
        _ptr(weight_scale, torch.float32, G * 2 * I, "weight_scale"),
        _ptr(group_off, torch.int64, G + 1, "group_off"), int(G), tp, tstride,
        _ptr(out, None, None, "out"), _ptr(dev_status, torch.int32, 1, "dev_status"),
        _stream(stream))
    return _check(st, "moe_swiglu_quant_grouped")


def moe_deq_combine(shape, expert_acc, weight_scale, row_scale, topk_idx,
                    topk_weights, send_idx, put_offset, rank_recv_base, out,
                    dev_status, stream=None):
    """DeqCombine over int32 expert outputs [rows, H]; row_scale is
    (tensor, byte_offset, byte_stride) of each row's fp32 scale."""
    T, k, H = shape.R * shape.bs, shape.k, shape.H
    E = shape.R * shape.experts_per_rank
    rows = expert_acc.shape[0]
    rp, rstride = _strided(row_scale, rows, "row_scale")
    st = _lib.moe_deq_combine(
        ctypes.byref(shape), _ptr(expert_acc, torch.int32, rows * H, "expert_acc"),
        int(rows), _ptr(weight_scale, torch.float32, E * H, "weight_scale"), rp,
        rstride, _ptr(topk_idx, torch.int32, T * k, "topk_idx"),
        _ptr(topk_weights, torch.float32, T * k, "topk_weights"),
        _ptr(send_idx, torch.int32, T * k, "send_idx"),
        _ptr(put_offset, torch.int32, E * shape.R, "put_offset"),
        _ptr(rank_recv_base, torch.int64, shape.R + 1, "rank_recv_base"),
        _ptr(out, None, T * H, "out"), _ptr(dev_status, torch.int32, 1, "dev_status"),
        _stream(stream))
    return _check(st, "moe_deq_combine")


def moe_grouped_gemm_i8_dequant(a, w, group_rows, col_scale, row_scale, y, dev_status,
                                stream=None):
    """y [a_rows, N] fp32 = (fp32(a x w[g]^T) * col_scale[g]) * row scale;
    row_scale is (tensor, byte_offset, byte_stride)."""
    if a.dim() != 2 or w.dim() != 3 or w.shape[2] != a.shape[1]:
        raise ValueError("a must be [rows, K] and w [G, N, K]")
    rows, K = a.shape
    G, N = w.shape[0], w.shape[1]
    if group_rows.numel() != G:
        raise ValueError("group_rows must have G entries")
    if rows == 0:
        return MOE_OK
    rp, rstride = _strided(row_scale, rows, "row_scale")
    st = _lib.moe_grouped_gemm_i8_dequant(
        _ptr(a, torch.bfloat16, rows * K, "a"), int(rows), int(K),
        _ptr(w, torch.bfloat16, G * N * K, "w"), int(G), int(N),
        _ptr(group_rows, torch.int32, G, "group_rows"),
        _ptr(col_scale, torch.float32, G * N, "col_scale"), rp, rstride,
        _ptr(y, torch.float32, rows * N, "y"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_grouped_gemm_i8_dequant")


def moe_combine_f32(shape, expert_out, topk_idx, topk_weights, send_idx, put_offset,
                    rank_recv_base, out, dev_status, stream=None):
    """Combine over fp32 expert outputs [rows, H]."""
    T, k, H = shape.R * shape.bs, shape.k, shape.H
    E = shape.R * shape.experts_per_rank
    rows = expert_out.shape[0]
    st = _lib.moe_combine_f32(
        ctypes.byref(shape), _ptr(expert_out, torch.float32, rows * H, "expert_out"),
        int(rows), _ptr(topk_idx, torch.int32, T * k, "topk_idx"),
        _ptr(topk_weights, torch.float32, T * k, "topk_weights"),
        _ptr(send_idx, torch.int32, T * k, "send_idx"),
        _ptr(put_offset, torch.int32, E * shape.R, "put_offset"),
        _ptr(rank_recv_base, torch.int64, shape.R + 1, "rank_recv_base"),
        _ptr(out, None, T * H, "out"), _ptr(dev_status, torch.int32, 1, "dev_status"),
        _stream(stream))
    return _check(st, "moe_combine_f32")


def moe_dispatch_expand(shape, x, topk_idx, send_idx, put_offset, rank_recv_base,
                        expand_x, dynamic_scale, capacity_rows, dev_status, stream=None):
    """Dispatch with INT8 quantisation into bf16-valued codes expand_x
    [capacity_rows, H] and a packed fp32 1/scale per row."""
    T, k, H = shape.R * shape.bs, shape.k, shape.H
    E = shape.R * shape.experts_per_rank
    st = _lib.moe_dispatch_expand(
        ctypes.byref(shape), _ptr(x, None, T * H, "x"),
        _ptr(topk_idx, torch.int32, T * k, "topk_idx"),
        _ptr(send_idx, torch.int32, T * k, "send_idx"),
        _ptr(put_offset, torch.int32, E * shape.R, "put_offset"),
        _ptr(rank_recv_base, torch.int64, shape.R + 1, "rank_recv_base"),
        _ptr(expand_x, torch.bfloat16, capacity_rows * H, "expand_x"),
        _ptr(dynamic_scale, torch.float32, capacity_rows, "dynamic_scale"),
        int(capacity_rows), _ptr(dev_status, torch.int32, 1, "dev_status"),
        _stream(stream))
    return _check(st, "moe_dispatch_expand")


def moe_swiglu_quant_grouped_bf16(acc, weight_scale, group_off, token_scale, codes,
                                  inv_scale, dev_status, stream=None):
    """Grouped GMM1 epilogue writing bf16-valued codes [M, I] and a packed
    fp32 1/scale per row; token_scale is (tensor, byte_offset, byte_stride)."""
    if acc.dim() != 2 or acc.shape[1] % 2 or weight_scale.dim() != 2:
        raise ValueError("acc must be [M, 2I] and weight_scale [G, 2I]")
    M, I = acc.shape[0], acc.shape[1] // 2
    G = weight_scale.shape[0]
    if weight_scale.shape[1] != 2 * I or group_off.numel() != G + 1:
        raise ValueError("weight_scale / group_off do not match acc")
    tp, tstride = _strided(token_scale, M, "token_scale")
    st = _lib.moe_swiglu_quant_grouped_bf16(
        _ptr(acc, torch.int32, M * 2 * I, "acc"), int(M), int(I),
        _ptr(weight_scale, torch.float32, G * 2 * I, "weight_scale"),
        _ptr(group_off, torch.int64, G + 1, "group_off"), int(G), tp, tstride,
        _ptr(codes, torch.bfloat16, M * I, "codes"),
        _ptr(inv_scale, torch.float32, M, "inv_scale"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_swiglu_quant_grouped_bf16")


def moe_interleave_gate_up(w1, ws1, w1_interleaved, ws1_interleaved, stream=None):
    """w1 int8 [G, 2I, K] -> bf16 with gate/up rows interleaved; ws1 likewise."""
    G, N1, K = w1.shape
    I = N1 // 2
    st = _lib.moe_interleave_gate_up(
        _ptr(w1, (torch.int8, torch.uint8), G * N1 * K, "w1"),
        _ptr(ws1, torch.float32, G * N1, "ws1"), int(G), int(I), int(K),
        _ptr(w1_interleaved, torch.bfloat16, G * N1 * K, "w1_interleaved"),
        _ptr(ws1_interleaved, torch.float32, G * N1, "ws1_interleaved"), _stream(stream))
    return _check(st, "moe_interleave_gate_up")


def moe_grouped_gemm_i8_swiglu(a, w_interleaved, group_rows, col_scale_interleaved,
                               row_scale, h, dev_status, stream=None):
    """h [a_rows, I] fp32 = SwiGLU of the dequantised GMM1 (gate/up
    interleaved weights [G, 2I, K]); row_scale is (tensor, byte_offset,
    byte_stride)."""
    if a.dim() != 2 or w_interleaved.dim() != 3 or w_interleaved.shape[2] != a.shape[1]:
        raise ValueError("a must be [rows, K] and w [G, 2I, K]")
    rows, K = a.shape
    G, N = w_interleaved.shape[0], w_interleaved.shape[1]
    I = N // 2
    if group_rows.numel() != G:
        raise ValueError("group_rows must have G entries")
    if rows == 0:
        return MOE_OK
    rp, rstride = _strided(row_scale, rows, "row_scale")
    st = _lib.moe_grouped_gemm_i8_swiglu(
        _ptr(a, torch.bfloat16, rows * K, "a"), int(rows), int(K),
        _ptr(w_interleaved, torch.bfloat16, G * N * K, "w_interleaved"), int(G), int(I),
        _ptr(group_rows, torch.int32, G, "group_rows"),
        _ptr(col_scale_interleaved, torch.float32, G * N, "col_scale_interleaved"), rp,
        rstride, _ptr(h, torch.float32, rows * I, "h"),
        _ptr(dev_status, torch.int32, 1, "dev_status"), _stream(stream))
    return _check(st, "moe_grouped_gemm_i8_swiglu")


def moe_quant_rows_bf16(h, group_off, codes, inv_scale, stream=None):
    """Requantise fp32 rows h [M, I] into bf16-valued codes and 1/scale."""
    M, I = h.shape
    G = 0 if group_off is None else group_off.numel() - 1
    st = _lib.moe_quant_rows_bf16(
        _ptr(h, torch.float32, M * I, "h"), int(M), int(I),
        None if group_off is None else _ptr(group_off, torch.int64, G + 1, "group_off"),
        int(G), _ptr(codes, torch.bfloat16, M * I, "codes"),
        _ptr(inv_scale, torch.float32, M, "inv_scale"), _stream(stream))
    return _check(st, "moe_quant_rows_bf16")


# the size queries and the status names under the C entry points' own names
moe_status_string = status_string
moe_recv_row_bytes = recv_row_bytes
moe_layout_workspace_bytes = layout_workspace_bytes
moe_fused_workspace_bytes = fused_workspace_bytes
moe_gmm_block_n = gmm_block_n
