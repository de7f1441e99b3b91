"""Device buffers for one EP pipeline problem and the four calls in order.

Plumbing above the binding: ``PipelineBuffers`` allocates (with torch) every
output and scratch buffer the four stages need for one shape, and
``run_pipeline`` enqueues dispatch layout -> notify -> dispatch -> combine on
one stream.  The receive buffer is sized for the worst case, T*k rows, which
is also the exact row count when every expert id is valid, so no host
synchronisation is needed between the stages.
"""
import torch

from . import (fused_workspace_bytes, make_shape, layout_workspace_bytes,
               moe_codes_to_bf16, moe_combine, moe_combine_f32, moe_combine_quant,
               moe_dispatch, moe_dispatch_expand, moe_dispatch_fused,
               moe_dispatch_layout, moe_group_offsets, moe_grouped_gemm_i8,
               moe_grouped_gemm_i8_dequant, moe_grouped_gemm_i8_swiglu,
               moe_interleave_gate_up, moe_notify_dispatch, moe_quant_rows_bf16,
               moe_swiglu_quant_grouped_bf16, recv_row_bytes)


class PipelineBuffers:
    def __init__(self, R, bs, k, epr, H, dtype, quant, device="cuda"):
        self.shape = make_shape(R, bs, k, epr, H, dtype)
        self.quant = bool(quant)
        self.torch_dtype = dtype if isinstance(dtype, torch.dtype) else (
            torch.bfloat16 if dtype == 0 else torch.float16)
        E, T, P = R * epr, R * bs, R * bs * k
        i32 = dict(dtype=torch.int32, device=device)
        self.count = torch.empty((R, E), **i32)
        self.rank_send = torch.empty((R, R), **i32)
        self.send_idx = torch.empty((T, k), **i32)
        # zero-filled once; the layout kernel leaves it reusable
        self.workspace = torch.zeros(max(16, layout_workspace_bytes(self.shape)),
                                     dtype=torch.uint8, device=device)
        self.put_offset = torch.empty((E * R,), **i32)
        self.total_recv = torch.empty((R,), **i32)
        self.rank_recv_base = torch.empty((R + 1,), dtype=torch.int64,
                                          device=device)
        self.recv_per_expert = torch.empty((E,), **i32)
        self.max_bs = torch.empty((1,), **i32)
        self.dev_status = torch.zeros((1,), **i32)
        self.row_bytes = recv_row_bytes(self.shape, quant)
        self.capacity = P
        self.recv = torch.empty((P, self.row_bytes), dtype=torch.uint8,
                                device=device)
        self.out = torch.empty((T, H), dtype=self.torch_dtype, device=device)
        self.device = device
        self._fused_ws = None

    @property
    def fused_workspace(self):
        """Workspace of the one-launch dispatch (allocated zeroed on first
        use)."""
        if self._fused_ws is None:
            self._fused_ws = torch.zeros(
                max(16, fused_workspace_bytes(self.shape)), dtype=torch.uint8,
                device=self.device)
        return self._fused_ws

    def status(self):
        """First device-side error code of the calls so far (syncs)."""
        return int(self.dev_status.item())


def run_layout_notify(b, topk_idx, stream=None):
    moe_dispatch_layout(b.shape, topk_idx, b.count, b.rank_send, b.send_idx,
                        b.workspace, b.dev_status, stream)
    moe_notify_dispatch(b.shape, b.count, b.put_offset, b.total_recv,
                        b.rank_recv_base, b.recv_per_expert, b.max_bs,
                        b.dev_status, stream)


def run_dispatch(b, x, topk_idx, stream=None):
    moe_dispatch(b.shape, x, topk_idx, b.send_idx, b.put_offset,
                 b.rank_recv_base, b.quant, b.recv, b.capacity, b.dev_status,
                 stream)


def run_combine(b, y, topk_idx, topk_weights, stream=None):
    moe_combine(b.shape, y, y.shape[0], topk_idx, topk_weights, b.send_idx,
                b.put_offset, b.rank_recv_base, b.out, b.dev_status, stream)


def run_dispatch_fused(b, x, topk_idx, stream=None):
    """Layout + notify + dispatch in one launch (the low-latency path)."""
    moe_dispatch_fused(b.shape, x, topk_idx, b.quant, b.count, b.rank_send,
                       b.send_idx, b.put_offset, b.total_recv,
                       b.rank_recv_base, b.recv_per_expert, b.max_bs, b.recv,
                       b.capacity, b.fused_workspace, b.dev_status, stream)


def run_combine_quant(b, yq, topk_idx, topk_weights, stream=None):
    """Combine over INT8 expert outputs (row images, 1/scale per row)."""
    moe_combine_quant(b.shape, yq, yq.shape[0], topk_idx, topk_weights,
                      b.send_idx, b.put_offset, b.rank_recv_base, b.out,
                      b.dev_status, stream)


def run_pipeline(b, x, topk_idx, topk_weights, y, stream=None):
    """All four stages on one stream; results stay in ``b``."""
    run_layout_notify(b, topk_idx, stream)
    run_dispatch(b, x, topk_idx, stream)
    run_combine(b, y, topk_idx, topk_weights, stream)


# ---- fused deep MoE: dispatch -> GMM1 -> DeqSwigluQuant -> GMM2 -> DeqCombine

def _align32(n):
    return (n + 31) // 32 * 32


class DeepMoeWeights:
    """Expert weights for the deep MoE: INT8 codes converted once to bf16
    (exact) for the tensor-core GEMMs, plus fp32 per-column scales.
    w1 int8 [E, 2I, H], ws1 [E, 2I], w2 int8 [E, H, I], ws2 [E, H]."""

    def __init__(self, w1, ws1, w2, ws2, stream=None, plain=True, interleaved=True):
        E, N1, H = w1.shape
        I = N1 // 2
        assert w2.shape == (E, H, I)
        self.E, self.H, self.I = E, H, I
        dev = w1.device
        self.ws1 = ws1.contiguous()
        self.ws2 = ws2.contiguous()
        # plain copy for GMM1 with int32 output (the standalone epilogue)
        self.w1 = self.w1i = self.ws1i = None
        if plain:
            self.w1 = torch.empty((E, N1, H), dtype=torch.bfloat16, device=dev)
            moe_codes_to_bf16(w1, E * N1, H, H, self.w1, stream)
        # gate/up interleaved copy for GMM1 with the SwiGLU epilogue
        if interleaved:
            self.w1i = torch.empty((E, N1, H), dtype=torch.bfloat16, device=dev)
            self.ws1i = torch.empty((E, N1), dtype=torch.float32, device=dev)
            moe_interleave_gate_up(w1, self.ws1, self.w1i, self.ws1i, stream)
        self.w2 = torch.empty((E, H, I), dtype=torch.bfloat16, device=dev)
        moe_codes_to_bf16(w2, E * H, I, I, self.w2, stream)


class DeepMoeBuffers(PipelineBuffers):
    """PipelineBuffers plus the deep MoE's intermediates, all sized for T*k
    rows: the dispatched codes as bf16 (expand_x) and their 1/scale, GMM1's
    int32 accumulators, the requantised codes as bf16 and their 1/scale,
    GMM2's dequantised fp32 outputs, and the expert row offsets."""

    def __init__(self, R, bs, k, epr, H, I, dtype, device="cuda"):
        super().__init__(R, bs, k, epr, H, dtype, True, device)
        P = R * bs * k
        self.I = I
        f32 = dict(dtype=torch.float32, device=device)
        self.group_off = torch.empty((R * epr + 1,), dtype=torch.int64, device=device)
        self.a1 = torch.empty((P, H), dtype=torch.bfloat16, device=device)
        self.ts1 = torch.empty((P,), **f32)
        self.acc1 = torch.empty((P, 2 * I), dtype=torch.int32, device=device)
        self.h = torch.empty((P, I), **f32)
        self.a2 = torch.empty((P, I), dtype=torch.bfloat16, device=device)
        self.ts2 = torch.empty((P,), **f32)
        self.y2 = torch.empty((P, H), **f32)


def run_dispatch_expand(b, x, topk_idx, stream=None):
    """Stage 1: INT8 quantisation into bf16-valued codes and packed 1/scale."""
    moe_dispatch_expand(b.shape, x, topk_idx, b.send_idx, b.put_offset, b.rank_recv_base,
                        b.a1, b.ts1, b.capacity, b.dev_status, stream)


def run_deep_moe_experts(b, wts, stream=None, fused_swiglu=False):
    """Stages 2-3 up to the dequantised expert outputs ``b.y2``.  GMM1 to
    int32 + the standalone DeqSwigluQuant kernel (the faster route at the
    DeepSeek-V3 size), or with ``fused_swiglu`` GMM1 with DeqSwiglu in its
    epilogue (fp32 h, half the intermediate bytes) + the requantisation
    pass; then GMM2 with its dequantising epilogue."""
    moe_group_offsets(b.recv_per_expert, b.group_off, b.dev_status, stream)
    if fused_swiglu:
        moe_grouped_gemm_i8_swiglu(b.a1, wts.w1i, b.recv_per_expert, wts.ws1i,
                                   (b.ts1, 0, 4), b.h, b.dev_status, stream)
        moe_quant_rows_bf16(b.h, b.group_off, b.a2, b.ts2, stream)
    else:
        moe_grouped_gemm_i8(b.a1, wts.w1, b.recv_per_expert, b.acc1, b.dev_status, stream)
        moe_swiglu_quant_grouped_bf16(b.acc1, wts.ws1, b.group_off, (b.ts1, 0, 4), b.a2,
                                      b.ts2, b.dev_status, stream)
    moe_grouped_gemm_i8_dequant(b.a2, wts.w2, b.recv_per_expert, wts.ws2, (b.ts2, 0, 4),
                                b.y2, b.dev_status, stream)


def run_deep_combine(b, topk_idx, topk_weights, stream=None):
    """DeqCombine's remaining step: the weighted sum over the fp32 rows."""
    moe_combine_f32(b.shape, b.y2, topk_idx, topk_weights, b.send_idx, b.put_offset,
                    b.rank_recv_base, b.out, b.dev_status, stream)


def run_deep_moe(b, wts, x, topk_idx, topk_weights, stream=None):
    """The whole deep MoE on one stream; the result is ``b.out``."""
    run_layout_notify(b, topk_idx, stream)
    run_dispatch_expand(b, x, topk_idx, stream)
    run_deep_moe_experts(b, wts, stream)
    run_deep_combine(b, topk_idx, topk_weights, stream)
