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
               moe_combine, moe_combine_quant, moe_dispatch,
               moe_dispatch_fused, moe_dispatch_layout, moe_notify_dispatch,
               recv_row_bytes)


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
