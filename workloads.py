"""Seeded synthetic workloads for the MoE expert-parallel token pipeline.

This module only draws inputs: routing (``topk_idx``), gating weights
(``topk_weights``), token rows ``x`` and expert outputs ``y``.  It holds none
of the pipeline's arithmetic, so both the CUDA path and the CPU oracle can
take their inputs from it.  Everything is drawn on the host with
``torch.Generator`` (CPU), one generator per input stream, so the same seed
gives the same tensors whatever else is drawn.

The five named workloads are the pipeline's benchmark shapes: a tiny case, a
DeepSeek-V3-shaped case, a Zipf-skewed case, an fp16 case without
quantisation and the 384-rank case (CAM_MAX_RANK_SIZE on the UMDK/CAM page).
No public dataset is involved: the shapes and distributions are the recipe.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

BF16, FP16 = 0, 1
_TORCH_DTYPE = {BF16: torch.bfloat16, FP16: torch.float16}

# Input streams: each has its own generator seeded from (seed, stream).
_S_ROUTE, _S_WEIGHT, _S_X, _S_OUTLIER, _S_Y = range(5)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    R: int                 # logical EP ranks
    epr: int               # experts per rank
    bs: int                # tokens per rank
    H: int                 # hidden size
    k: int                 # top-k
    dtype: int = BF16      # token dtype (BF16 or FP16)
    quant: bool = True     # dynamic INT8 quantisation in dispatch
    x_dist: str = "normal"     # "normal" (x_scale = std) or "uniform" (+-x_scale)
    x_scale: float = 1.0
    outlier_p: float = 0.0     # fraction of x elements multiplied by outlier_mult
    outlier_mult: float = 20.0
    routing: str = "uniform"   # "uniform" (k distinct) or "zipf" (w/o replacement)
    zipf_s: float = 1.2
    weights: str = "softmax"   # "softmax" or "sigmoid" (sigmoid, normalised)
    seed: int = 1234

    @property
    def E(self) -> int:
        return self.R * self.epr

    @property
    def T(self) -> int:
        return self.R * self.bs

    @property
    def P(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five benchmark workloads (seed = 1234 + index).
WORKLOADS = {
    "tiny": Workload("tiny", R=2, epr=4, bs=16, H=128, k=2, seed=1234),
    "dsv3": Workload("dsv3", R=8, epr=32, bs=4096, H=7168, k=8,
                     outlier_p=0.01, seed=1235),
    "skew": Workload("skew", R=16, epr=4, bs=2048, H=4096, k=6, x_scale=2.0,
                     routing="zipf", weights="sigmoid", seed=1236),
    "fp16": Workload("fp16", R=32, epr=4, bs=1024, H=2048, k=8, dtype=FP16,
                     quant=False, x_dist="uniform", x_scale=4.0, seed=1237),
    "maxrank": Workload("maxrank", R=384, epr=2, bs=128, H=7168, k=8,
                        seed=1238),
}
ORDER = ["tiny", "dsv3", "skew", "fp16", "maxrank"]


def _gen(seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 16 + stream)
    return g


def routing(w: Workload):
    """topk_idx int32 [T, k] and topk_weights float32 [T, k] (CPU tensors).

    uniform: each token picks k distinct experts uniformly at random, in a
    random order.  zipf: expert e has weight (e+1)^-s and the k experts are
    drawn one after another without replacement.
    """
    T, E, k = w.T, w.E, w.k
    g = _gen(w.seed, _S_ROUTE)
    if T == 0:
        idx = torch.zeros((0, k), dtype=torch.int64)
    elif w.routing == "uniform":
        # k largest of E iid uniform keys = a uniform k-subset in random order
        idx = torch.rand((T, E), generator=g).topk(k, dim=1).indices
    elif w.routing == "zipf":
        p = (torch.arange(E, dtype=torch.float64) + 1.0) ** (-w.zipf_s)
        p = (p / p.sum()).to(torch.float32)
        idx = torch.multinomial(p.expand(T, E).contiguous(), k,
                                replacement=False, generator=g)
    else:
        raise ValueError(w.routing)
    gw = _gen(w.seed, _S_WEIGHT)
    z = torch.randn((T, k), generator=gw, dtype=torch.float32)
    if w.weights == "softmax":
        wt = torch.softmax(z, dim=1)
    elif w.weights == "sigmoid":
        sg = torch.sigmoid(z)
        wt = sg / sg.sum(dim=1, keepdim=True)
    else:
        raise ValueError(w.weights)
    return idx.to(torch.int32).contiguous(), wt.to(torch.float32).contiguous()


def _rows(n_rows: int, H: int, dtype: int, dist: str, scale: float,
          g: torch.Generator, outlier_p: float = 0.0, outlier_mult: float = 1.0,
          g_out: Optional[torch.Generator] = None,
          chunk_elems: int = 1 << 26) -> torch.Tensor:
    out = torch.empty((n_rows, H), dtype=_TORCH_DTYPE[dtype])
    rows_per_chunk = max(1, chunk_elems // max(H, 1))
    for r0 in range(0, n_rows, rows_per_chunk):
        r1 = min(n_rows, r0 + rows_per_chunk)
        if dist == "normal":
            v = torch.randn((r1 - r0, H), generator=g) * scale
        elif dist == "uniform":
            v = (torch.rand((r1 - r0, H), generator=g) * 2.0 - 1.0) * scale
        else:
            raise ValueError(dist)
        if outlier_p > 0.0:
            m = torch.rand((r1 - r0, H), generator=g_out) < outlier_p
            v = torch.where(m, v * outlier_mult, v)
        out[r0:r1] = v.to(out.dtype)  # round to nearest even
    return out


def tokens(w: Workload) -> torch.Tensor:
    """x [T, H] in the workload's dtype (CPU tensor)."""
    return _rows(w.T, w.H, w.dtype, w.x_dist, w.x_scale, _gen(w.seed, _S_X),
                 w.outlier_p, w.outlier_mult, _gen(w.seed, _S_OUTLIER))


def expert_outputs(w: Workload, rows: Optional[int] = None) -> torch.Tensor:
    """Synthetic expert outputs y [rows, H] ~ N(0,1) in the token dtype.

    ``rows`` defaults to T*k, the number of receive rows when every expert id
    is valid.  They stand for the grouped expert GEMM's output, which sits in
    the same row positions as the dispatched rows.
    """
    n = w.P if rows is None else rows
    return _rows(n, w.H, w.dtype, "normal", 1.0, _gen(w.seed, _S_Y))


def expert_outputs_device(w: Workload, device, rows: Optional[int] = None,
                          chunk_elems: int = 1 << 28) -> torch.Tensor:
    """Expert outputs y [rows, H] ~ N(0,1) in the token dtype, drawn on
    ``device`` with that device's generator (seeded like the host stream;
    the values differ from expert_outputs', the distribution does not).
    For benchmarks, where drawing billions of host normals would dominate
    start-up."""
    n = w.P if rows is None else rows
    g = torch.Generator(device=device)
    g.manual_seed(w.seed * 16 + _S_Y)
    out = torch.empty((n, w.H), dtype=_TORCH_DTYPE[w.dtype], device=device)
    rows_per_chunk = max(1, chunk_elems // max(w.H, 1))
    for r0 in range(0, n, rows_per_chunk):
        r1 = min(n, r0 + rows_per_chunk)
        out[r0:r1] = torch.randn((r1 - r0, w.H), generator=g, device=device).to(out.dtype)
    return out


def expert_outputs_int8(w: Workload, rows: Optional[int] = None) -> torch.Tensor:
    """Synthetic INT8 expert outputs: rows laid out like a dispatched INT8
    row (H int8 codes, zeros to align32(H), fp32 1/scale, zeros to
    align32(H) + 32 bytes).  Codes are uniform in [-127, 127]; 1/scale is
    amax/127 with amax = 0.1 + 3|N(0,1)|.  uint8 tensor [rows, row_bytes]."""
    n = w.P if rows is None else rows
    g = _gen(w.seed, _S_Y)
    h_align = (w.H + 31) // 32 * 32
    img = torch.zeros((n, h_align + 32), dtype=torch.uint8)
    codes = torch.randint(-127, 128, (n, w.H), generator=g, dtype=torch.int16)
    img[:, :w.H] = codes.to(torch.int8).view(torch.uint8)
    amax = 0.1 + 3.0 * torch.randn((n,), generator=g).abs()
    inv = (amax / 127.0).to(torch.float32)
    img[:, h_align:h_align + 4] = inv.view(torch.uint8).view(n, 4)
    return img


def gmm1_accumulators(M: int, I: int, seed: int = 99):
    """Synthetic grouped-GEMM outputs for the GMM1 epilogue: int32 acc
    [M, 2I] ~ round(N(0,1) * 2^17) with every 37th column x64 + 1 (beyond
    2^24, so the int-to-float cast rounds), per-column weight scales
    U(0.5, 1.5) * 4e-4 and per-row token scales U(0.005, 0.03)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 16 + 7)
    acc = torch.empty((M, 2 * I), dtype=torch.int32)
    rows_per_chunk = max(1, (1 << 24) // max(1, 2 * I))
    for r0 in range(0, M, rows_per_chunk):
        r1 = min(M, r0 + rows_per_chunk)
        v = torch.round(torch.randn((r1 - r0, 2 * I), generator=g) * 2.0 ** 17)
        v[:, ::37] = v[:, ::37] * 64 + 1
        acc[r0:r1] = v.to(torch.int32)
    ws = (torch.rand((2 * I,), generator=g) + 0.5) * 4e-4
    ts = torch.rand((M,), generator=g) * 0.025 + 0.005
    return acc, ws.to(torch.float32), ts.to(torch.float32)


def moe_weights(E: int, H: int, I: int, seed: int = 7, device="cpu"):
    """Synthetic INT8 expert weights for the fused deep MoE: w1 int8
    [E, 2I, H] (rows 0..I-1 gate, I..2I-1 up; row n = output column n),
    w2 int8 [E, H, I], codes uniform in [-127, 127] (standard deviation
    ~73.6); per-output-column weight scales ws1 [E, 2I] = U(0.5, 1.5) /
    (73.6 sqrt(H)) and ws2 [E, H] = U(0.5, 1.5) / (73.6 sqrt(I)) (fp32), so
    that a unit-variance input gives gate / up / output values of order one
    whatever the sizes.  Drawn with a generator on ``device`` (CPU and CUDA
    streams differ)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed * 16 + 8)
    w1 = torch.randint(-127, 128, (E, 2 * I, H), generator=g, dtype=torch.int8,
                       device=device)
    w2 = torch.randint(-127, 128, (E, H, I), generator=g, dtype=torch.int8,
                       device=device)
    ws1 = (torch.rand((E, 2 * I), generator=g, device=device) + 0.5) / (73.6 * H ** 0.5)
    ws2 = (torch.rand((E, H), generator=g, device=device) + 0.5) / (73.6 * I ** 0.5)
    return w1, ws1.float(), w2, ws2.float()


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a bf16/fp16 CPU tensor (no copy)."""
    assert t.dtype in (torch.bfloat16, torch.float16)
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def torch_dtype(dtype: int) -> torch.dtype:
    return _TORCH_DTYPE[dtype]
