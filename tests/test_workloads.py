"""The seeded input generator: shapes, distributions and determinism."""
import numpy as np
import pytest
import torch

import workloads as W


def test_named_workloads_shapes():
    w = W.WORKLOADS["dsv3"]
    assert (w.R, w.E, w.bs, w.T, w.k, w.H, w.P) == (
        8, 256, 4096, 32768, 8, 7168, 262144)
    assert W.WORKLOADS["maxrank"].R == 384 and W.WORKLOADS["maxrank"].E == 768
    assert W.WORKLOADS["fp16"].dtype == W.FP16
    assert not W.WORKLOADS["fp16"].quant
    assert [W.WORKLOADS[n].seed for n in W.ORDER] == [1234 + i for i in range(5)]


@pytest.mark.parametrize("name", ["tiny", "skew"])
def test_routing_distinct_and_weights(name):
    w = W.WORKLOADS[name]
    if name == "skew":
        w = w.with_(bs=64)
    idx, wt = W.routing(w)
    assert idx.dtype == torch.int32 and idx.shape == (w.T, w.k)
    assert int(idx.min()) >= 0 and int(idx.max()) < w.E
    srt = idx.sort(dim=1).values
    assert (srt[:, 1:] != srt[:, :-1]).all()           # k distinct experts
    assert torch.allclose(wt.sum(dim=1), torch.ones(w.T), atol=1e-6)
    assert (wt > 0).all()


def test_zipf_is_skewed():
    w = W.WORKLOADS["skew"].with_(bs=256)
    idx, _ = W.routing(w)
    hist = np.bincount(idx.numpy().reshape(-1), minlength=w.E)
    assert hist[0] > 5 * hist[-1]        # expert 0 is the hottest
    assert hist[0] == hist.max()


def test_determinism_and_stream_independence():
    w = W.WORKLOADS["tiny"]
    a = W.routing(w)
    b = W.routing(w)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    x1 = W.tokens(w)
    x2 = W.tokens(w.with_(k=1))          # routing change leaves x unchanged
    assert torch.equal(x1, x2)
    assert not torch.equal(W.tokens(w.with_(seed=7)), x1)


def test_outliers_and_uniform():
    w = W.WORKLOADS["dsv3"].with_(bs=4, R=2, H=4096)
    x = W.tokens(w).float()
    assert x.dtype == torch.float32 and x.shape == (8, 4096)
    frac_big = (x.abs() > 6).float().mean().item()
    assert 0.002 < frac_big < 0.02                       # ~1% x20 outliers
    u = W.tokens(W.WORKLOADS["fp16"].with_(bs=4, R=2)).float()
    assert u.abs().max() <= 4.0 and u.min() < -3.5 and u.max() > 3.5


def test_chunked_generation_matches_one_shot():
    w = W.WORKLOADS["tiny"].with_(bs=40)
    a = W._rows(w.T, w.H, w.dtype, "normal", 1.0, W._gen(1, 2))
    b = W._rows(w.T, w.H, w.dtype, "normal", 1.0, W._gen(1, 2),
                chunk_elems=w.H * 3)
    assert torch.equal(a, b)
