import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmoe_ep.so")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.lib()  # builds liboracle.so if it is missing
    return oracle


def assert_near_plain_exp(name, codes, inv, ref_images, I):
    """The GMM1 epilogue's INT8 output against the oracle that takes Exp as
    the float nearest to e^x (``swiglu_quant(..., exp="libm")``), written
    independently of any fast exp.

    codes: int64 [n, I] INT8 codes; inv: float32 [n] stored 1/scale;
    ref_images: the oracle's row images.  A fast fp32 exp within 1 ulp of
    the nearest float moves h, max|h| and the scale by a few ulp, so a code
    can change by one step where h * scale lies within ~1e-4 of a rounding
    tie (expected for ~1e-4 of the codes), and 1/scale by a few ulp.  The
    bounds: every code within one step, at most 1e-3 of the codes
    differing, 1/scale within 8 ulp."""
    ia = (I + 31) // 32 * 32
    rq = ref_images[:, :I].view(np.int8).astype(np.int64)
    rinv = ref_images[:, ia:ia + 4].copy().view(np.int32)[:, 0].astype(np.int64)
    d = np.abs(np.asarray(codes, np.int64).reshape(rq.shape) - rq)
    assert d.max(initial=0) <= 1, "%s: a code off by %d" % (name, d.max())
    frac = float((d != 0).mean()) if d.size else 0.0
    assert frac <= 1e-3, "%s: %.2e of the codes differ" % (name, frac)
    gi = np.asarray(inv, np.float32).reshape(-1).view(np.int32).astype(np.int64)
    du = np.abs(gi - rinv)
    assert du.max(initial=0) <= 8, "%s: 1/scale off by %d ulp" % (name, du.max())
