"""Every entry point of the C ABI rejects bad arguments on the host, before any
CUDA call, with MOE_ERR_INVALID_ARG: the argument types are read from the
declarations in include/moe_ep.h, so entry points added later are covered
too.  No GPU is needed (pointers are never dereferenced on the host)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INVALID_ARG = 1


class Shape(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int), ("bs", ctypes.c_int), ("k", ctypes.c_int),
                ("experts_per_rank", ctypes.c_int), ("H", ctypes.c_int),
                ("dtype", ctypes.c_int)]


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    import __graft_entry__
    return ctypes.CDLL(__graft_entry__._load_builder().build())


def declarations():
    """(name, [(ctype kind, parameter name), ...]) of every moe_status function."""
    src = open(os.path.join(ROOT, "include", "moe_ep.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    out = []
    for name, params in re.findall(r"moe_status\s+(moe_\w+)\s*\(([^)]*)\)\s*;", src, re.S):
        args = []
        for p in [p.strip() for p in params.split(",") if p.strip()]:
            pname = re.findall(r"(\w+)\s*$", p)[0]
            if "moe_shape" in p and "*" in p:
                kind = "shape"
            elif "*" in p:
                kind = "ptr"
            elif re.search(r"\b(int64_t|size_t)\b", p):
                kind = "i64"
            elif re.search(r"\bfloat\b", p):
                kind = "f32"
            else:
                kind = "i32"
            args.append((kind, pname))
        out.append((name, args))
    return out


DECLS = declarations()
CTYPE = {"shape": ctypes.POINTER(Shape), "ptr": ctypes.c_void_p, "i64": ctypes.c_int64,
         "i32": ctypes.c_int, "f32": ctypes.c_float}


def _call(lib, name, args, shape, ptr_of, scalar=16):
    fn = getattr(lib, name)
    fn.restype = ctypes.c_int
    fn.argtypes = [CTYPE[kind] for kind, _ in args]
    vals = []
    for kind, pname in args:
        if kind == "shape":
            vals.append(ctypes.byref(shape))
        elif kind == "ptr":
            vals.append(ptr_of(pname))
        elif kind == "f32":
            vals.append(1.0)
        else:
            vals.append(scalar)
    return fn(*vals)


def test_declarations_parsed():
    names = [n for n, _ in DECLS]
    for must in ("moe_dispatch_layout", "moe_notify_dispatch", "moe_dispatch", "moe_combine",
                 "moe_combine_quant", "moe_grouped_gemm_i8", "moe_swiglu_quant"):
        assert must in names
    assert all(any(pn == "dev_status" for _, pn in a) for n, a in DECLS
               if n not in ("moe_codes_to_bf16", "moe_interleave_gate_up",
                            "moe_quant_rows_bf16"))


@pytest.mark.parametrize("name,args", DECLS, ids=[n for n, _ in DECLS])
def test_missing_status_word_rejected(lib, name, args):
    """All pointers plausible (16-byte aligned, never dereferenced on the
    host) except the device status word: rejected before any CUDA call."""
    if not any(pn == "dev_status" for _, pn in args):
        pytest.skip("no device status word in this entry point")
    shape = Shape(2, 16, 2, 2, 64, 0)
    assert _call(lib, name, args, shape,
                 lambda pn: None if pn == "dev_status" else 0x10000) == INVALID_ARG


@pytest.mark.parametrize("name,args", [d for d in DECLS if any(k == "shape" for k, _ in d[1])],
                         ids=[n for n, a in DECLS if any(k == "shape" for k, _ in a)])
def test_bad_shape_rejected(lib, name, args):
    """R = 0 (and, separately, H not a multiple of 8) with every pointer
    plausible: rejected by the shape check."""
    for bad in (Shape(0, 16, 2, 2, 64, 0), Shape(2, 16, 2, 2, 60, 0)):
        assert _call(lib, name, args, bad, lambda pn: 0x10000) == INVALID_ARG


@pytest.mark.parametrize("name,args", DECLS, ids=[n for n, _ in DECLS])
def test_all_null_pointers_rejected(lib, name, args):
    """Every pointer NULL (sizes plausible): rejected before any CUDA call."""
    shape = Shape(2, 16, 2, 2, 64, 0)
    assert _call(lib, name, args, shape, lambda pn: None) == INVALID_ARG
