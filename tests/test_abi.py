"""The C ABI without a GPU: the library builds and loads, exports every
function ``include/*.h`` declares, and rejects bad arguments on the host
(before any CUDA call) with MOE_ERR_INVALID_ARG."""
import ctypes
import glob
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists(
            "/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    import __graft_entry__
    path = __graft_entry__._load_builder().build()
    return ctypes.CDLL(path)


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        src = re.sub(r"#[^\n]*", "", src)
        names.update(re.findall(r"\b(moe_\w+)\s*\(", src))
    return sorted(names)


def test_header_declares_the_four_stages():
    names = declared_functions()
    for n in ("moe_dispatch_layout", "moe_notify_dispatch", "moe_dispatch",
              "moe_combine", "moe_combine_quant", "moe_token_layout",
              "moe_dispatch_fused", "moe_fused_workspace_bytes",
              "moe_swiglu_quant",
              "moe_status_string",
              "moe_recv_row_bytes", "moe_layout_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, "not exported: %s" % missing


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("R", "bs", "k", "experts_per_rank", "H", "dtype")]


def _setup(lib):
    lib.moe_recv_row_bytes.restype = ctypes.c_int64
    lib.moe_recv_row_bytes.argtypes = [ctypes.POINTER(Shape), ctypes.c_int]
    lib.moe_layout_workspace_bytes.restype = ctypes.c_size_t
    lib.moe_status_string.restype = ctypes.c_char_p
    lib.moe_dispatch.argtypes = [ctypes.POINTER(Shape)] + [ctypes.c_void_p] * 5 \
        + [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
           ctypes.c_void_p]
    lib.moe_combine.argtypes = [ctypes.POINTER(Shape), ctypes.c_void_p,
                                ctypes.c_int64] + [ctypes.c_void_p] * 8


def test_row_bytes_and_workspace(lib):
    _setup(lib)
    s = Shape(8, 4096, 8, 32, 7168, 0)
    assert lib.moe_recv_row_bytes(ctypes.byref(s), 1) == 7168 + 32
    assert lib.moe_recv_row_bytes(ctypes.byref(s), 0) == 7168 * 2
    s2 = Shape(2, 4, 2, 2, 40, 0)
    assert lib.moe_recv_row_bytes(ctypes.byref(s2), 1) == 64 + 32
    assert lib.moe_layout_workspace_bytes(ctypes.byref(s)) > 0
    bad = Shape(0, 4, 2, 2, 40, 0)
    assert lib.moe_recv_row_bytes(ctypes.byref(bad), 1) == -1
    assert lib.moe_layout_workspace_bytes(ctypes.byref(bad)) == 0


BAD_SHAPES = [
    (0, 4, 2, 2, 64, 0),        # R < 1
    (385, 4, 2, 2, 64, 0),      # R > 384
    (2, 4, 2, 0, 64, 0),        # epr < 1
    (8, 4, 2, 513, 64, 0),      # E > 4096
    (2, 4, 0, 2, 64, 0),        # k < 1
    (2, 4, 5, 2, 64, 0),        # k > E
    (64, 4, 65, 2, 64, 0),      # k > 64
    (2, -1, 2, 2, 64, 0),       # bs < 0
    (2, 4, 2, 2, 60, 0),        # H % 8 != 0
    (2, 4, 2, 2, 0, 0),         # H < 8
    (2, 4, 2, 2, 65544, 0),     # H > 65536
    (2, 4, 2, 2, 64, 2),        # unknown dtype
    (384, 1 << 20, 8, 2, 64, 0),  # T*k >= 2^31
]


@pytest.mark.parametrize("shape", BAD_SHAPES)
def test_invalid_shapes_rejected_on_host(lib, shape):
    _setup(lib)
    s = Shape(*shape)
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: rejected first
    assert lib.moe_dispatch_layout(ctypes.byref(s), fake, fake, fake, fake,
                                   fake, fake, None) == 1
    assert lib.moe_notify_dispatch(ctypes.byref(s), fake, fake, fake, fake,
                                   fake, fake, fake, None) == 1
    assert lib.moe_dispatch(ctypes.byref(s), fake, fake, fake, fake, fake, 1,
                            fake, 10, fake, None) == 1
    assert lib.moe_combine(ctypes.byref(s), fake, 10, fake, fake, fake, fake,
                           fake, fake, fake, None) == 1


def test_null_and_misaligned_pointers_rejected(lib):
    _setup(lib)
    s = Shape(2, 4, 2, 2, 64, 0)
    ok = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)    # 8-byte aligned, not 16
    assert lib.moe_dispatch_layout(ctypes.byref(s), None, ok, ok, ok, ok, ok,
                                   None) == 1
    assert lib.moe_dispatch_layout(ctypes.byref(s), ok, ok, ok, ok, odd, ok,
                                   None) == 1        # workspace needs 16 B
    assert lib.moe_notify_dispatch(ctypes.byref(s), ok, ok, ok,
                                   ctypes.c_void_p(0x10004), ok, ok, ok,
                                   None) == 1        # int64 base needs 8 B
    assert lib.moe_dispatch(ctypes.byref(s), odd, ok, ok, ok, ok, 1, ok, 16,
                            ok, None) == 1           # x needs 16 B
    assert lib.moe_dispatch(ctypes.byref(s), ok, ok, ok, ok, ok, 1, odd, 16,
                            ok, None) == 1           # recv needs 16 B
    assert lib.moe_dispatch(ctypes.byref(s), ok, ok, ok, ok, ok, 1, ok, -1,
                            ok, None) == 1           # negative capacity
    assert lib.moe_combine(ctypes.byref(s), ok, 16, ok, ok, ok, ok, ok, odd,
                           ok, None) == 1            # out needs 16 B
    assert lib.moe_combine(ctypes.byref(s), ok, 16, ok, ok, ok, ok, ok, ok,
                           None, None) == 1          # dev_status required


def test_status_strings(lib):
    _setup(lib)
    assert lib.moe_status_string(0) == b"ok"
    assert b"expert" in lib.moe_status_string(2)
    assert lib.moe_status_string(99) == b"unknown status"


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "moe_ep.h"

typedef void (*any_fn)(void);
/* every declared entry point, so the declarations are type-checked */
static any_fn all_entry_points[] = { %s };

int main(void) {
  moe_shape s;
  int32_t dummy = 0;
  s.R = 8; s.bs = 16; s.k = 8; s.experts_per_rank = 32; s.H = 7168; s.dtype = MOE_BF16;
  if (moe_recv_row_bytes(&s, 1) != 7168 + 32) return 1;
  if (moe_recv_row_bytes(&s, 0) != 2 * 7168) return 2;
  if (moe_layout_workspace_bytes(&s) == 0) return 3;
  if (strcmp(moe_status_string(MOE_OK), "ok") != 0) return 4;
  /* host-side checks only: nothing here reaches the GPU */
  if (moe_dispatch(&s, NULL, NULL, NULL, NULL, NULL, 1, NULL, 0, &dummy, NULL)
      != MOE_ERR_INVALID_ARG) return 5;
  s.H = 60;
  if (moe_recv_row_bytes(&s, 1) != -1) return 6;
  printf("%%d entry points\n", (int)(sizeof all_entry_points / sizeof all_entry_points[0]));
  return 0;
}
"""


@pytest.mark.parametrize("compiler,std", [("gcc", "-std=c99"), ("g++", "-std=c++17")])
def test_header_is_plain_c_and_links(lib, tmp_path, compiler, std):
    """The header compiles as strict C99 (and as C++) with warnings as errors,
    and a C program linked to libmoe_ep.so calls the host-side entry points."""
    if shutil.which(compiler) is None:
        pytest.skip(compiler + " not available")
    import __graft_entry__
    so = __graft_entry__._load_builder().build()
    names = declared_functions()
    src = tmp_path / ("abi.c" if compiler == "gcc" else "abi.cpp")
    src.write_text(C_PROGRAM % ", ".join("(any_fn)%s" % n for n in names))
    exe = tmp_path / "abi"
    import subprocess
    r = subprocess.run([compiler, std, "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", os.path.join(ROOT, "include"), str(src), so,
                        "-Wl,-rpath," + os.path.dirname(so), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr[-2000:])
    assert r.stdout.strip() == "%d entry points" % len(names)


def test_python_binding_mirrors_the_header(lib):
    """Every declared entry point has a Python function of the same name, and
    the marshalling of the layout wrappers reaches the C side, which rejects
    an invalid shape before any CUDA call (no GPU needed)."""
    import combine_moe_dispatch_layout_gb300 as ep
    missing = [n for n in declared_functions() if not callable(getattr(ep, n, None))]
    assert not missing, missing

    class HostStream:          # a stream handle the C side never uses here
        cuda_stream = 0

    bad = ep.make_shape(0, 16, 2, 2, 64)
    for call in (lambda: ep.moe_dispatch_layout(bad, None, None, None, None, None, None,
                                                HostStream()),
                 lambda: ep.moe_dispatch_layout_static(bad, None, None, None, None, None,
                                                       HostStream())):
        with pytest.raises(ep.MoeError) as err:
            call()
        assert err.value.status == ep.MOE_ERR_INVALID_ARG
    good = ep.make_shape(8, 16, 8, 32, 7168)
    assert ep.moe_recv_row_bytes(good, 1) == 7200 and ep.moe_recv_row_bytes(good, 0) == 14336
    assert ep.moe_layout_workspace_bytes(good) == ep.layout_workspace_bytes(good)
    assert ep.moe_status_string(ep.MOE_ERR_CAPACITY) == "row outside the receive buffer"
    assert ep.moe_gmm_block_n() > 0 and ep.moe_fused_workspace_bytes(good) > 0
