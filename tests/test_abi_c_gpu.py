"""The four stages driven from C, the way a C caller uses the library: a
C99 program that includes only moe_ep.h and the CUDA runtime, allocates
every device buffer with cudaMalloc, zero-fills the layout workspace, runs
moe_dispatch_layout -> moe_notify_dispatch -> moe_dispatch -> moe_combine on
a stream of its own, and writes the outputs back to files.  The test
compares them with the CPU oracle bit for bit (integer outputs, INT8 row
images and 1/scale, and the combine, whose fixed operation order makes it
exact)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_DRIVER = r"""
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime_api.h>
#include "moe_ep.h"

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
  fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 10; } } while (0)
#define MK(x) do { moe_status s_ = (x); if (s_ != MOE_OK) { \
  fprintf(stderr, "%s: %s\n", #x, moe_status_string(s_)); return 11; } } while (0)

static char dir[4096];

static int load(const char* name, void* dst, size_t n) {
  char p[4200]; FILE* f; size_t got;
  snprintf(p, sizeof p, "%s/%s", dir, name);
  f = fopen(p, "rb");
  if (!f) return 1;
  got = fread(dst, 1, n, f);
  fclose(f);
  return got != n;
}

static int save(const char* name, const void* src, size_t n) {
  char p[4200]; FILE* f; size_t put;
  snprintf(p, sizeof p, "%s/%s", dir, name);
  f = fopen(p, "wb");
  if (!f) return 1;
  put = fwrite(src, 1, n, f);
  fclose(f);
  return put != n;
}

/* device -> file */
static int fetch(const char* name, const void* dev, size_t n) {
  void* h = malloc(n ? n : 1);
  int rc;
  if (!h) return 1;
  if (cudaMemcpy(h, dev, n, cudaMemcpyDeviceToHost) != cudaSuccess) { free(h); return 1; }
  rc = save(name, h, n);
  free(h);
  return rc;
}

int main(int argc, char** argv) {
  moe_shape s;
  int quant, E, k;
  long long T, P, rows;
  long long row_bytes, es = 2;
  size_t ws_bytes;
  void *h_idx, *h_w, *h_x, *h_y;
  int32_t *d_idx, *d_count, *d_rank_send, *d_send_idx, *d_put, *d_total, *d_rpe, *d_maxbs,
      *d_status;
  int64_t* d_base;
  float* d_w;
  void *d_x, *d_y, *d_recv, *d_out, *d_ws;
  cudaStream_t st;
  if (argc != 9) return 2;
  strncpy(dir, argv[1], sizeof dir - 1);
  s.R = atoi(argv[2]); s.bs = atoi(argv[3]); s.k = atoi(argv[4]);
  s.experts_per_rank = atoi(argv[5]); s.H = atoi(argv[6]);
  s.dtype = atoi(argv[7]) ? MOE_FP16 : MOE_BF16;
  quant = atoi(argv[8]);
  E = s.R * s.experts_per_rank; k = s.k;
  T = (long long)s.R * s.bs; P = T * k; rows = P;
  row_bytes = moe_recv_row_bytes(&s, quant);
  ws_bytes = moe_layout_workspace_bytes(&s);
  if (row_bytes <= 0 || ws_bytes == 0) return 3;

  h_idx = malloc(P * 4); h_w = malloc(P * 4); h_x = malloc(T * s.H * es);
  h_y = malloc(rows * s.H * es);
  if (!h_idx || !h_w || !h_x || !h_y) return 4;
  if (load("topk_idx.bin", h_idx, P * 4) || load("topk_weights.bin", h_w, P * 4) ||
      load("x.bin", h_x, T * s.H * es) || load("y.bin", h_y, rows * s.H * es)) return 5;

  CK(cudaStreamCreate(&st));
  CK(cudaMalloc((void**)&d_idx, P * 4));
  CK(cudaMalloc((void**)&d_w, P * 4));
  CK(cudaMalloc(&d_x, T * s.H * es));
  CK(cudaMalloc(&d_y, rows * s.H * es));
  CK(cudaMalloc((void**)&d_count, (size_t)s.R * E * 4));
  CK(cudaMalloc((void**)&d_rank_send, (size_t)s.R * s.R * 4));
  CK(cudaMalloc((void**)&d_send_idx, P * 4));
  CK(cudaMalloc((void**)&d_put, (size_t)E * s.R * 4));
  CK(cudaMalloc((void**)&d_total, (size_t)s.R * 4));
  CK(cudaMalloc((void**)&d_base, (size_t)(s.R + 1) * 8));
  CK(cudaMalloc((void**)&d_rpe, (size_t)E * 4));
  CK(cudaMalloc((void**)&d_maxbs, 4));
  CK(cudaMalloc((void**)&d_status, 4));
  CK(cudaMalloc(&d_recv, rows * row_bytes));
  CK(cudaMalloc(&d_out, T * s.H * es));
  CK(cudaMalloc(&d_ws, ws_bytes));
  CK(cudaMemsetAsync(d_ws, 0, ws_bytes, st));          /* zero-filled before first use */
  CK(cudaMemsetAsync(d_status, 0, 4, st));
  CK(cudaMemcpyAsync(d_idx, h_idx, P * 4, cudaMemcpyHostToDevice, st));
  CK(cudaMemcpyAsync(d_w, h_w, P * 4, cudaMemcpyHostToDevice, st));
  CK(cudaMemcpyAsync(d_x, h_x, T * s.H * es, cudaMemcpyHostToDevice, st));
  CK(cudaMemcpyAsync(d_y, h_y, rows * s.H * es, cudaMemcpyHostToDevice, st));

  MK(moe_dispatch_layout(&s, d_idx, d_count, d_rank_send, d_send_idx, d_ws, d_status, st));
  MK(moe_notify_dispatch(&s, d_count, d_put, d_total, d_base, d_rpe, d_maxbs, d_status, st));
  MK(moe_dispatch(&s, d_x, d_idx, d_send_idx, d_put, d_base, quant, d_recv, rows, d_status,
                  st));
  MK(moe_combine(&s, d_y, rows, d_idx, d_w, d_send_idx, d_put, d_base, d_out, d_status, st));
  CK(cudaStreamSynchronize(st));

  if (fetch("status.bin", d_status, 4) || fetch("count.bin", d_count, (size_t)s.R * E * 4) ||
      fetch("rank_send.bin", d_rank_send, (size_t)s.R * s.R * 4) ||
      fetch("send_idx.bin", d_send_idx, P * 4) ||
      fetch("put_offset.bin", d_put, (size_t)E * s.R * 4) ||
      fetch("total_recv.bin", d_total, (size_t)s.R * 4) ||
      fetch("rank_recv_base.bin", d_base, (size_t)(s.R + 1) * 8) ||
      fetch("recv_per_expert.bin", d_rpe, (size_t)E * 4) ||
      fetch("max_bs.bin", d_maxbs, 4) || fetch("recv.bin", d_recv, rows * row_bytes) ||
      fetch("out.bin", d_out, T * s.H * es))
    return 6;
  CK(cudaStreamDestroy(st));
  printf("ok\n");
  return 0;
}
"""


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    import __graft_entry__
    so = __graft_entry__._load_builder().build()
    d = tmp_path_factory.mktemp("c_driver")
    src = d / "driver.c"
    src.write_text(C_DRIVER)
    exe = d / "driver"
    cuda = _cuda_home()
    libdirs = [p for p in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                           os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                           os.path.join(cuda, "targets", "x86_64-linux", "lib"))
               if os.path.isdir(p)]
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), "-isystem", os.path.join(cuda, "include"),
           str(src), so, "-Wl,-rpath," + os.path.dirname(so)]
    for p in libdirs:
        cmd += ["-L" + p, "-Wl,-rpath," + p]
    cmd += ["-lcudart", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-3000:]
    return exe


@pytest.mark.parametrize("w", [
    W.Workload("c_ragged", R=3, epr=5, bs=37, H=96, k=4, seed=61),
    W.Workload("c_fp16", R=4, epr=2, bs=50, H=264, k=3, dtype=W.FP16, quant=False,
               x_dist="uniform", x_scale=4.0, seed=62),
], ids=lambda w: w.name)
def test_four_stages_from_c(oracle_mod, driver, tmp_path, w):
    idx, wt = W.routing(w)
    x, y = W.tokens(w), W.expert_outputs(w)
    idx.numpy().tofile(tmp_path / "topk_idx.bin")
    wt.numpy().tofile(tmp_path / "topk_weights.bin")
    W.bits(x).tofile(tmp_path / "x.bin")
    W.bits(y).tofile(tmp_path / "y.bin")
    r = subprocess.run([str(driver), str(tmp_path), str(w.R), str(w.bs), str(w.k),
                        str(w.epr), str(w.H), str(w.dtype), str(int(w.quant))],
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stderr[-2000:])

    def rd(name, dtype, shape):
        return np.fromfile(tmp_path / name, dtype=dtype).reshape(shape)

    assert int(rd("status.bin", np.int32, (1,))[0]) == 0
    L = oracle_mod.layout(idx.numpy(), w.R, w.epr)
    N = oracle_mod.notify(L["count"], w.R, w.bs, w.epr)
    np.testing.assert_array_equal(rd("count.bin", np.int32, (w.R, w.E)), L["count"])
    np.testing.assert_array_equal(rd("rank_send.bin", np.int32, (w.R, w.R)), L["rank_send"])
    np.testing.assert_array_equal(rd("send_idx.bin", np.int32, (w.T, w.k)), L["send_idx"])
    np.testing.assert_array_equal(rd("put_offset.bin", np.int32, (w.E * w.R,)),
                                  N["put_offset"])
    np.testing.assert_array_equal(rd("total_recv.bin", np.int32, (w.R,)), N["total_recv"])
    np.testing.assert_array_equal(rd("rank_recv_base.bin", np.int64, (w.R + 1,)),
                                  N["rank_recv_base"])
    np.testing.assert_array_equal(rd("recv_per_expert.bin", np.int32, (w.E,)),
                                  N["recv_per_expert"])
    assert int(rd("max_bs.bin", np.int32, (1,))[0]) == N["max_bs"]
    recv, st = oracle_mod.dispatch(W.bits(x), idx.numpy(), L["send_idx"], N["put_offset"],
                                   N["rank_recv_base"], w.R, w.epr, w.dtype, w.quant)
    assert st == 0
    np.testing.assert_array_equal(rd("recv.bin", np.uint8, recv.shape), recv)
    out, st = oracle_mod.combine(W.bits(y), idx.numpy(), wt.numpy(), L["send_idx"],
                                 N["put_offset"], N["rank_recv_base"], w.R, w.epr, w.dtype)
    assert st == 0
    np.testing.assert_array_equal(rd("out.bin", np.uint16, out.shape), out)
