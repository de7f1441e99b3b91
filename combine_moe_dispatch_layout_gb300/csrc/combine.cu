// combine.cu -- stage 4, combine (UMDK/CAM deep analysis v2, section 2.6
// moe_combine_normal_zb, ReadBufferAndWeightedSum).
//
// Per token the page zeroes an fp32 accumulator, then for each of the k
// experts in order reads the expert's output row from the destination rank
// (shmem_ptr), casts it to fp32, multiplies by the gate weight (Muls) and
// adds (Add), and finally casts back with round-to-nearest-even.
//
// GB300 design: a persistent grid (as many CTAs as fit on the SMs) walks the
// tokens.  The last warp of each CTA is a producer: while the compute warps
// gather token g's k rows, it resolves token g+grid's rows (topk_idx ->
// rank_recv_base / put_offset / send_idx, a chain of dependent loads) and
// weights into the other half of a double-buffered shared table, so the
// gather never waits on index arithmetic.  Each compute thread owns 16-byte
// chunks of the hidden dimension and issues the loads of up to 8 expert
// rows before doing any arithmetic.  The arithmetic is exactly the page's:
// acc = 0; acc = acc + (y * w), one rounding for the multiply and one for
// the add (__fmul_rn / __fadd_rn; the unit is also built with -fmad=false),
// k in order; out = round-to-nearest-even in the token dtype.
//
// combine_quant_kernel is the same gather over INT8 expert outputs (the
// "+ dequant" of the pipeline diagram, section 2.1): each row is a
// dispatched-style INT8 image (codes, fp32 1/scale at align32(H)); the
// producer also fetches each row's 1/scale, and every element is
// dequantised as float(q) * (1/scale) (one rounding) before the same
// multiply-then-add.  Rows are half the bytes of bf16 rows.
#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int kBatch = 8;          // expert rows loaded before accumulating
constexpr int kMaxThreads = 1024;

// Resolve the rows and weights of token g into the shared tables (one warp).
__device__ __forceinline__ void resolve_token(
    int64_t g, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ weights, const int32_t* __restrict__ send_idx,
    const int32_t* __restrict__ put_offset,
    const int64_t* __restrict__ rank_recv_base, int R, int bs, int k, int epr,
    int64_t y_rows, int64_t* rows, float* w, int32_t* dev_status, int lane) {
  const int E = R * epr;
  const int s = static_cast<int>(g / bs);
  for (int kk = lane; kk < k; kk += 32) {
    const int64_t pair = g * k + kk;
    const int e = __ldg(topk_idx + pair);
    const int32_t sidx = __ldg(send_idx + pair);
    const float wt = __ldg(weights + pair);
    int64_t row = -1;
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
      set_status(dev_status, MOE_ERR_EXPERT_ID);
    } else {
      row = __ldg(rank_recv_base + e / epr) + __ldg(put_offset + int64_t(e) * R + s) + sidx;
      if (row < 0 || row >= y_rows) {
        set_status(dev_status, MOE_ERR_CAPACITY);
        row = -1;
      }
    }
    rows[kk] = row;
    w[kk] = wt;
  }
}

template <int DT>
__global__ void __launch_bounds__(kMaxThreads)
combine_kernel(const uint4* __restrict__ y, int64_t y_rows,
               const int32_t* __restrict__ topk_idx,
               const float* __restrict__ weights,
               const int32_t* __restrict__ send_idx,
               const int32_t* __restrict__ put_offset,
               const int64_t* __restrict__ rank_recv_base, int R, int bs, int k,
               int epr, int H, int64_t T, uint4* __restrict__ out,
               int32_t* dev_status) {
  __shared__ int64_t s_rows[2][MOE_EP_MAX_TOPK];
  __shared__ float s_w[2][MOE_EP_MAX_TOPK];
  const int tid = threadIdx.x, lane = tid & 31;
  const int ncomp = blockDim.x - 32;            // compute threads
  const bool producer = tid >= ncomp;           // the last warp
  const int nch = H / 8;

  int64_t g = blockIdx.x;
  if (producer)
    resolve_token(g, topk_idx, weights, send_idx, put_offset, rank_recv_base, R,
                  bs, k, epr, y_rows, s_rows[0], s_w[0], dev_status, lane);
  __syncthreads();

  for (int it = 0; g < T; ++it, g += gridDim.x) {
    const int buf = it & 1;
    if (producer) {
      const int64_t gn = g + gridDim.x;
      if (gn < T)
        resolve_token(gn, topk_idx, weights, send_idx, put_offset, rank_recv_base,
                      R, bs, k, epr, y_rows, s_rows[buf ^ 1], s_w[buf ^ 1],
                      dev_status, lane);
    } else {
      const int64_t* rows = s_rows[buf];
      const float* w = s_w[buf];
      for (int c = tid; c < nch; c += ncomp) {
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        for (int k0 = 0; k0 < k; k0 += kBatch) {
          uint4 v[kBatch];
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int kk = k0 + b;
            const int64_t row = kk < k ? rows[kk] : -1;
            v[b] = row >= 0 ? ld_stream_16(y + row * nch + c) : make_uint4(0u, 0u, 0u, 0u);
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int kk = k0 + b;
            if (kk < k && rows[kk] >= 0) {
              const float wk = w[kk];
              float f[8];
              unpack8<DT>(v[b], f);
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], __fmul_rn(f[j], wk));
            }
          }
        }
        out[g * nch + c] = pack8<DT>(acc);
      }
    }
    __syncthreads();   // this token's table is free, the next one is ready
  }
}

// Compute threads per CTA: about 4 chunks each, a multiple of 32, at most
// 992 (plus the producer warp).
int compute_threads(int nch) {
  int t = ((nch + 3) / 4 + 31) / 32 * 32;
  return std::max(32, std::min(kMaxThreads - 32, t));
}

// ---------------------------------------------------------------------------
// INT8 expert outputs
// ---------------------------------------------------------------------------
constexpr int kQuantMaxThreads = 512;

__device__ __forceinline__ uint2 ld_stream_8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

// The i-th signed byte of a 32-bit word, as float (exact).
__device__ __forceinline__ float code_f(uint32_t w, int i) {
  return static_cast<float>(static_cast<int32_t>(w << (24 - 8 * i)) >> 24);
}

template <int DT>
__global__ void __launch_bounds__(kQuantMaxThreads)
combine_quant_kernel(const unsigned char* __restrict__ yq, int64_t y_rows,
                     int64_t row_bytes, const int32_t* __restrict__ topk_idx,
                     const float* __restrict__ weights,
                     const int32_t* __restrict__ send_idx,
                     const int32_t* __restrict__ put_offset,
                     const int64_t* __restrict__ rank_recv_base, int R, int bs,
                     int k, int epr, int H, int64_t T, uint4* __restrict__ out,
                     int32_t* dev_status) {
  __shared__ int64_t s_rows[2][MOE_EP_MAX_TOPK];
  __shared__ float s_w[2][MOE_EP_MAX_TOPK];
  __shared__ float s_inv[2][MOE_EP_MAX_TOPK];
  const int tid = threadIdx.x, lane = tid & 31;
  const int ncomp = blockDim.x - 32;
  const bool producer = tid >= ncomp;
  const int nq = (H + 15) / 16;                 // 16-code chunks (last may be 8)
  const int64_t h_align = align_up(H, 32);
  const int nch8 = H / 8;                       // uint4 outputs per row

  auto resolve = [&](int64_t gt, int b) {
    resolve_token(gt, topk_idx, weights, send_idx, put_offset, rank_recv_base, R, bs,
                  k, epr, y_rows, s_rows[b], s_w[b], dev_status, lane);
    __syncwarp();
    for (int kk = lane; kk < k; kk += 32) {
      const int64_t row = s_rows[b][kk];
      s_inv[b][kk] = row >= 0 ? __ldg(reinterpret_cast<const float*>(
                                    yq + row * row_bytes + h_align))
                              : 0.0f;
    }
  };

  int64_t g = blockIdx.x;
  if (producer) resolve(g, 0);
  __syncthreads();

  for (int it = 0; g < T; ++it, g += gridDim.x) {
    const int buf = it & 1;
    if (producer) {
      __syncwarp();
      const int64_t gn = g + gridDim.x;
      if (gn < T) resolve(gn, buf ^ 1);
    } else {
      const int64_t* rows = s_rows[buf];
      const float* w = s_w[buf];
      const float* inv = s_inv[buf];
      for (int c = tid; c < nq; c += ncomp) {
        const bool half = 16 * c + 8 >= H;      // only 8 codes left
        float acc[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
        for (int k0 = 0; k0 < k; k0 += kBatch) {
          uint4 v[kBatch];
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int kk = k0 + b;
            const int64_t row = kk < k ? rows[kk] : -1;
            v[b] = make_uint4(0u, 0u, 0u, 0u);
            if (row >= 0) {
              const unsigned char* src = yq + row * row_bytes + 16 * c;
              if (half) {
                const uint2 h2 = ld_stream_8(src);
                v[b].x = h2.x;
                v[b].y = h2.y;
              } else {
                v[b] = ld_stream_16(src);
              }
            }
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int kk = k0 + b;
            if (kk < k && rows[kk] >= 0) {
              const float wk = w[kk], sk = inv[kk];
              const uint32_t wd[4] = {v[b].x, v[b].y, v[b].z, v[b].w};
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float t = __fmul_rn(code_f(wd[j >> 2], j & 3), sk);   // dequantise
                acc[j] = __fadd_rn(acc[j], __fmul_rn(t, wk));              // Muls, Add
              }
            }
          }
        }
        float lo[8], hi[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          lo[j] = acc[j];
          hi[j] = acc[8 + j];
        }
        out[g * nch8 + 2 * c] = pack8<DT>(lo);
        if (!half) out[g * nch8 + 2 * c + 1] = pack8<DT>(hi);
      }
    }
    __syncthreads();
  }
}

template <int DT>
cudaError_t launch_quant_t(const Shape& s, const void* yq, int64_t y_rows,
                           const int32_t* topk_idx, const float* weights,
                           const int32_t* send_idx, const int32_t* put_offset,
                           const int64_t* rank_recv_base, void* out,
                           int32_t* dev_status, cudaStream_t st) {
  const int nq = (s.H + 15) / 16;
  const int ncomp = std::max(32, std::min(kQuantMaxThreads - 32, ((nq + 3) / 4 + 31) / 32 * 32));
  const int threads = ncomp + 32;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_quant_kernel<DT>, threads, 0);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(s.T(), int64_t(std::max(1, per_sm)) * sms);
  combine_quant_kernel<DT><<<static_cast<unsigned>(grid), threads, 0, st>>>(
      static_cast<const unsigned char*>(yq), y_rows, align_up(s.H, 32) + 32, topk_idx,
      weights, send_idx, put_offset, rank_recv_base, s.R, s.bs, s.k, s.epr, s.H, s.T(),
      static_cast<uint4*>(out), dev_status);
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_t(const Shape& s, const void* y, int64_t y_rows,
                     const int32_t* topk_idx, const float* weights,
                     const int32_t* send_idx, const int32_t* put_offset,
                     const int64_t* rank_recv_base, void* out,
                     int32_t* dev_status, cudaStream_t st) {
  const int nch = s.H / 8;
  const int threads = compute_threads(nch) + 32;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<DT>, threads, 0);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(s.T(), int64_t(std::max(1, per_sm)) * sms);
  combine_kernel<DT><<<static_cast<unsigned>(grid), threads, 0, st>>>(
      static_cast<const uint4*>(y), y_rows, topk_idx, weights, send_idx,
      put_offset, rank_recv_base, s.R, s.bs, s.k, s.epr, s.H, s.T(),
      static_cast<uint4*>(out), dev_status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine_quant(const Shape& s, const void* yq, int64_t y_rows,
                                 const int32_t* topk_idx, const float* weights,
                                 const int32_t* send_idx, const int32_t* put_offset,
                                 const int64_t* rank_recv_base, void* out,
                                 int32_t* dev_status, cudaStream_t st) {
  if (s.T() == 0) return cudaSuccess;
  if (s.dtype == MOE_BF16)
    return launch_quant_t<MOE_BF16>(s, yq, y_rows, topk_idx, weights, send_idx,
                                    put_offset, rank_recv_base, out, dev_status, st);
  return launch_quant_t<MOE_FP16>(s, yq, y_rows, topk_idx, weights, send_idx,
                                  put_offset, rank_recv_base, out, dev_status, st);
}

cudaError_t launch_combine(const Shape& s, const void* y, int64_t y_rows,
                           const int32_t* topk_idx, const float* weights,
                           const int32_t* send_idx, const int32_t* put_offset,
                           const int64_t* rank_recv_base, void* out,
                           int32_t* dev_status, cudaStream_t st) {
  if (s.T() == 0) return cudaSuccess;
  if (s.dtype == MOE_BF16)
    return launch_t<MOE_BF16>(s, y, y_rows, topk_idx, weights, send_idx,
                              put_offset, rank_recv_base, out, dev_status, st);
  return launch_t<MOE_FP16>(s, y, y_rows, topk_idx, weights, send_idx,
                            put_offset, rank_recv_base, out, dev_status, st);
}

}  // namespace moe_ep
