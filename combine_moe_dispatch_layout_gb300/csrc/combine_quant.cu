// combine_quant.cu -- stage 4 over INT8 expert outputs: the "+ dequant" of
// the pipeline diagram (UMDK/CAM deep analysis v2, section 2.1, stage 4:
// shmem read + weighted sum + dequant) on top of section 2.6's
// ReadBufferAndWeightedSum.
//
// Each expert-output row is a dispatched-style INT8 row image (codes, fp32
// 1/scale at align32(H)).  Same persistent producer/compute structure as
// combine.cu: the producer warp resolves the next token's rows and weights
// and also fetches each row's 1/scale; compute threads load 16 codes per
// 16-byte load (8 rows in flight) and dequantise every element as
// float(q) * (1/scale) (one rounding) before the same multiply-then-add
// (__fmul_rn / __fadd_rn, k in order), then round to the token dtype.
// Rows are half the bytes of bf16 rows.
#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {

namespace {

constexpr int kBatch = 8;          // expert rows loaded before accumulating

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

}  // namespace moe_ep
