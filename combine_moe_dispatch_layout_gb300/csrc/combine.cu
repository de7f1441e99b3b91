// combine.cu -- stage 4, combine (UMDK/CAM deep analysis v2, section 2.6
// moe_combine_normal_zb, ReadBufferAndWeightedSum).
//
// Per token the page zeroes an fp32 accumulator, then for each of the k
// experts in order reads the expert's output row from the destination rank
// (shmem_ptr), casts it to fp32, multiplies by the gate weight (Muls) and
// adds (Add), and finally casts back with round-to-nearest-even.  Here one
// CTA owns one token; each thread owns 16-byte chunks of the hidden
// dimension and issues the loads of up to 8 expert rows before doing any
// arithmetic, so every thread keeps 8 x 16 bytes of the gather in flight.
// The arithmetic is exactly the page's: acc = 0; acc = acc + (y * w) with
// one rounding for the multiply and one for the add (__fmul_rn / __fadd_rn;
// the translation unit is also compiled with -fmad=false); k in order.
#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int kBatch = 8;    // expert rows loaded before accumulating
constexpr int kMaxCpt = 8;   // 16-byte chunks per thread (H <= 65536)

template <int DT>
__global__ void __launch_bounds__(1024)
combine_kernel(const uint4* __restrict__ y, int64_t y_rows,
               const int32_t* __restrict__ topk_idx,
               const float* __restrict__ weights,
               const int32_t* __restrict__ send_idx,
               const int32_t* __restrict__ put_offset,
               const int64_t* __restrict__ rank_recv_base, int R, int bs, int k,
               int epr, int H, uint4* __restrict__ out, int32_t* dev_status) {
  __shared__ int64_t s_rows[MOE_EP_MAX_TOPK];
  __shared__ float s_w[MOE_EP_MAX_TOPK];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x;
  const int64_t g = blockIdx.x;
  const int s = static_cast<int>(g / bs);
  const int nch = H / 8;
  const int E = R * epr;

  if (warp == 0) {
    for (int kk = lane; kk < k; kk += 32) {
      const int64_t pair = g * k + kk;
      const int e = __ldg(topk_idx + pair);
      int64_t row = -1;
      if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
        set_status(dev_status, MOE_ERR_EXPERT_ID);
      } else {
        row = __ldg(rank_recv_base + e / epr) +
              __ldg(put_offset + int64_t(e) * R + s) + __ldg(send_idx + pair);
        if (row < 0 || row >= y_rows) {
          set_status(dev_status, MOE_ERR_CAPACITY);
          row = -1;
        }
      }
      s_rows[kk] = row;
      s_w[kk] = __ldg(weights + pair);
    }
  }
  __syncthreads();

#pragma unroll
  for (int i = 0; i < kMaxCpt; ++i) {
    const int c = tid + i * nthreads;
    if (c >= nch) break;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int k0 = 0; k0 < k; k0 += kBatch) {
      uint4 v[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int kk = k0 + b;
        const int64_t row = kk < k ? s_rows[kk] : -1;
        v[b] = row >= 0 ? ld_stream_16(y + row * nch + c) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int kk = k0 + b;
        if (kk < k && s_rows[kk] >= 0) {
          const float w = s_w[kk];
          float f[8];
          unpack8<DT>(v[b], f);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[j] = __fadd_rn(acc[j], __fmul_rn(f[j], w));
        }
      }
    }
    out[g * nch + c] = pack8<DT>(acc);
  }
}

template <int DT>
cudaError_t launch_t(const Shape& s, const void* y, int64_t y_rows,
                     const int32_t* topk_idx, const float* weights,
                     const int32_t* send_idx, const int32_t* put_offset,
                     const int64_t* rank_recv_base, void* out,
                     int32_t* dev_status, cudaStream_t st) {
  const int nch = s.H / 8;
  int threads = std::max(32, std::min(1024, (nch + 31) / 32 * 32));
  while ((nch + threads - 1) / threads > kMaxCpt) threads += 32;
  combine_kernel<DT><<<static_cast<unsigned>(s.T()), threads, 0, st>>>(
      static_cast<const uint4*>(y), y_rows, topk_idx, weights, send_idx,
      put_offset, rank_recv_base, s.R, s.bs, s.k, s.epr, s.H,
      static_cast<uint4*>(out), dev_status);
  return cudaGetLastError();
}

}  // namespace

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
