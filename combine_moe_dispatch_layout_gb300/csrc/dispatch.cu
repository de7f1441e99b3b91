// dispatch.cu -- stage 3, dispatch with optional dynamic INT8 quantisation
// (UMDK/CAM deep analysis v2, section 2.5 moe_dispatch_normal_zb and
// QuantProcess).
//
// The page moves each token row through the vector core's unified buffer
// (MTE DMA in, vector quantise, DMA out to the peer's expandXOut).  Here one
// CTA owns one token: its threads read the row once with 16-byte streaming
// loads straight into registers, reduce max|x| with warp shuffles and one
// shared-memory step, quantise in registers, and store the same image into
// each of the token's k receive rows (k-fold write amplification is the
// stage's inherent HBM cost; the read side is one pass over x).
//
// Quantisation, element by element: f = fp32(x) (exact); amax = max |f|;
// scale = 127 / (amax + 1e-12f) with IEEE add and divide; q = round half to
// even of (f * scale) (one fp32 multiply, then cvt.rni); |q| <= 127, so the
// page's int32 -> int16 -> int8 casts are exact.  1/scale (IEEE divide) goes
// to byte align32(H) of the row, every other byte after the codes is zero.
#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int kMaxCpt = 8;   // 16-byte chunks per thread (registers)

// Destination row of pair (g, kk), -1 when the pair is skipped.
__device__ __forceinline__ int64_t dst_row(
    const int32_t* topk_idx, const int32_t* send_idx, const int32_t* put_offset,
    const int64_t* rank_recv_base, int R, int epr, int s, int64_t pair,
    int64_t capacity, int32_t* dev_status) {
  const int E = R * epr;
  const int e = __ldg(topk_idx + pair);
  if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
    set_status(dev_status, MOE_ERR_EXPERT_ID);
    return -1;
  }
  const int64_t row = __ldg(rank_recv_base + e / epr) +
                      __ldg(put_offset + int64_t(e) * R + s) +
                      __ldg(send_idx + pair);
  if (row < 0 || row >= capacity) {
    set_status(dev_status, MOE_ERR_CAPACITY);
    return -1;
  }
  return row;
}

template <int DT, bool QUANT>
__global__ void __launch_bounds__(1024)
dispatch_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ topk_idx,
                const int32_t* __restrict__ send_idx,
                const int32_t* __restrict__ put_offset,
                const int64_t* __restrict__ rank_recv_base, int R, int bs, int k,
                int epr, int H, unsigned char* __restrict__ recv,
                int64_t row_bytes, int64_t capacity, int32_t* dev_status) {
  __shared__ int64_t s_rows[MOE_EP_MAX_TOPK];
  __shared__ float s_wmax[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x;
  const int64_t g = blockIdx.x;
  const int s = static_cast<int>(g / bs);
  const int nch = H / 8;                        // 16-byte chunks per row

  if (warp == 0) {
    for (int kk = lane; kk < k; kk += 32)
      s_rows[kk] = dst_row(topk_idx, send_idx, put_offset, rank_recv_base, R,
                           epr, s, g * k + kk, capacity, dev_status);
  }

  uint4 v[kMaxCpt];
  const uint4* xrow = x + g * nch;
#pragma unroll
  for (int i = 0; i < kMaxCpt; ++i) {
    const int c = tid + i * nthreads;
    v[i] = c < nch ? ld_stream_16(xrow + c) : make_uint4(0u, 0u, 0u, 0u);
  }

  if constexpr (QUANT) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxCpt; ++i) {
      if (tid + i * nthreads < nch) {
        float f[8];
        unpack8<DT>(v[i], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if (lane == 0) s_wmax[warp] = amax;
    __syncthreads();
    amax = s_wmax[0];
    for (int w = 1; w < nthreads / 32; ++w) amax = fmaxf(amax, s_wmax[w]);
    const float scale = __fdiv_rn(127.0f, __fadd_rn(amax, 1e-12f));
    const float inv = __fdiv_rn(1.0f, scale);

    uint2 q[kMaxCpt];
#pragma unroll
    for (int i = 0; i < kMaxCpt; ++i) {
      float f[8];
      unpack8<DT>(v[i], f);
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int qi = __float2int_rn(__fmul_rn(f[j], scale));
        w[j >> 2] |= (static_cast<uint32_t>(qi) & 0xffu) << (8 * (j & 3));
      }
      q[i] = make_uint2(w[0], w[1]);
    }
    // tail: zero pad to align32(H), fp32 1/scale, zero pad to the row end
    const int h_align = static_cast<int>(align_up(H, 32));
    const int ntail = static_cast<int>((row_bytes - H) / 8);
    const int inv_word = (h_align - H) / 8;
    for (int kk = 0; kk < k; ++kk) {
      const int64_t row = s_rows[kk];
      if (row < 0) continue;
      unsigned char* dst = recv + row * row_bytes;
#pragma unroll
      for (int i = 0; i < kMaxCpt; ++i) {
        const int c = tid + i * nthreads;
        if (c < nch) *reinterpret_cast<uint2*>(dst + int64_t(c) * 8) = q[i];
      }
      if (tid < ntail)
        *reinterpret_cast<uint2*>(dst + H + 8 * tid) =
            make_uint2(tid == inv_word ? __float_as_uint(inv) : 0u, 0u);
    }
  } else {
    __syncthreads();   // s_rows
    for (int kk = 0; kk < k; ++kk) {
      const int64_t row = s_rows[kk];
      if (row < 0) continue;
      uint4* dst = reinterpret_cast<uint4*>(recv + row * row_bytes);
#pragma unroll
      for (int i = 0; i < kMaxCpt; ++i) {
        const int c = tid + i * nthreads;
        if (c < nch) dst[c] = v[i];
      }
    }
  }
}

template <int DT, bool QUANT>
cudaError_t launch_t(const Shape& s, const void* x, const int32_t* topk_idx,
                     const int32_t* send_idx, const int32_t* put_offset,
                     const int64_t* rank_recv_base, void* recv,
                     int64_t row_bytes, int64_t capacity, int32_t* dev_status,
                     cudaStream_t st) {
  const int nch = s.H / 8;
  // about 2 chunks per thread: enough bytes in flight per SM without
  // starving the amax reduction of threads
  int threads = ((nch + 1) / 2 + 31) / 32 * 32;
  threads = std::max(32, std::min(1024, threads));
  while ((nch + threads - 1) / threads > kMaxCpt) threads += 32;   // H large
  dispatch_kernel<DT, QUANT><<<static_cast<unsigned>(s.T()), threads, 0, st>>>(
      static_cast<const uint4*>(x), topk_idx, send_idx, put_offset,
      rank_recv_base, s.R, s.bs, s.k, s.epr, s.H,
      static_cast<unsigned char*>(recv), row_bytes, capacity, dev_status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dispatch(const Shape& s, const void* x,
                            const int32_t* topk_idx, const int32_t* send_idx,
                            const int32_t* put_offset,
                            const int64_t* rank_recv_base, bool quant,
                            void* recv, int64_t row_bytes,
                            int64_t capacity_rows, int32_t* dev_status,
                            cudaStream_t st) {
  if (s.T() == 0) return cudaSuccess;
  if (s.dtype == MOE_BF16)
    return quant ? launch_t<MOE_BF16, true>(s, x, topk_idx, send_idx, put_offset,
                                            rank_recv_base, recv, row_bytes,
                                            capacity_rows, dev_status, st)
                 : launch_t<MOE_BF16, false>(s, x, topk_idx, send_idx, put_offset,
                                             rank_recv_base, recv, row_bytes,
                                             capacity_rows, dev_status, st);
  return quant ? launch_t<MOE_FP16, true>(s, x, topk_idx, send_idx, put_offset,
                                          rank_recv_base, recv, row_bytes,
                                          capacity_rows, dev_status, st)
               : launch_t<MOE_FP16, false>(s, x, topk_idx, send_idx, put_offset,
                                           rank_recv_base, recv, row_bytes,
                                           capacity_rows, dev_status, st);
}

}  // namespace moe_ep
