// deq_combine.cu -- DeqCombine of the fused deep MoE (UMDK/CAM deep analysis
// v2, section 4.3, stage 3: read INT32, cast to FP32, x weight_scale,
// x per_token_scale, then the combine's score multiply and add), and the
// expert row offsets that the grouped stages use.
//
// Expert-output rows are GMM2's int32 accumulators [rows][H].  For token g
// and slot k (row = the dispatch row of (g, k), e = its expert):
//   y = (fp32(acc2[row][h]) * weight_scale[e][h]) * row_scale[row]
//   acc = acc + (y * w[g][k])          (k in order; acc starts at 0)
// and out[g][h] = acc rounded to nearest even in the token dtype.  Each step
// is one fp32 operation rounded to nearest even (_rn intrinsics; the unit is
// built with -fmad=false).
//
// moe_combine_f32 runs the same kernel on fp32 rows that the GMM2 epilogue
// has already dequantised (the two multiplies in the same order), so the
// combine reads 4H bytes per (token, k) and no weight scales.
//
// Same persistent producer / compute structure as the combine: the last
// warp resolves the next token's rows, weights, experts and row scales into
// a double-buffered shared table; compute threads own 8 outputs each (two
// 16-byte loads of int32 and of the expert's weight scales per row, 4 rows
// in flight).  HBM-bound: 4H bytes
// read per (token, k), 2H written per token; the per-expert weight scales
// (E x H fp32) stay in L2.
#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int kMaxThreads = 512;   // <= 128 registers per thread

// DEQ: int32 rows dequantised with the expert's column scales and the row
// scale (DeqCombine).  !DEQ: fp32 rows already dequantised (by the GEMM's
// epilogue), weight_scale and row_scale unused.
template <int DT, bool DEQ>
__global__ void __launch_bounds__(kMaxThreads)
deq_combine_kernel(const int32_t* __restrict__ acc2, int64_t y_rows,
                   const float* __restrict__ weight_scale,
                   const unsigned char* __restrict__ row_scale, int64_t rs_stride,
                   const int32_t* __restrict__ topk_idx, const float* __restrict__ weights,
                   const int32_t* __restrict__ send_idx,
                   const int32_t* __restrict__ put_offset,
                   const int64_t* __restrict__ rank_recv_base, int R, int bs, int k,
                   int epr, int H, int64_t T, uint4* __restrict__ out,
                   int32_t* dev_status) {
  constexpr int kBatch = DEQ ? 4 : 8;   // rows in flight (DEQ: + weight scales)
  __shared__ int64_t s_rows[2][MOE_EP_MAX_TOPK];
  __shared__ float s_w[2][MOE_EP_MAX_TOPK];
  __shared__ int32_t s_e[2][MOE_EP_MAX_TOPK];
  __shared__ float s_ts[2][MOE_EP_MAX_TOPK];
  const int tid = threadIdx.x, lane = tid & 31;
  const int ncomp = blockDim.x - 32;
  const bool producer = tid >= ncomp;
  const int nch = H / 8;

  auto resolve = [&](int64_t gt, int b) {
    resolve_token(gt, topk_idx, weights, send_idx, put_offset, rank_recv_base, R, bs, k,
                  epr, y_rows, s_rows[b], s_w[b], dev_status, lane);
    __syncwarp();
    for (int kk = lane; DEQ && kk < k; kk += 32) {
      const int64_t row = s_rows[b][kk];
      s_e[b][kk] = row >= 0 ? __ldg(topk_idx + gt * k + kk) : 0;
      s_ts[b][kk] = row >= 0 ? __ldg(reinterpret_cast<const float*>(row_scale + row * rs_stride))
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
      for (int c = tid; c < nch; c += ncomp) {
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        for (int k0 = 0; k0 < k; k0 += kBatch) {
          uint4 v[kBatch][2];
          float4 wsv[kBatch][2];
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int kk = k0 + b;
            const int64_t row = kk < k ? rows[kk] : -1;
            if (row >= 0) {
              const int32_t* src = acc2 + row * H + 8 * c;
              v[b][0] = ld_stream_16(src);
              v[b][1] = ld_stream_16(src + 4);
              if (DEQ) {
                const float* ws = weight_scale + int64_t(s_e[buf][kk]) * H + 8 * c;
                wsv[b][0] = __ldg(reinterpret_cast<const float4*>(ws));
                wsv[b][1] = __ldg(reinterpret_cast<const float4*>(ws + 4));
              }
            } else {
              v[b][0] = v[b][1] = make_uint4(0u, 0u, 0u, 0u);
              wsv[b][0] = wsv[b][1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            const int kk = k0 + b;
            if (kk < k && rows[kk] >= 0) {
              const float wk = s_w[buf][kk], ts = s_ts[buf][kk];
              const float wsr[8] = {wsv[b][0].x, wsv[b][0].y, wsv[b][0].z, wsv[b][0].w,
                                    wsv[b][1].x, wsv[b][1].y, wsv[b][1].z, wsv[b][1].w};
              const uint32_t a[8] = {v[b][0].x, v[b][0].y, v[b][0].z, v[b][0].w,
                                     v[b][1].x, v[b][1].y, v[b][1].z, v[b][1].w};
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                float y;
                if (DEQ) {
                  y = __int2float_rn(static_cast<int32_t>(a[j]));       // Cast FP32
                  y = __fmul_rn(y, wsr[j]);                             // x weight_scale
                  y = __fmul_rn(y, ts);                                 // x per-token scale
                } else {
                  y = __uint_as_float(a[j]);                            // already fp32
                }
                acc[j] = __fadd_rn(acc[j], __fmul_rn(y, wk));           // Muls, Add
              }
            }
          }
        }
        out[g * nch + c] = pack8<DT>(acc);
      }
    }
    __syncthreads();
  }
}

int compute_threads(int nch) {
  const int t = ((nch + 3) / 4 + 31) / 32 * 32;
  return std::max(32, std::min(kMaxThreads - 32, t));
}

template <int DT, bool DEQ>
cudaError_t launch_t(const Shape& s, const int32_t* acc2, int64_t y_rows,
                     const float* weight_scale, const void* row_scale, int64_t rs_stride,
                     const int32_t* topk_idx, const float* weights, const int32_t* send_idx,
                     const int32_t* put_offset, const int64_t* rank_recv_base, void* out,
                     int32_t* dev_status, cudaStream_t st) {
  const int threads = compute_threads(s.H / 8) + 32;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e == cudaSuccess)
    e = kernel_blocks_per_sm(reinterpret_cast<const void*>(deq_combine_kernel<DT, DEQ>),
                             threads, 0, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(s.T(), int64_t(std::max(1, per_sm)) * sms);
  deq_combine_kernel<DT, DEQ><<<static_cast<unsigned>(grid), threads, 0, st>>>(
      acc2, y_rows, weight_scale, static_cast<const unsigned char*>(row_scale), rs_stride,
      topk_idx, weights, send_idx, put_offset, rank_recv_base, s.R, s.bs, s.k, s.epr, s.H,
      s.T(), static_cast<uint4*>(out), dev_status);
  return cudaGetLastError();
}

// Exclusive prefix of the per-expert row counts (one CTA, G <= 4096).
__global__ void __launch_bounds__(1024)
group_offsets_kernel(const int32_t* __restrict__ counts, int G, int64_t* __restrict__ off,
                     int32_t* dev_status) {
  __shared__ int64_t s_part[1024];
  const int tid = threadIdx.x;
  const int per = (G + blockDim.x - 1) / blockDim.x;
  const int g0 = tid * per < G ? tid * per : G, g1 = g0 + per < G ? g0 + per : G;
  int64_t sum = 0;
  for (int g = g0; g < g1; ++g) {
    const int32_t c = __ldg(counts + g);
    if (c < 0) set_status(dev_status, MOE_ERR_INVALID_ARG);
    sum += c < 0 ? 0 : c;
  }
  s_part[tid] = sum;
  __syncthreads();
  for (int d = 1; d < blockDim.x; d <<= 1) {   // inclusive Hillis-Steele scan
    const int64_t v = tid >= d ? s_part[tid - d] : 0;
    __syncthreads();
    s_part[tid] += v;
    __syncthreads();
  }
  int64_t run = s_part[tid] - sum;
  for (int g = g0; g < g1; ++g) {
    off[g] = run;
    const int32_t c = __ldg(counts + g);
    run += c < 0 ? 0 : c;
  }
  if (tid == blockDim.x - 1) off[G] = s_part[tid];
}

}  // namespace

cudaError_t launch_deq_combine(const Shape& s, const int32_t* acc2, int64_t y_rows,
                               const float* weight_scale, const void* row_scale,
                               int64_t row_scale_stride, const int32_t* topk_idx,
                               const float* weights, const int32_t* send_idx,
                               const int32_t* put_offset, const int64_t* rank_recv_base,
                               void* out, int32_t* dev_status, cudaStream_t st) {
  if (s.T() == 0) return cudaSuccess;
  if (s.dtype == MOE_BF16)
    return launch_t<MOE_BF16, true>(s, acc2, y_rows, weight_scale, row_scale, row_scale_stride,
                                    topk_idx, weights, send_idx, put_offset, rank_recv_base,
                                    out, dev_status, st);
  return launch_t<MOE_FP16, true>(s, acc2, y_rows, weight_scale, row_scale, row_scale_stride,
                                  topk_idx, weights, send_idx, put_offset, rank_recv_base, out,
                                  dev_status, st);
}

cudaError_t launch_combine_f32(const Shape& s, const float* y, int64_t y_rows,
                               const int32_t* topk_idx, const float* weights,
                               const int32_t* send_idx, const int32_t* put_offset,
                               const int64_t* rank_recv_base, void* out, int32_t* dev_status,
                               cudaStream_t st) {
  if (s.T() == 0) return cudaSuccess;
  const int32_t* yy = reinterpret_cast<const int32_t*>(y);
  if (s.dtype == MOE_BF16)
    return launch_t<MOE_BF16, false>(s, yy, y_rows, nullptr, nullptr, 4, topk_idx, weights,
                                     send_idx, put_offset, rank_recv_base, out, dev_status, st);
  return launch_t<MOE_FP16, false>(s, yy, y_rows, nullptr, nullptr, 4, topk_idx, weights,
                                   send_idx, put_offset, rank_recv_base, out, dev_status, st);
}

cudaError_t launch_group_offsets(const int32_t* counts, int G, int64_t* off,
                                 int32_t* dev_status, cudaStream_t st) {
  group_offsets_kernel<<<1, 1024, 0, st>>>(counts, G, off, dev_status);
  return cudaGetLastError();
}

}  // namespace moe_ep
