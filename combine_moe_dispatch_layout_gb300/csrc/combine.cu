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
// gather never waits on index arithmetic; for wide rows it also asks L2 for
// that token's rows with one bulk prefetch each.  Each compute thread owns 16-byte
// chunks of the hidden dimension and issues the loads of up to 8 expert
// rows before doing any arithmetic.  The arithmetic is exactly the page's:
// acc = 0; acc = acc + (y * w), one rounding for the multiply and one for
// the add (__fmul_rn / __fadd_rn; the unit is also built with -fmad=false),
// k in order; out = round-to-nearest-even in the token dtype.
#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int kBatch = 8;          // expert rows loaded before accumulating
constexpr int kMaxThreads = 1024;

template <int DT>
__global__ void __launch_bounds__(kMaxThreads)
combine_kernel(const uint4* __restrict__ y, int64_t y_rows,
               const int32_t* __restrict__ topk_idx,
               const float* __restrict__ weights,
               const int32_t* __restrict__ send_idx,
               const int32_t* __restrict__ put_offset,
               const int64_t* __restrict__ rank_recv_base, int R, int bs, int k,
               int epr, int H, int64_t T, uint4* __restrict__ out,
               int32_t* dev_status, bool prefetch_next) {
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
      if (gn < T) {
        resolve_token(gn, topk_idx, weights, send_idx, put_offset, rank_recv_base,
                      R, bs, k, epr, y_rows, s_rows[buf ^ 1], s_w[buf ^ 1],
                      dev_status, lane);
        // wide rows: the next token's rows start streaming into L2 while
        // this one is summed (one bulk prefetch per row, no shared memory
        // or registers)
        for (int kk = lane; prefetch_next && kk < k; kk += 32) {
          const int64_t row = s_rows[buf ^ 1][kk];
          if (row >= 0) bulk_prefetch_l2(y + row * nch, static_cast<uint32_t>(nch) * 16u);
        }
      }
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

// Compute threads per CTA for `cpt` chunks each: a multiple of 32, at most
// 992 (plus the producer warp).
int compute_threads(int nch, int cpt) {
  int t = ((nch + cpt - 1) / cpt + 31) / 32 * 32;
  return std::max(32, std::min(kMaxThreads - 32, t));
}

// Rows in flight per SM below which fewer, wider CTAs stop paying: a token's
// k rows are in flight while its CTA gathers them.
constexpr int64_t kInFlightBytes = 160 * 1024;

// Rows at least this wide (two CTAs per SM) gain from prefetching the next
// token's rows into L2 (measured: 14 KB rows, dsv3 630 -> 622 us, maxrank
// 944 -> 924 us); narrower rows, with more CTAs per SM, lose (skew's 8 KB
// rows 295 -> 318 us, fp16's 4 KB rows 189 -> 200 us).
constexpr int64_t kPrefetchRowBytes = 12 * 1024;

template <int DT>
cudaError_t launch_t(const Shape& s, const void* y, int64_t y_rows,
                     const int32_t* topk_idx, const float* weights,
                     const int32_t* send_idx, const int32_t* put_offset,
                     const int64_t* rank_recv_base, void* out,
                     int32_t* dev_status, cudaStream_t st) {
  const int nch = s.H / 8;
  int dev = 0, sms = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e != cudaSuccess) return e;
  // Two chunks per compute thread (a shorter gather per token) when the CTAs
  // that fit still keep kInFlightBytes of rows in flight per SM, else four
  // (more CTAs).  Measured: with two, dsv3 (2 CTAs x 112 KB per SM) 634 ->
  // 625 us, fp16 (6 x 32 KB) 196 -> 188, maxrank 951 -> 937; skew (3 x 48 KB)
  // 294 -> 301, so it keeps four.
  int threads = 0, per_sm = 0;
  for (int cpt = 2; cpt <= 4; cpt += 2) {
    threads = compute_threads(nch, cpt) + 32;
    e = kernel_blocks_per_sm(reinterpret_cast<const void*>(combine_kernel<DT>), threads, 0,
                             &per_sm);
    if (e != cudaSuccess) return e;
    if (int64_t(per_sm) * s.k * s.H * 2 >= kInFlightBytes) break;
  }
  const int64_t grid = std::min<int64_t>(s.T(), int64_t(std::max(1, per_sm)) * sms);
  combine_kernel<DT><<<static_cast<unsigned>(grid), threads, 0, st>>>(
      static_cast<const uint4*>(y), y_rows, topk_idx, weights, send_idx,
      put_offset, rank_recv_base, s.R, s.bs, s.k, s.epr, s.H, s.T(),
      static_cast<uint4*>(out), dev_status, int64_t(s.H) * 2 >= kPrefetchRowBytes);
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
