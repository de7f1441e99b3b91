// notify.cu -- stage 2, notify dispatch (UMDK/CAM deep analysis v2, section
// 2.4 moe_notify_dispatch_zb).
//
// On the page every rank AllGathers the others' tokenPerExpert after a
// BarrierAll and then builds putOffset (a prefix sum), maxBs, the total
// receive count and the per-expert receive counts.  Here the R x E count
// matrix is already whole in HBM (and in L2: the layout stage has just
// written it), so the AllGather is the identity.
//
// Each destination rank is scanned by one warp.  Rank r's values, in (local
// expert j, source rank s) order, are walked 32 at a time: lane l of row t
// holds value i = 32t + l = j*R + s, read straight from count[s][r*epr + j]
// (up to 16 rows of loads in flight), and scanned with warp shuffles plus a
// running carry.  The exclusive prefix is the contiguous slice
// put_offset[r*epr*R ...], so the stores are coalesced.  Rows per expert
// come from the prefix just written (next expert's first offset, or the
// rank total, minus this expert's first offset).  Then rank_recv_base is
// the exclusive scan (int64) of the rank totals.
//
//   * R <= 64: one CTA does everything in one launch;
//   * larger R: the column reads are scattered, so the number of SMs issuing
//     them sets the pace: notify_scan_kernel spreads the ranks over many
//     CTAs (one warp each), then notify_base_kernel (one CTA) scans the
//     totals.
#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int kScanWarps = 4;                 // destination ranks per CTA
constexpr int kRowBatch = 16;                 // 32-value rows loaded per batch
constexpr int kBaseThreads = 512;             // >= MOE_EP_MAX_RANKS
constexpr int kSmallR = 64;                   // one-CTA path up to this R
constexpr int kSmallThreads = 1024;

// Scan destination rank r (one warp); returns the rank total.
__device__ __forceinline__ int scan_rank(const int32_t* __restrict__ count, int R,
                                         int epr, int r, int lane,
                                         int32_t* __restrict__ put_offset,
                                         int32_t* __restrict__ recv_per_expert) {
  const int E = R * epr;
  const int n = E;                                 // values of this rank
  int32_t* po = put_offset + int64_t(r) * n;       // == &put_offset[(r*epr)*R]
  const int32_t* col = count + int64_t(r) * epr;   // column block of rank r
  int carry = 0;
  for (int t0 = 0; t0 * 32 < n; t0 += kRowBatch) {
    int v[kRowBatch];
#pragma unroll
    for (int b = 0; b < kRowBatch; ++b) {
      const int i = (t0 + b) * 32 + lane;
      const int j = i / R, s = i - j * R;
      v[b] = i < n ? __ldg(col + int64_t(s) * E + j) : 0;
    }
#pragma unroll
    for (int b = 0; b < kRowBatch; ++b) {
      if ((t0 + b) * 32 >= n) break;              // warp-uniform
      const int i = (t0 + b) * 32 + lane;
      int incl = v[b];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += u;
      }
      if (i < n) po[i] = carry + incl - v[b];
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
  __syncwarp();   // this warp's put_offset stores are visible to its lanes
  for (int j = lane; j < epr; j += 32) {
    const int start = po[j * R];
    const int end = (j + 1 < epr) ? po[(j + 1) * R] : carry;
    recv_per_expert[r * epr + j] = end - start;
  }
  return carry;
}

__global__ void __launch_bounds__(kScanWarps * 32)
notify_scan_kernel(const int32_t* __restrict__ count, int R, int epr,
                   int32_t* __restrict__ put_offset, int32_t* __restrict__ total_recv,
                   int32_t* __restrict__ recv_per_expert) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kScanWarps + (threadIdx.x >> 5);
  if (r >= R) return;
  const int total = scan_rank(count, R, epr, r, lane, put_offset, recv_per_expert);
  if (lane == 0) total_recv[r] = total;
}

// R <= kSmallR: all of notify in one CTA.
__global__ void __launch_bounds__(kSmallThreads)
notify_small_kernel(const int32_t* __restrict__ count, int R, int bs, int epr,
                    int32_t* __restrict__ put_offset, int32_t* __restrict__ total_recv,
                    int64_t* __restrict__ rank_recv_base,
                    int32_t* __restrict__ recv_per_expert, int32_t* __restrict__ max_bs) {
  __shared__ int32_t s_tot[kSmallR];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int r = warp; r < R; r += kSmallThreads / 32) {
    const int total = scan_rank(count, R, epr, r, lane, put_offset, recv_per_expert);
    if (lane == 0) {
      total_recv[r] = total;
      s_tot[r] = total;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int64_t off = 0;
    for (int r = 0; r < R; ++r) {
      rank_recv_base[r] = off;
      off += s_tot[r];
    }
    rank_recv_base[R] = off;
    max_bs[0] = bs;   // every rank holds bs tokens
  }
}

__global__ void __launch_bounds__(kBaseThreads)
notify_base_kernel(const int32_t* __restrict__ total_recv, int R, int bs,
                   int64_t* __restrict__ rank_recv_base, int32_t* __restrict__ max_bs) {
  __shared__ int64_t s_warp[kBaseThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t v = tid < R ? total_recv[tid] : 0;
  int64_t incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int64_t u = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += u;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int64_t off = 0;
  for (int w = 0; w < warp; ++w) off += s_warp[w];
  if (tid < R) rank_recv_base[tid] = off + incl - v;
  if (tid == R - 1) rank_recv_base[R] = off + incl;
  if (tid == 0) max_bs[0] = bs;   // every rank holds bs tokens
}

}  // namespace

cudaError_t launch_notify(const Shape& s, const int32_t* count,
                          int32_t* put_offset, int32_t* total_recv,
                          int64_t* rank_recv_base, int32_t* recv_per_expert,
                          int32_t* max_bs, cudaStream_t st) {
  if (s.R <= kSmallR) {
    notify_small_kernel<<<1, kSmallThreads, 0, st>>>(count, s.R, s.bs, s.epr, put_offset,
                                                      total_recv, rank_recv_base,
                                                      recv_per_expert, max_bs);
    return cudaGetLastError();
  }
  const int grid = (s.R + kScanWarps - 1) / kScanWarps;
  notify_scan_kernel<<<grid, kScanWarps * 32, 0, st>>>(count, s.R, s.epr, put_offset,
                                                        total_recv, recv_per_expert);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  notify_base_kernel<<<1, kBaseThreads, 0, st>>>(total_recv, s.R, s.bs, rank_recv_base,
                                                 max_bs);
  return cudaGetLastError();
}

}  // namespace moe_ep
