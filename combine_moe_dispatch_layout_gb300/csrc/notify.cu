// notify.cu -- stage 2, notify dispatch (UMDK/CAM deep analysis v2, section
// 2.4 moe_notify_dispatch_zb).
//
// On the page every rank AllGathers the others' tokenPerExpert after a
// BarrierAll and then builds putOffset (a prefix sum), maxBs, the total
// receive count and the per-expert receive counts.  Here the R x E count
// matrix is already whole in HBM, so the AllGather is the identity and the
// stage is one launch of a single 8-CTA thread-block cluster:
//
//   * CTA c owns destination ranks [c*R/8, (c+1)*R/8).  It stages the count
//     columns of a group of its ranks in shared memory, transposed to
//     (expert, source) order (coalesced global reads, padded rows);
//   * one warp per destination rank scans that rank's E = epr*R values in
//     (local expert, source rank) order; the exclusive prefix IS the
//     contiguous slice put_offset[r*epr*R ...], so writes are coalesced;
//   * per-rank totals are scanned across the cluster through distributed
//     shared memory (each CTA reads the totals of the CTAs before it) to give
//     rank_recv_base; no global workspace, no spin-waits: the cluster barrier
//     is the only synchronisation.
#include <cooperative_groups.h>

#include <algorithm>

#include "moe_ep_internal.cuh"

namespace cg = cooperative_groups;

namespace moe_ep {
namespace {

constexpr int kCluster = 8;
constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRanksPerCta = (MOE_EP_MAX_RANKS + kCluster - 1) / kCluster;
constexpr int kStageInts = 16384;   // 64 KB of staged counts per group

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
notify_kernel(const int32_t* __restrict__ count, int R, int bs, int epr,
              int32_t* __restrict__ put_offset, int32_t* __restrict__ total_recv,
              int64_t* __restrict__ rank_recv_base,
              int32_t* __restrict__ recv_per_expert, int32_t* __restrict__ max_bs) {
  extern __shared__ __align__(16) int32_t stage[];   // [group experts][R + 1]
  __shared__ int32_t s_tot[kMaxRanksPerCta];
  __shared__ int64_t s_cta_sum;

  cg::cluster_group cluster = cg::this_cluster();
  const int cta = static_cast<int>(cluster.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = R * epr;
  const int ld = R + 1;                       // padded row of the staged block
  const int r_lo = static_cast<int>(int64_t(cta) * R / kCluster);
  const int r_hi = static_cast<int>(int64_t(cta + 1) * R / kCluster);
  // destination ranks per staged group: bounded by the stage and by one warp
  // per rank
  const int group = max(1, min(kWarps, kStageInts / (epr * ld)));

  for (int g0 = r_lo; g0 < r_hi; g0 += group) {
    const int g1 = min(r_hi, g0 + group);
    const int e0 = g0 * epr;
    const int ne = (g1 - g0) * epr;
    // stage count[s][e0 .. e0+ne) transposed to stage[(e - e0) * ld + s]
    for (int i = tid; i < R * ne; i += kThreads) {
      const int s = i / ne, el = i - s * ne;
      stage[el * ld + s] = __ldg(count + int64_t(s) * E + e0 + el);
    }
    __syncthreads();
    // one warp per destination rank: exclusive scan over (j, s)
    if (warp < g1 - g0) {
      const int r = g0 + warp;
      const int n = epr * R;                  // values of this rank
      const int per = (n + 31) / 32;          // contiguous values per lane
      const int i0 = min(n, lane * per), i1 = min(n, i0 + per);
      const int32_t* blk = stage + warp * epr * ld;
      int local = 0;
      for (int i = i0; i < i1; ++i) {
        const int j = i / R, s = i - j * R;
        local += blk[j * ld + s];
      }
      int incl = local;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      int run = incl - local;
      int32_t* po = put_offset + int64_t(r) * n;   // == &put_offset[(r*epr)*R]
      int32_t* blk_w = stage + warp * epr * ld;
      for (int i = i0; i < i1; ++i) {
        const int j = i / R, s = i - j * R;
        const int v = blk_w[j * ld + s];
        po[i] = run;
        blk_w[j * ld + s] = run;   // keep the prefix for recv_per_expert
        run += v;
      }
      const int total = __shfl_sync(0xffffffffu, incl, 31);
      if (lane == 0) {
        total_recv[r] = total;
        s_tot[r - r_lo] = total;
      }
    }
    __syncthreads();
    // rows per expert = next expert's first offset (or the rank total) minus
    // this expert's first offset
    for (int el = tid; el < ne; el += kThreads) {
      const int j = el % epr;
      const int start = stage[el * ld];
      const int end = (j + 1 < epr) ? stage[(el + 1) * ld] : s_tot[g0 + el / epr - r_lo];
      recv_per_expert[e0 + el] = end - start;
    }
    __syncthreads();   // the stage is refilled by the next group
  }

  // ---- rank_recv_base: scan of the totals across the cluster -----------------
  if (tid == 0) {
    int64_t sum = 0;
    for (int i = 0; i < r_hi - r_lo; ++i) sum += s_tot[i];
    s_cta_sum = sum;
  }
  cluster.sync();
  if (tid == 0) {
    int64_t off = 0;
    for (int q = 0; q < cta; ++q) off += *cluster.map_shared_rank(&s_cta_sum, q);
    for (int i = 0; i < r_hi - r_lo; ++i) {
      rank_recv_base[r_lo + i] = off;
      off += s_tot[i];
    }
    if (cta == kCluster - 1) rank_recv_base[R] = off;
    if (cta == 0) max_bs[0] = bs;   // every rank holds bs tokens
  }
  cluster.sync();   // keep s_cta_sum alive until every CTA has read it
}

}  // namespace

cudaError_t launch_notify(const Shape& s, const int32_t* count,
                          int32_t* put_offset, int32_t* total_recv,
                          int64_t* rank_recv_base, int32_t* recv_per_expert,
                          int32_t* max_bs, cudaStream_t st) {
  const int ld = s.R + 1;
  const int group = std::max(1, std::min(kWarps, kStageInts / (s.epr * ld)));
  const size_t smem = sizeof(int32_t) * size_t(group) * s.epr * ld;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(
        notify_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  notify_kernel<<<kCluster, kThreads, smem, st>>>(
      count, s.R, s.bs, s.epr, put_offset, total_recv, rank_recv_base,
      recv_per_expert, max_bs);
  return cudaGetLastError();
}

}  // namespace moe_ep
