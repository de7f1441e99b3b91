// token_layout.cu -- distinct tokens per destination rank (UMDK/CAM deep
// analysis v2, section 2.3: the per-rank receive count, read at token
// granularity).  moe_dispatch_layout counts
// (token, k) pairs; this stage counts a token once per destination rank it
// reaches, and records the token x rank membership map, as an expert-
// parallel runtime that sends one copy of a token per rank would need.
//
// One thread per token: it loads its k expert ids (all loads in flight),
// sets one bit per destination rank in a private shared-memory bitmask and
// bumps the CTA's per-rank counters.  Membership rows are written in 4-byte
// words (R % 4 == 0): by their own thread when rows are short (R <= 32,
// neighbouring rows are then contiguous), else by the whole warp, one row
// at a time, 32 lanes x 4 contiguous bytes.  A CTA covers tokens of one
// source rank; its counters are added to tokens_per_rank[s][:] with integer
// atomics, which are order-independent, so the counts are deterministic.
// tokens_per_rank is zeroed on the stream first.
#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int kThreads = 128;
constexpr int kMaskWords = (MOE_EP_MAX_RANKS + 31) / 32;   // 12

__global__ void __launch_bounds__(kThreads)
token_layout_kernel(const int32_t* __restrict__ topk_idx, int R, int bs, int k,
                    int epr, int chunks_per_rank, int32_t* __restrict__ tokens_per_rank,
                    uint8_t* __restrict__ in_rank, int32_t* dev_status) {
  __shared__ uint32_t s_mask[kMaskWords][kThreads];   // [word][thread]: no conflicts
  __shared__ int32_t s_cnt[MOE_EP_MAX_RANKS];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int s = blockIdx.x / chunks_per_rank;
  const int chunk = blockIdx.x - s * chunks_per_rank;
  const int t = chunk * kThreads + tid;
  const int E = R * epr;
  const int words = (R + 31) / 32;
  for (int r = tid; r < R; r += kThreads) s_cnt[r] = 0;
  for (int j = 0; j < words; ++j) s_mask[j][tid] = 0u;
  __syncthreads();

  if (t < bs) {
    const int64_t g = int64_t(s) * bs + t;
    const int32_t* ids = topk_idx + g * k;
    for (int k0 = 0; k0 < k; k0 += 8) {
      int e[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) e[u] = k0 + u < k ? __ldg(ids + k0 + u) : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (k0 + u >= k) break;
        if (static_cast<unsigned>(e[u]) >= static_cast<unsigned>(E)) {
          set_status(dev_status, MOE_ERR_EXPERT_ID);
          continue;
        }
        const int r = e[u] / epr;
        s_mask[r >> 5][tid] |= 1u << (r & 31);
      }
    }
    uint8_t* row = in_rank + g * R;
    if ((R & 3) == 0 && R <= 32) {
      for (int r0 = 0; r0 < R; r0 += 4) {
        const uint32_t m = s_mask[r0 >> 5][tid] >> (r0 & 31);
        *reinterpret_cast<uint32_t*>(row + r0) =
            (m & 1u) | ((m >> 1) & 1u) << 8 | ((m >> 2) & 1u) << 16 | ((m >> 3) & 1u) << 24;
      }
    } else if ((R & 3) != 0) {
      for (int r = 0; r < R; ++r) row[r] = (s_mask[r >> 5][tid] >> (r & 31)) & 1u;
    }
    for (int j = 0; j < words; ++j) {
      uint32_t m = s_mask[j][tid];
      while (m) {
        const int b = __ffs(m) - 1;
        m &= m - 1;
        atomicAdd(&s_cnt[j * 32 + b], 1);
      }
    }
  }
  __syncwarp();
  if ((R & 3) == 0 && R > 32) {   // long rows: the warp writes them one by one
    const int t0 = chunk * kThreads + warp * 32;
    for (int j = 0; j < 32 && t0 + j < bs; ++j) {
      uint8_t* row = in_rank + (int64_t(s) * bs + t0 + j) * R;
      for (int r0 = 4 * lane; r0 < R; r0 += 128) {
        const uint32_t m = s_mask[r0 >> 5][warp * 32 + j] >> (r0 & 31);
        *reinterpret_cast<uint32_t*>(row + r0) =
            (m & 1u) | ((m >> 1) & 1u) << 8 | ((m >> 2) & 1u) << 16 | ((m >> 3) & 1u) << 24;
      }
    }
  }
  __syncthreads();
  for (int r = tid; r < R; r += kThreads)
    if (s_cnt[r]) atomicAdd(tokens_per_rank + int64_t(s) * R + r, s_cnt[r]);
}

}  // namespace

cudaError_t launch_token_layout(const Shape& s, const int32_t* topk_idx,
                                int32_t* tokens_per_rank, uint8_t* in_rank,
                                int32_t* dev_status, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(tokens_per_rank, 0, sizeof(int32_t) * size_t(s.R) * s.R, st);
  if (e != cudaSuccess || s.T() == 0) return e;
  const int chunks = (s.bs + kThreads - 1) / kThreads;
  token_layout_kernel<<<s.R * chunks, kThreads, 0, st>>>(
      topk_idx, s.R, s.bs, s.k, s.epr, chunks, tokens_per_rank, in_rank, dev_status);
  return cudaGetLastError();
}

}  // namespace moe_ep
