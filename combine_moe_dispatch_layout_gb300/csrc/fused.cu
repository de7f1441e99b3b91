// fused.cu -- low-latency dispatch: layout + notify + dispatch in one launch
// (UMDK/CAM deep analysis v2, section 3.2 moe_dispatch_lowlatency_zb: local
// layout, layout status, count notify, prefix, token output, sync flags, all
// inside one kernel).
//
// For small batches the three separate launches cost more in launch and
// drain latency than in work.  Here one cooperative launch of persistent
// CTAs runs four phases separated by a grid barrier:
//
//   A. layout tiles (2048 pairs inside one source rank): per-warp stable
//      ranks with __match_any_sync and shared counters, a column scan over
//      the warps, the tile histogram to the workspace, the in-tile rank to
//      send_idx;
//   B. one thread per (source rank, expert): exclusive scan of that column
//      over the rank's tiles (in place in the workspace) and the count;
//   C. send_idx += the tile's prefix; rank_send; one warp per destination
//      rank scans (local expert, source rank) into put_offset,
//      recv_per_expert and total_recv (the notify stage);
//   D. every CTA scans the R totals into the partition bases (CTA 0 writes
//      rank_recv_base and maxBs) and dispatches tokens: rows resolved by one
//      warp, max|x| by a block reduction, codes and 1/scale exactly as
//      moe_dispatch (scale = 127/(amax + 1e-12f), round half to even).
//      When the rows fit (STAGED), the CTA's first two x rows are requested
//      with cp.async.bulk at kernel start, so they arrive while phases A-C
//      run; each token's row image (or x itself, verbatim) is built in
//      shared memory and written to its k rows with k bulk stores, and the
//      token two steps ahead is loaded into the freed stage, as moe_dispatch
//      does.  Otherwise threads store the image with 8-byte stores.
//
// The grid barrier is a generation counter in the workspace; a wait that
// exceeds its bound (about a second) sets MOE_ERR_TIMEOUT and the CTA goes
// on (every receive-row write is still checked against the capacity).  Data
// written in an earlier phase by another CTA is read through L2 (__ldcg).
#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRounds = 8;
constexpr int kTile = kWarps * kRounds * 32;     // 2048 pairs
constexpr uint32_t kBarrierSpin = 1u << 20;
// CTAs per SM (CPS, a template parameter: the register cap that lets them
// all be resident): 2 when x rows are 12 KB or wider, else 4 on the INT8
// path and 3 on the verbatim path (measured fastest per shape).

struct BarrierWs {
  uint32_t count;
  uint32_t gen;
  uint32_t pad[14];
};

__device__ void grid_sync(BarrierWs* bw, uint32_t nblocks, int32_t* dev_status) {
  __syncthreads();
  if (nblocks == 1u) return;   // one CTA: the block barrier is the grid barrier
  if (threadIdx.x == 0) {
    const uint32_t g = ld_acquire_gpu(&bw->gen);
    __threadfence();
    if (atomicAdd(&bw->count, 1u) == nblocks - 1u) {
      bw->count = 0u;   // all have arrived: nobody reads it again this round
      __threadfence();
      st_release_gpu(&bw->gen, g + 1u);
    } else {
      for (uint32_t spins = 0; ld_acquire_gpu(&bw->gen) == g; ++spins) {
        if (spins >= kBarrierSpin) {
          set_status(dev_status, MOE_ERR_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
    }
    __threadfence();
  }
  __syncthreads();
}

struct Params {
  const unsigned char* x;
  const int32_t* topk_idx;
  int R, bs, k, epr, H;
  int tiles_per_rank, num_tiles;
  int32_t* count;
  int32_t* rank_send;
  int32_t* send_idx;
  int32_t* put_offset;
  int32_t* total_recv;
  int64_t* rank_recv_base;
  int32_t* recv_per_expert;
  int32_t* max_bs;
  unsigned char* recv;
  int64_t row_bytes, capacity;
  void* workspace;
  int32_t* dev_status;
};

// x stages of the token phase: two with the INT8 image (the block computes
// each token), four on the verbatim path (one warp copies, stages refilled
// three tokens ahead).
constexpr int kQuantStages = 2, kCopyStages = 4;

// Dynamic shared memory: warp counters, partition bases, then (STAGED) the x
// stages, two image stages (QUANT) and one mbarrier per x stage.
struct FusedSmem {
  int64_t xs, os, bar, bytes;   // byte offsets of the x stages, images, barriers; total
  int64_t x_stride, o_stride;
};
__host__ __device__ inline FusedSmem fused_smem(int R, int E, int H, int64_t row_bytes,
                                                bool staged, bool quant) {
  FusedSmem L;
  const int nst = quant ? kQuantStages : kCopyStages;
  const int64_t head = align_up(2 * kWarps * int64_t(E), 16) + 8 * int64_t(R + 1);
  L.x_stride = staged ? align_up(int64_t(H) * 2, 128) : 0;
  L.o_stride = staged && quant ? align_up(row_bytes, 128) : 0;
  L.xs = align_up(head, 128);
  L.os = L.xs + nst * L.x_stride;
  L.bar = L.os + 2 * L.o_stride;
  L.bytes = staged ? L.bar + 8 * nst : head;
  return L;
}

template <int DT, bool QUANT, bool STAGED, int CPS>
__global__ void __launch_bounds__(kThreads, CPS)
fused_dispatch_kernel(Params p) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int R = p.R, epr = p.epr, k = p.k, H = p.H, E = R * epr;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t G = gridDim.x;
  const int64_t gthreads = int64_t(G) * kThreads;
  const int64_t gtid = int64_t(blockIdx.x) * kThreads + tid;
  const int64_t per_rank = int64_t(p.bs) * k;
  const int64_t P = per_rank * R;
  BarrierWs* bw = static_cast<BarrierWs*>(p.workspace);
  int32_t* agg = reinterpret_cast<int32_t*>(static_cast<char*>(p.workspace) + 64);

  uint16_t* wcnt = reinterpret_cast<uint16_t*>(smem);                      // [8][E]
  int64_t* s_base = reinterpret_cast<int64_t*>(smem + align_up(2 * kWarps * E, 16));  // [R+1]
  __shared__ int64_t s_rows2[2][MOE_EP_MAX_TOPK];
  int64_t* s_rows = s_rows2[0];
  __shared__ float s_wmax[kWarps];
  __shared__ int s_abort;

  const FusedSmem SL = fused_smem(R, E, H, p.row_bytes, STAGED, QUANT);
  unsigned char* xs = smem + SL.xs;
  unsigned char* os = smem + SL.os;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + SL.bar);
  const int64_t T = int64_t(R) * p.bs;
  const uint32_t xbytes = static_cast<uint32_t>(H) * 2u;
  constexpr int kNst = QUANT ? kQuantStages : kCopyStages;
  int pend[kNst];           // issuer: completion parity of the x load in flight per stage
#pragma unroll
  for (int st = 0; st < kNst; ++st) pend[st] = -1;
  // The thread that issues the token phase's copies (and owns their bulk
  // groups and pend[]): lane 0 of the last warp on the INT8 path -- its warp
  // holds the fewest x chunks, so the copy duties do not delay a block barrier
  // (thread 0, on the busiest warp, made every token ~4% slower) -- and thread
  // 0 on the verbatim path, whose warp 0 runs the token loop alone.
  const int issuer = QUANT ? kThreads - 32 : 0;
  if (STAGED && tid == issuer) {  // this CTA's first x rows arrive during phases A-C
    for (int st = 0; st < kNst; ++st) mbar_init(&mbar[st], 1);
    fence_mbar_init();
    for (int st = 0; st < kNst; ++st) {
      const int64_t gs = blockIdx.x + int64_t(st) * G;
      if (gs < T) {
        mbar_arrive_expect_tx(&mbar[st], xbytes);
        bulk_load(xs + st * SL.x_stride, p.x + gs * xbytes, xbytes, &mbar[st]);
        pend[st] = 0;
      }
    }
  }
  if (tid == 0) s_abort = 0;

  // ---- A: layout tiles -------------------------------------------------------
  for (int tile = blockIdx.x; tile < p.num_tiles; tile += G) {
    for (int i = tid; i < (kWarps * E + 1) / 2; i += kThreads)
      reinterpret_cast<uint32_t*>(wcnt)[i] = 0u;
    __syncthreads();
    const int s = tile / p.tiles_per_rank;
    const int c = tile - s * p.tiles_per_rank;
    const int64_t p0 = int64_t(c) * kTile;
    const int64_t p_end = min(p0 + kTile, per_rank);
    const int32_t* idx_rank = p.topk_idx + int64_t(s) * per_rank;
    int32_t* out_rank = p.send_idx + int64_t(s) * per_rank;
    const int64_t seg0 = p0 + int64_t(warp) * kRounds * 32;
    int ev[kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int64_t q = seg0 + r * 32 + lane;
      ev[r] = q < p_end ? __ldg(idx_rank + q) : -1;
    }
    unsigned grp[kRounds];
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int64_t q = seg0 + r * 32 + lane;
      const bool valid = static_cast<unsigned>(ev[r]) < static_cast<unsigned>(E);
      if (q < p_end && !valid) set_status(p.dev_status, MOE_ERR_EXPERT_ID);
      if (!valid) ev[r] = -1 - lane;
      grp[r] = __match_any_sync(0xffffffffu, ev[r]);
    }
    int rk[kRounds];
    const unsigned lt = lanemask_lt();
    uint16_t* my_cnt = wcnt + warp * E;
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int e = ev[r];
      const int lrank = __popc(grp[r] & lt);
      const int base = e >= 0 ? my_cnt[e] : 0;
      __syncwarp();
      if (e >= 0 && lrank == 0) my_cnt[e] = static_cast<uint16_t>(base + __popc(grp[r]));
      __syncwarp();
      rk[r] = e >= 0 ? base + lrank : -1;
    }
    __syncthreads();
    for (int e = tid; e < E; e += kThreads) {
      int v[kWarps];
#pragma unroll
      for (int w = 0; w < kWarps; ++w) v[w] = wcnt[w * E + e];
      int run = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        wcnt[w * E + e] = static_cast<uint16_t>(run);
        run += v[w];
      }
      agg[int64_t(tile) * E + e] = run;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int64_t q = seg0 + r * 32 + lane;
      if (q < p_end) out_rank[q] = rk[r] < 0 ? -1 : my_cnt[ev[r]] + rk[r];
    }
    __syncthreads();   // wcnt is cleared by the next tile
  }
  grid_sync(bw, G, p.dev_status);

  // ---- B: per (source rank, expert) scan over the rank's tiles --------------
  for (int64_t col = gtid; col < int64_t(R) * E; col += gthreads) {
    const int s = static_cast<int>(col / E), e = static_cast<int>(col - int64_t(s) * E);
    int run = 0;
    for (int c = 0; c < p.tiles_per_rank; ++c) {
      int32_t* a = agg + (int64_t(s) * p.tiles_per_rank + c) * E + e;
      const int v = __ldcg(a);
      *a = run;
      run += v;
    }
    p.count[col] = run;
  }
  grid_sync(bw, G, p.dev_status);

  // ---- C: send indices, rank_send, notify ------------------------------------
  for (int64_t q = gtid; q < P; q += gthreads) {
    const int e = __ldg(p.topk_idx + q);
    if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
      const int s = static_cast<int>(q / per_rank);
      const int c = static_cast<int>((q - s * per_rank) / kTile);
      p.send_idx[q] = __ldcg(p.send_idx + q) +
                      __ldcg(agg + (int64_t(s) * p.tiles_per_rank + c) * E + e);
    }
  }
  for (int64_t q = gtid; q < int64_t(R) * R; q += gthreads) {
    const int s = static_cast<int>(q / R), r = static_cast<int>(q - int64_t(s) * R);
    int sum = 0;
    for (int j = 0; j < epr; ++j) sum += __ldcg(p.count + int64_t(s) * E + r * epr + j);
    p.rank_send[q] = sum;
  }
  const int64_t gwarp = gtid / 32, nwarps = gthreads / 32;
  for (int64_t rr = gwarp; rr < R; rr += nwarps) {
    const int r = static_cast<int>(rr);
    int32_t* po = p.put_offset + int64_t(r) * E;       // == &put_offset[(r*epr)*R]
    const int32_t* col = p.count + int64_t(r) * epr;
    int carry = 0;
    for (int t0 = 0; t0 * 32 < E; ++t0) {
      const int i = t0 * 32 + lane;
      const int j = i / R, s = i - j * R;
      const int v = i < E ? __ldcg(col + int64_t(s) * E + j) : 0;
      int incl = v;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += u;
      }
      if (i < E) po[i] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    __syncwarp();
    for (int j = lane; j < epr; j += 32) {
      const int start = __ldcg(po + j * R);
      const int end = (j + 1 < epr) ? __ldcg(po + (j + 1) * R) : carry;
      p.recv_per_expert[r * epr + j] = end - start;
    }
    if (lane == 0) p.total_recv[r] = carry;
  }
  grid_sync(bw, G, p.dev_status);

  // ---- D: partition bases, then the tokens -----------------------------------
  if (warp == 0) {   // exclusive scan of the R totals (int64), contiguous per lane
    const int per = (R + 31) / 32, i0 = min(R, lane * per), i1 = min(R, i0 + per);
    int64_t local = 0;
    for (int i = i0; i < i1; ++i) local += __ldcg(p.total_recv + i);
    int64_t incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t u = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += u;
    }
    int64_t run = incl - local;
    for (int i = i0; i < i1; ++i) {
      s_base[i] = run;
      run += __ldcg(p.total_recv + i);
    }
    if (lane == 31) s_base[R] = incl;
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int r = tid; r <= R; r += kThreads) p.rank_recv_base[r] = s_base[r];
    if (tid == 0) p.max_bs[0] = p.bs;
  }
  const int nch = H / 8;
  const int h_align = static_cast<int>(align_up(H, 32));
  const int ntail = static_cast<int>((p.row_bytes - H) / 8);
  const int inv_word = (h_align - H) / 8;
  if constexpr (STAGED && !QUANT) {
    // verbatim: warp 0 alone; lane 0 waits for a token's x row, stores it to
    // the k rows and refills the previous token's stage (its stores have read
    // it once at most one group -- this token's -- is still reading)
    if (warp == 0) {
      int it = 0;
      for (int64_t g = blockIdx.x; g < T; g += G, ++it) {
        int64_t* rows = s_rows2[it & 1];
        const int s = static_cast<int>(g / p.bs);
        for (int kk = lane; kk < k; kk += 32) {
          const int64_t q = g * k + kk;
          const int e = __ldg(p.topk_idx + q);
          int64_t row = -1;
          if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
            row = s_base[e / epr] + __ldcg(p.put_offset + int64_t(e) * R + s) +
                  __ldcg(p.send_idx + q);
            if (row < 0 || row >= p.capacity) {
              set_status(p.dev_status, MOE_ERR_CAPACITY);
              row = -1;
            }
          }
          rows[kk] = row;
        }
        __syncwarp();
        int ab = 0;
        if (lane == 0) {
          const int b = it % kNst;
          if (!mbar_wait_bounded(&mbar[b], static_cast<uint32_t>(it / kNst) & 1u,
                                 kBarrierSpin)) {
            set_status(p.dev_status, MOE_ERR_TIMEOUT);
            ab = 1;
          } else {
            pend[b] = -1;
            for (int kk = 0; kk < k; ++kk)
              if (rows[kk] >= 0)
                bulk_store(p.recv + rows[kk] * p.row_bytes, xs + b * SL.x_stride,
                           static_cast<uint32_t>(p.row_bytes));
            bulk_commit();
            if (it >= 1) {
              bulk_wait_read<1>();
              const int pb = (it - 1) % kNst;
              const int64_t gn = g + int64_t(kNst - 1) * G;   // iteration it - 1 + kNst
              if (gn < T) {
                mbar_arrive_expect_tx(&mbar[pb], xbytes);
                bulk_load(xs + pb * SL.x_stride, p.x + gn * xbytes, xbytes, &mbar[pb]);
                pend[pb] = ((it - 1 + kNst) / kNst) & 1;
              }
            }
          }
        }
        if (__shfl_sync(0xffffffffu, ab, 0)) break;
      }
    }
  } else {
  int it = 0;
  for (int64_t g = blockIdx.x; g < T; g += G, ++it) {
    const int s = static_cast<int>(g / p.bs);
    if (STAGED) s_rows = s_rows2[it & 1];   // the previous token's stores may still read the other
    if (warp == 0) {
      for (int kk = lane; kk < k; kk += 32) {
        const int64_t q = g * k + kk;
        const int e = __ldg(p.topk_idx + q);
        int64_t row = -1;
        if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
          row = s_base[e / epr] + __ldcg(p.put_offset + int64_t(e) * R + s) +
                __ldcg(p.send_idx + q);
          if (row < 0 || row >= p.capacity) {
            set_status(p.dev_status, MOE_ERR_CAPACITY);
            row = -1;
          }
        }
        s_rows[kk] = row;
      }
    }
    if constexpr (STAGED) {   // QUANT here: the verbatim path runs above
      const int b = it & 1;
      const unsigned char* xsb = xs + b * SL.x_stride;
      unsigned char* osb = os + b * SL.o_stride;
      if (tid == issuer && QUANT) bulk_wait_read<1>();   // image b: iteration it-2's stores read it
      if (!mbar_wait_bounded(&mbar[b], static_cast<uint32_t>(it >> 1) & 1u, kBarrierSpin)) {
        set_status(p.dev_status, MOE_ERR_TIMEOUT);
        s_abort = 1;
      }
      if constexpr (QUANT) {
        float amax = 0.0f;
        for (int c = tid; c < nch; c += kThreads) {
          float f[8];
          unpack8<DT>(*reinterpret_cast<const uint4*>(xsb + c * 16), f);
#pragma unroll
          for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
        }
#pragma unroll
        for (int d = 16; d > 0; d >>= 1)
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
        if (lane == 0) s_wmax[warp] = amax;
      }
      __syncthreads();   // (A) maxima, rows and the abort flag visible
      if (s_abort) break;
      if (tid == issuer) pend[b] = -1;
      if constexpr (QUANT) {
        float amax = s_wmax[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, s_wmax[w]);
        const float scale = __fdiv_rn(127.0f, __fadd_rn(amax, 1e-12f));
        const float inv = __fdiv_rn(1.0f, scale);
        for (int c = tid; c < nch; c += kThreads) {
          float f[8];
          unpack8<DT>(*reinterpret_cast<const uint4*>(xsb + c * 16), f);
          uint32_t w2[2] = {0u, 0u};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int qv = __float2int_rn(__fmul_rn(f[j], scale));
            w2[j >> 2] |= (static_cast<uint32_t>(qv) & 0xffu) << (8 * (j & 3));
          }
          *reinterpret_cast<uint2*>(osb + c * 8) = make_uint2(w2[0], w2[1]);
        }
        if (tid < ntail)
          *reinterpret_cast<uint2*>(osb + H + 8 * tid) =
              make_uint2(tid == inv_word ? __float_as_uint(inv) : 0u, 0u);
        fence_proxy_async_smem();
        __syncthreads();   // (B) the image is complete; x stage b is free
      }
      if (tid == issuer) {
        const unsigned char* src = QUANT ? osb : xsb;
        for (int kk = 0; kk < k; ++kk)
          if (s_rows[kk] >= 0)
            bulk_store(p.recv + s_rows[kk] * p.row_bytes, src,
                       static_cast<uint32_t>(p.row_bytes));
        bulk_commit();
        if (!QUANT) bulk_wait_read<0>();   // the stores read x stage b; refill it
        const int64_t g2 = g + 2 * int64_t(G);
        if (g2 < T) {
          mbar_arrive_expect_tx(&mbar[b], xbytes);
          bulk_load(const_cast<unsigned char*>(xsb), p.x + g2 * xbytes, xbytes, &mbar[b]);
          pend[b] = ((it + 2) >> 1) & 1;
        }
      }
      continue;
    } else {
    const uint4* xrow = reinterpret_cast<const uint4*>(p.x + g * int64_t(H) * 2);
    if constexpr (QUANT) {
      float amax = 0.0f;
      for (int c = tid; c < nch; c += kThreads) {
        float f[8];
        unpack8<DT>(ld_stream_16(xrow + c), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
      if (lane == 0) s_wmax[warp] = amax;
      __syncthreads();
      amax = s_wmax[0];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) amax = fmaxf(amax, s_wmax[w]);
      const float scale = __fdiv_rn(127.0f, __fadd_rn(amax, 1e-12f));
      const float inv = __fdiv_rn(1.0f, scale);
      for (int c = tid; c < nch; c += kThreads) {
        float f[8];
        unpack8<DT>(__ldg(xrow + c), f);
        uint32_t w2[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int qv = __float2int_rn(__fmul_rn(f[j], scale));
          w2[j >> 2] |= (static_cast<uint32_t>(qv) & 0xffu) << (8 * (j & 3));
        }
        const uint2 img = make_uint2(w2[0], w2[1]);
        for (int kk = 0; kk < k; ++kk) {
          const int64_t row = s_rows[kk];
          if (row >= 0) *reinterpret_cast<uint2*>(p.recv + row * p.row_bytes + c * 8) = img;
        }
      }
      if (tid < ntail) {
        const uint2 t = make_uint2(tid == inv_word ? __float_as_uint(inv) : 0u, 0u);
        for (int kk = 0; kk < k; ++kk) {
          const int64_t row = s_rows[kk];
          if (row >= 0) *reinterpret_cast<uint2*>(p.recv + row * p.row_bytes + H + 8 * tid) = t;
        }
      }
    } else {
      __syncthreads();   // s_rows
      for (int c = tid; c < nch; c += kThreads) {
        const uint4 v = ld_stream_16(xrow + c);
        for (int kk = 0; kk < k; ++kk) {
          const int64_t row = s_rows[kk];
          if (row >= 0) reinterpret_cast<uint4*>(p.recv + row * p.row_bytes)[c] = v;
        }
      }
    }
    }
    __syncthreads();   // s_rows and s_wmax are reused by the next token
  }
  }
  if (STAGED && tid == issuer) {
    bulk_wait_all<0>();   // stores done before shared memory goes away
    for (int st = 0; st < kNst; ++st)   // only after an abort: loads still in flight
      if (pend[st] >= 0 &&
          !mbar_wait_bounded(&mbar[st], static_cast<uint32_t>(pend[st]), kBarrierSpin))
        set_status(p.dev_status, MOE_ERR_TIMEOUT);
  }
}

int tiles_per_rank_of(const Shape& s) {
  return static_cast<int>((int64_t(s.bs) * s.k + kTile - 1) / kTile);
}

constexpr int64_t kStagedSmemMax = 110 * 1024;   // two CTAs per SM still fit

template <int DT, bool QUANT, bool STAGED, int CPS>
cudaError_t launch_t(const Shape& s, Params p, cudaStream_t st) {
  auto kernel = fused_dispatch_kernel<DT, QUANT, STAGED, CPS>;
  const size_t smem = static_cast<size_t>(
      fused_smem(s.R, s.E(), s.H, p.row_bytes, STAGED, QUANT).bytes);
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e == cudaSuccess)
    e = kernel_blocks_per_sm(reinterpret_cast<const void*>(kernel), kThreads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  // a CTA per token (or tile), few enough for a cheap barrier; all co-resident
  const int64_t want = std::max<int64_t>(p.num_tiles, s.T());
  const int grid = static_cast<int>(std::max<int64_t>(
      1, std::min<int64_t>(want, int64_t(std::min(per_sm, CPS)) * sms)));
  void* args[] = {&p};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kernel), dim3(grid),
                                     dim3(kThreads), args, smem, st);
}

template <int DT>
cudaError_t launch_dt(const Shape& s, Params p, bool quant, bool staged, bool wide,
                      cudaStream_t st) {
  if (quant) {
    if (!staged) return launch_t<DT, true, false, 2>(s, p, st);
    return wide ? launch_t<DT, true, true, 2>(s, p, st) : launch_t<DT, true, true, 4>(s, p, st);
  }
  if (!staged) return launch_t<DT, false, false, 2>(s, p, st);
  return wide ? launch_t<DT, false, true, 2>(s, p, st) : launch_t<DT, false, true, 3>(s, p, st);
}

}  // namespace

size_t fused_workspace_bytes(const Shape& s) {
  return static_cast<size_t>(64 + int64_t(s.R) * tiles_per_rank_of(s) * s.E() * 4);
}

cudaError_t launch_fused_dispatch(const Shape& s, const void* x, const int32_t* topk_idx,
                                  bool quant, int32_t* count, int32_t* rank_send,
                                  int32_t* send_idx, int32_t* put_offset,
                                  int32_t* total_recv, int64_t* rank_recv_base,
                                  int32_t* recv_per_expert, int32_t* max_bs, void* recv,
                                  int64_t row_bytes, int64_t capacity, void* workspace,
                                  int32_t* dev_status, cudaStream_t st) {
  Params p;
  p.x = static_cast<const unsigned char*>(x);
  p.topk_idx = topk_idx;
  p.R = s.R;
  p.bs = s.bs;
  p.k = s.k;
  p.epr = s.epr;
  p.H = s.H;
  p.tiles_per_rank = tiles_per_rank_of(s);
  p.num_tiles = s.R * p.tiles_per_rank;
  p.count = count;
  p.rank_send = rank_send;
  p.send_idx = send_idx;
  p.put_offset = put_offset;
  p.total_recv = total_recv;
  p.rank_recv_base = rank_recv_base;
  p.recv_per_expert = recv_per_expert;
  p.max_bs = max_bs;
  p.recv = static_cast<unsigned char*>(recv);
  p.row_bytes = row_bytes;
  p.capacity = capacity;
  p.workspace = workspace;
  p.dev_status = dev_status;
  const bool staged =
      fused_smem(s.R, s.E(), s.H, row_bytes, true, quant).bytes <= kStagedSmemMax;
  const bool wide = int64_t(s.H) * 2 >= 12 * 1024;
  return s.dtype == MOE_BF16 ? launch_dt<MOE_BF16>(s, p, quant, staged, wide, st)
                             : launch_dt<MOE_FP16>(s, p, quant, staged, wide, st);
}

}  // namespace moe_ep
