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
// When every source rank's pairs fit one tile, A writes the count rows and
// the final send indices itself and B (with its barrier) is skipped.
// Problems small enough for one SM's shared memory run in a separate
// one-CTA kernel with no grid barrier at all (fused_small_kernel below).
//
// The grid barrier is an arrival count and generation in one workspace word
// (see grid_sync); a wait that exceeds its bound (about a second) sets
// MOE_ERR_TIMEOUT and the CTA goes on (every receive-row write is still
// checked against the capacity).  Data written in an earlier phase by
// another CTA is read through L2 (__ldcg).
#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRounds = 8;
constexpr int kTile = kWarps * kRounds * 32;     // 2048 pairs
constexpr uint32_t kBarrierSpin = 1u << 20;
constexpr int kScanBatch = 8;                    // count rows in flight per notify warp
// CTAs per SM (CPS, a template parameter: the register cap that lets them
// all be resident): 2 when x rows are 12 KB or wider, else 4 on the INT8
// path and 3 on the verbatim path (measured fastest per shape).

// Grid barrier state: one 32-bit word in the workspace, the arrival count in
// the low 16 bits and a generation in the high 16 (grids stay far below
// 65536 CTAs).  Thread 0 of each CTA adds 1 (acquire-release); the CTA that
// completes the count adds 0x10000 - n, which in one release operation
// returns the count to zero and advances the generation; the others poll
// (acquire) until the generation moves.  One round trip per CTA plus the
// last one's fire-and-forget add, instead of a generation read, two fences
// and a reset store.  The word is zero at the start and the end of every
// launch that completes.
struct BarrierWs {
  uint32_t word;
  uint32_t pad[15];
};

__device__ void grid_sync(BarrierWs* bw, uint32_t nblocks, int32_t* dev_status) {
  __syncthreads();
  if (nblocks == 1u) return;   // one CTA: the block barrier is the grid barrier
  if (threadIdx.x == 0) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;"
                 : "=r"(old)
                 : "l"(&bw->word)
                 : "memory");
    const uint32_t gen = old >> 16;
    if ((old & 0xffffu) == nblocks - 1u) {
      asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(&bw->word),
                   "r"(0x10000u - nblocks)
                   : "memory");
    } else {
      for (uint32_t spins = 0; (ld_acquire_gpu(&bw->word) >> 16) == gen; ++spins) {
        if (spins >= kBarrierSpin) {
          set_status(dev_status, MOE_ERR_TIMEOUT);
          break;
        }
        __nanosleep(32);
      }
    }
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
  // Every source rank is one tile: phase A's tile histograms are the count
  // rows and its in-tile ranks the final send indices, so phase B, its grid
  // barrier and the send-index fix-up of phase C are skipped.
  const bool single = p.tiles_per_rank == 1;

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
      if (single)   // the rank's only tile: its histogram is the count row
        p.count[int64_t(s) * E + e] = run;
      else
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
  if (!single) {   // (grid-uniform)
    grid_sync(bw, G, p.dev_status);

    // ---- B: per (source rank, expert) scan over the rank's tiles ------------
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
  }
  grid_sync(bw, G, p.dev_status);

  // ---- C: send indices, rank_send, notify ------------------------------------
  // send_idx += the tile's prefix (nothing to add when a rank is one tile);
  // four pairs per thread per step, their loads issued before any store
  for (int64_t q0 = single ? P : gtid; q0 < P; q0 += 4 * gthreads) {
    int e[4], cur[4], pre[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t q = q0 + u * gthreads;
      e[u] = q < P ? __ldg(p.topk_idx + q) : -1;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t q = q0 + u * gthreads;
      cur[u] = pre[u] = 0;
      if (q < P && static_cast<unsigned>(e[u]) < static_cast<unsigned>(E)) {
        const int s = static_cast<int>(q / per_rank);
        const int c = static_cast<int>((q - s * per_rank) / kTile);
        cur[u] = __ldcg(p.send_idx + q);
        pre[u] = __ldcg(agg + (int64_t(s) * p.tiles_per_rank + c) * E + e[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t q = q0 + u * gthreads;
      if (q < P && static_cast<unsigned>(e[u]) < static_cast<unsigned>(E))
        p.send_idx[q] = cur[u] + pre[u];
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
    // the column reads are scattered (one count row per source rank): issue
    // kScanBatch rows of them before scanning, so their latencies overlap
    for (int t0 = 0; t0 * 32 < E; t0 += kScanBatch) {
      int v[kScanBatch];
#pragma unroll
      for (int b = 0; b < kScanBatch; ++b) {
        const int i = (t0 + b) * 32 + lane;
        const int j = i / R, s = i - j * R;
        v[b] = i < E ? __ldcg(col + int64_t(s) * E + j) : 0;
      }
#pragma unroll
      for (int b = 0; b < kScanBatch; ++b) {
        if ((t0 + b) * 32 >= E) break;                // warp-uniform
        const int i = (t0 + b) * 32 + lane;
        int incl = v[b];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, incl, d);
          if (lane >= d) incl += u;
        }
        if (i < E) po[i] = carry + incl - v[b];
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
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
    constexpr int kPer = (MOE_EP_MAX_RANKS + 31) / 32;   // totals per lane, at most
    const int per = (R + 31) / 32, i0 = min(R, lane * per), i1 = min(R, i0 + per);
    int tv[kPer];
    int64_t local = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {   // all of the lane's loads in flight at once
      tv[u] = i0 + u < i1 ? __ldcg(p.total_recv + i0 + u) : 0;
      local += tv[u];
    }
    int64_t incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t u = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += u;
    }
    int64_t run = incl - local;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      if (i0 + u < i1) s_base[i0 + u] = run;
      run += tv[u];
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
          // as moe_dispatch: the next row after it starts for L2 (INT8 path)
          if (QUANT && g2 + G < T) bulk_prefetch_l2(p.x + (g2 + G) * xbytes, xbytes);
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

// ---- one CTA for decode-size batches ----------------------------------------
//
// When the whole problem fits one SM's shared memory, the grid barriers cost
// more than the work: each is a round trip through L2 for every CTA (about
// 2.7 us measured at 32 CTAs), three of them per launch.  This kernel runs
// the same four phases in one CTA of 32 warps with every intermediate in
// shared memory and the block barrier in place of the grid barrier:
//   * x (all T rows) is requested with one cp.async.bulk at kernel start and
//     arrives while the index phases run;
//   * layout: one warp per source rank walks its pairs 32 at a time in
//     order; __match_any_sync groups the lanes holding the same expert, so a
//     pair's send index is the expert's running count plus the popcount of
//     its lower group-mates (stable (token, k) order);
//   * notify: one warp per destination rank scans (local expert, source
//     rank) with shuffles; one warp scans the rank totals;
//   * tokens: one warp per token (x row from shared memory, max|x| by warp
//     shuffles, the same fp32 quantisation as moe_dispatch), each lane
//     storing 8-byte words of the row image (16-byte chunks on the verbatim
//     path) to the token's k rows.
// Results are bit-identical to the multi-CTA kernel's.
constexpr int kSmallWarps = 32;
constexpr int kSmallThreads = kSmallWarps * 32;
constexpr int64_t kSmallMaxXBytes = 64 * 1024;   // x rows in shared memory
constexpr int64_t kSmallMaxPairs = 4096;
constexpr int64_t kSmallMaxCounts = 8192;        // R * E
constexpr int64_t kSmallMaxTokens = 256;

struct SmallSmem {
  int64_t idx, sidx, cnt, po, base, tot, x, bar, bytes;
};
__host__ __device__ inline SmallSmem small_smem(int R, int E, int64_t P, int64_t xbytes) {
  SmallSmem L;
  L.idx = 0;                                          // int32 [P] topk_idx
  L.sidx = align_up(L.idx + 4 * P, 16);               // int32 [P] send_idx
  L.cnt = align_up(L.sidx + 4 * P, 16);               // int32 [R][E] count
  L.po = align_up(L.cnt + 4 * int64_t(R) * E, 16);    // int32 [E*R] put_offset
  L.base = align_up(L.po + 4 * int64_t(R) * E, 16);   // int64 [R+1] partition bases
  L.tot = align_up(L.base + 8 * int64_t(R + 1), 16);  // int32 [R] rank totals
  L.x = align_up(L.tot + 4 * int64_t(R), 16);         // x [T][H] (bulk copy: 16-byte aligned)
  L.bar = align_up(L.x + xbytes, 8);
  L.bytes = L.bar + 8;
  return L;
}

template <int DT, bool QUANT>
__global__ void __launch_bounds__(kSmallThreads, 1)
fused_small_kernel(Params p) {
  extern __shared__ __align__(16) unsigned char smem[];   // same declaration as above
  const int R = p.R, epr = p.epr, k = p.k, H = p.H, E = R * epr;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t per_rank = int64_t(p.bs) * k;
  const int64_t P = per_rank * R;
  const int64_t T = int64_t(R) * p.bs;
  const int64_t xbytes = T * H * 2;
  const SmallSmem L = small_smem(R, E, P, xbytes);
  int32_t* s_idx = reinterpret_cast<int32_t*>(smem + L.idx);
  int32_t* s_sidx = reinterpret_cast<int32_t*>(smem + L.sidx);
  int32_t* s_cnt = reinterpret_cast<int32_t*>(smem + L.cnt);
  int32_t* s_po = reinterpret_cast<int32_t*>(smem + L.po);
  int64_t* s_base = reinterpret_cast<int64_t*>(smem + L.base);
  int32_t* s_tot = reinterpret_cast<int32_t*>(smem + L.tot);
  const unsigned char* xs = smem + L.x;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L.bar);
  __shared__ int s_xok;

  if (tid == 0) {   // all of x, in flight during the index phases
    mbar_init(mbar, 1);
    fence_mbar_init();
    if (xbytes > 0) {
      mbar_arrive_expect_tx(mbar, static_cast<uint32_t>(xbytes));
      bulk_load(smem + L.x, p.x, static_cast<uint32_t>(xbytes), mbar);
    }
  }
  for (int64_t i = tid; i < P; i += kSmallThreads) s_idx[i] = __ldg(p.topk_idx + i);
  for (int64_t i = tid; i < int64_t(R) * E; i += kSmallThreads) s_cnt[i] = 0;
  __syncthreads();

  // ---- layout: one warp per source rank -----------------------------------------
  const unsigned lt = lanemask_lt();
  for (int s = warp; s < R; s += kSmallWarps) {
    const int32_t* idx_r = s_idx + int64_t(s) * per_rank;
    int32_t* sidx_r = s_sidx + int64_t(s) * per_rank;
    int32_t* cnt_r = s_cnt + int64_t(s) * E;
    for (int64_t q0 = 0; q0 < per_rank; q0 += 32) {
      const int64_t q = q0 + lane;
      const int e = q < per_rank ? idx_r[q] : -1;
      const bool valid = q < per_rank && static_cast<unsigned>(e) < static_cast<unsigned>(E);
      if (q < per_rank && !valid) set_status(p.dev_status, MOE_ERR_EXPERT_ID);
      const unsigned grp = __match_any_sync(0xffffffffu, valid ? e : -1 - lane);
      const int base = valid ? cnt_r[e] : 0;
      __syncwarp();
      if (valid && (grp & lt) == 0u) cnt_r[e] = base + __popc(grp);
      __syncwarp();
      if (q < per_rank) sidx_r[q] = valid ? base + __popc(grp & lt) : -1;
    }
  }
  __syncthreads();

  // ---- notify: one warp per destination rank --------------------------------------
  for (int r = warp; r < R; r += kSmallWarps) {
    int32_t* po = s_po + int64_t(r) * E;                // == put_offset[(r*epr)*R ...]
    int carry = 0;
    for (int i0 = 0; i0 < E; i0 += 32) {
      const int i = i0 + lane;
      const int j = i / R, s = i - j * R;
      const int v = i < E ? s_cnt[int64_t(s) * E + r * epr + j] : 0;
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
      const int start = po[j * R];
      const int end = (j + 1 < epr) ? po[(j + 1) * R] : carry;
      p.recv_per_expert[r * epr + j] = end - start;
    }
    if (lane == 0) {
      s_tot[r] = carry;
      p.total_recv[r] = carry;
    }
  }
  // the layout's and the prefix's outputs (coalesced copies of shared memory)
  for (int64_t i = tid; i < P; i += kSmallThreads) p.send_idx[i] = s_sidx[i];
  for (int64_t i = tid; i < int64_t(R) * E; i += kSmallThreads) p.count[i] = s_cnt[i];
  for (int64_t i = tid; i < int64_t(R) * R; i += kSmallThreads) {
    const int s = static_cast<int>(i / R), r = static_cast<int>(i - int64_t(s) * R);
    int sum = 0;
    for (int j = 0; j < epr; ++j) sum += s_cnt[int64_t(s) * E + r * epr + j];
    p.rank_send[i] = sum;
  }
  __syncthreads();   // s_po and s_tot complete
  for (int64_t i = tid; i < int64_t(R) * E; i += kSmallThreads) p.put_offset[i] = s_po[i];
  if (warp == 0) {   // exclusive scan of the rank totals (R <= 32: one per lane)
    const int64_t v = lane < R ? s_tot[lane] : 0;
    int64_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t u = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += u;
    }
    if (lane < R) {
      s_base[lane] = incl - v;
      p.rank_recv_base[lane] = incl - v;
    }
    if (lane == R - 1) {
      s_base[R] = incl;
      p.rank_recv_base[R] = incl;
    }
    if (lane == 0) p.max_bs[0] = p.bs;
    if (lane == 0)   // x has landed (bounded wait)
      s_xok = xbytes == 0 || mbar_wait_bounded(mbar, 0u, kBarrierSpin);
  }
  __syncthreads();
  if (!s_xok) {
    if (tid == 0) {
      set_status(p.dev_status, MOE_ERR_TIMEOUT);
      mbar_wait_bounded(mbar, 0u, kBarrierSpin);   // the copy lands before the CTA retires
    }
    return;
  }

  // ---- tokens: one warp per token ---------------------------------------------------
  const int nch = H / 8;
  const int h_align = static_cast<int>(align_up(H, 32));
  const int ntail = static_cast<int>((p.row_bytes - H) / 8);
  const int inv_word = (h_align - H) / 8;
  for (int64_t g = warp; g < T; g += kSmallWarps) {
    const int s = static_cast<int>(g / p.bs);
    int64_t row_lo = -1, row_hi = -1;   // rows of pairs kk = lane and kk = lane + 32
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int kk = lane + 32 * half;
      if (kk < k) {
        const int64_t q = g * k + kk;
        const int e = s_idx[q];
        int64_t row = -1;
        if (static_cast<unsigned>(e) < static_cast<unsigned>(E)) {
          row = s_base[e / epr] + s_po[int64_t(e) * R + s] + s_sidx[q];
          if (row < 0 || row >= p.capacity) {
            set_status(p.dev_status, MOE_ERR_CAPACITY);
            row = -1;
          }
        }
        if (half == 0) row_lo = row; else row_hi = row;
      }
    }
    const unsigned char* xrow = xs + g * int64_t(H) * 2;
    if constexpr (QUANT) {
      float amax = 0.0f;
      for (int c = lane; c < nch; c += 32) {
        float f[8];
        unpack8<DT>(*reinterpret_cast<const uint4*>(xrow + c * 16), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
      const float scale = __fdiv_rn(127.0f, __fadd_rn(amax, 1e-12f));
      const float inv = __fdiv_rn(1.0f, scale);
      for (int c0 = 0; c0 < nch; c0 += 32) {
        const int c = c0 + lane;
        uint2 img = make_uint2(0u, 0u);
        if (c < nch) {
          float f[8];
          unpack8<DT>(*reinterpret_cast<const uint4*>(xrow + c * 16), f);
          uint32_t w2[2] = {0u, 0u};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int qv = __float2int_rn(__fmul_rn(f[j], scale));
            w2[j >> 2] |= (static_cast<uint32_t>(qv) & 0xffu) << (8 * (j & 3));
          }
          img = make_uint2(w2[0], w2[1]);
        }
        for (int kk = 0; kk < k; ++kk) {
          const int64_t row = __shfl_sync(0xffffffffu, kk < 32 ? row_lo : row_hi, kk & 31);
          if (c < nch && row >= 0)
            *reinterpret_cast<uint2*>(p.recv + row * p.row_bytes + c * 8) = img;
        }
      }
      for (int t0 = 0; t0 < ntail; t0 += 32) {
        const int t = t0 + lane;
        const uint2 w = make_uint2(t == inv_word ? __float_as_uint(inv) : 0u, 0u);
        for (int kk = 0; kk < k; ++kk) {
          const int64_t row = __shfl_sync(0xffffffffu, kk < 32 ? row_lo : row_hi, kk & 31);
          if (t < ntail && row >= 0)
            *reinterpret_cast<uint2*>(p.recv + row * p.row_bytes + H + 8 * t) = w;
        }
      }
    } else {
      for (int c0 = 0; c0 < nch; c0 += 32) {
        const int c = c0 + lane;
        const uint4 v = c < nch ? *reinterpret_cast<const uint4*>(xrow + c * 16)
                                : make_uint4(0u, 0u, 0u, 0u);
        for (int kk = 0; kk < k; ++kk) {
          const int64_t row = __shfl_sync(0xffffffffu, kk < 32 ? row_lo : row_hi, kk & 31);
          if (c < nch && row >= 0)
            reinterpret_cast<uint4*>(p.recv + row * p.row_bytes)[c] = v;
        }
      }
    }
  }
}

bool small_fits(const Shape& s) {
  const int64_t P = int64_t(s.T()) * s.k;
  const int64_t xbytes = int64_t(s.T()) * s.H * 2;
  return s.R <= kSmallWarps && s.T() <= kSmallMaxTokens && P <= kSmallMaxPairs &&
         int64_t(s.R) * s.E() <= kSmallMaxCounts && xbytes <= kSmallMaxXBytes;
}

template <int DT, bool QUANT>
cudaError_t launch_small_t(const Shape& s, const Params& p, cudaStream_t st) {
  auto kernel = fused_small_kernel<DT, QUANT>;
  const int64_t P = int64_t(s.T()) * s.k;
  const size_t smem =
      static_cast<size_t>(small_smem(s.R, s.E(), P, int64_t(s.T()) * s.H * 2).bytes);
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  kernel<<<1, kSmallThreads, smem, st>>>(p);
  return cudaGetLastError();
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
  if (small_fits(s)) {   // the whole problem in one SM: no grid barriers
    if (s.dtype == MOE_BF16)
      return quant ? launch_small_t<MOE_BF16, true>(s, p, st)
                   : launch_small_t<MOE_BF16, false>(s, p, st);
    return quant ? launch_small_t<MOE_FP16, true>(s, p, st)
                 : launch_small_t<MOE_FP16, false>(s, p, st);
  }
  const bool staged =
      fused_smem(s.R, s.E(), s.H, row_bytes, true, quant).bytes <= kStagedSmemMax;
  const bool wide = int64_t(s.H) * 2 >= 12 * 1024;
  return s.dtype == MOE_BF16 ? launch_dt<MOE_BF16>(s, p, quant, staged, wide, st)
                             : launch_dt<MOE_FP16>(s, p, quant, staged, wide, st);
}

}  // namespace moe_ep
