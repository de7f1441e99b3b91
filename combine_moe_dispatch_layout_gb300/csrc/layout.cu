// layout.cu -- stage 1, dispatch layout (UMDK/CAM deep analysis v2, section
// 2.3 moe_dispatch_layout_zb).
//
// The page counts tokens per rank/expert with cross-core atomics and a
// SyncAll per round, then computes each pair's send index in a second pass.
// Here one launch does both, deterministically, without order-dependent
// atomics:
//
//   * the pairs of each source rank are cut into tiles whose size follows the
//     shape (one warp x 8 rounds of 32 pairs when a rank has at most 256
//     pairs, eight warps x 4 rounds up to 1024 pairs, else eight warps x 8
//     rounds); a CTA takes the next tile from an
//     atomic ticket, so a tile only ever waits for tiles that started before
//     it (forward progress without assuming co-residency);
//   * inside a tile each warp walks its contiguous segment 32 pairs at a
//     time, all index loads issued up front; __match_any_sync groups the
//     lanes holding the same expert, so a lane's rank inside the warp
//     segment is a shared-memory counter plus the popcount of its lower
//     group-mates (stable order);
//   * a column scan over the warp counters gives each warp's offset and the
//     tile histogram;
//   * decoupled look-back across the tiles of the same source rank turns the
//     tile histograms into exclusive prefixes (vector-valued: one entry per
//     expert).  One warp polls the status words of up to 32 predecessors at
//     once; the nearest one that has published its inclusive prefix ends the
//     walk, and every thread then adds the vectors in between in one pass.
//     Status words carry a per-launch epoch (the page's "magic" counter,
//     section 2.2.2) so the workspace never needs clearing between calls; the
//     last CTA to finish advances the epoch and resets the ticket.  When a
//     rank's pairs fit in one tile there is nothing to look back on and the
//     workspace is not touched at all.
//
// send_idx[p] = tile prefix[e] + warp offset[e] + rank in warp; the last tile
// of each rank also writes count[s][:] and rank_send[s][:].
#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr uint32_t kStateAgg = 1;   // tile aggregate published
constexpr uint32_t kStateInc = 2;   // inclusive prefix published
constexpr uint32_t kSpinLimit = 1u << 20;   // polls (an L2 round trip each): ~1 s

struct WsHeader {
  uint32_t ticket;   // next tile id
  uint32_t done;     // CTAs finished in this launch
  uint32_t magic;    // launch counter; epoch = magic % 0x3fffffff + 1
  uint32_t pad[13];
};
static_assert(sizeof(WsHeader) == 64, "header is one 64-byte line");

struct WsView {
  WsHeader* hdr;
  uint32_t* status;   // [num_tiles]
  int32_t* agg;       // [num_tiles][E]
  int32_t* inc;       // [num_tiles][E]
};

__host__ __device__ inline WsView ws_view(void* ws, int num_tiles, int E) {
  char* b = static_cast<char*>(ws);
  WsView v;
  v.hdr = reinterpret_cast<WsHeader*>(b);
  v.status = reinterpret_cast<uint32_t*>(b + 64);
  const int64_t vec_off = 64 + align_up(int64_t(num_tiles) * 4, 64);
  v.agg = reinterpret_cast<int32_t*>(b + vec_off);
  v.inc = v.agg + int64_t(num_tiles) * E;
  return v;
}

__device__ __forceinline__ uint32_t make_status(uint32_t epoch, uint32_t st) {
  return (epoch << 2) | st;
}

// Called by one thread of every CTA as its last action: the last CTA of the
// launch advances the epoch (so this launch's status words look stale to the
// next one) and resets the ticket and done counters.
__device__ __forceinline__ void finish_launch(WsHeader* hdr, int num_tiles) {
  __threadfence();
  const uint32_t d = atomicAdd(&hdr->done, 1u);
  if (d == static_cast<uint32_t>(num_tiles) - 1u) {
    hdr->magic = hdr->magic + 1u;
    hdr->ticket = 0u;
    hdr->done = 0u;
    __threadfence();
  }
}

template <int W, int ROUNDS>   // warps per CTA, 32-pair rounds per warp
__global__ void __launch_bounds__(W * 32)
layout_kernel(const int32_t* __restrict__ topk_idx, int R, int epr,
              int64_t pairs_per_rank, int tiles_per_rank, int num_tiles,
              int32_t* __restrict__ count, int32_t* __restrict__ rank_send,
              int32_t* __restrict__ send_idx, void* workspace,
              int32_t* dev_status) {
  constexpr int kWarps = W;
  constexpr int kThreads = W * 32;
  constexpr int kSegment = ROUNDS * 32;     // pairs per warp
  constexpr int kTile = W * kSegment;       // pairs per tile
  extern __shared__ __align__(16) unsigned char smem[];
  const int E = R * epr;
  uint16_t* wcnt = reinterpret_cast<uint16_t*>(smem);            // [W][E]
  int32_t* excl = reinterpret_cast<int32_t*>(smem + align_up(2 * kWarps * E, 16));
  int32_t* tagg = excl + E;                                      // [E]
  __shared__ uint32_t s_tile, s_epoch, s_state;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  WsView ws = ws_view(workspace, num_tiles, E);

  const bool chained = tiles_per_rank > 1;   // look-back needed
  if (tid == 0) {
    if (chained) {
      s_tile = atomicAdd(&ws.hdr->ticket, 1u);
      s_epoch = __ldcg(&ws.hdr->magic) % 0x3fffffffu + 1u;
    } else {
      s_tile = blockIdx.x;   // independent tiles: no ordering needed
      s_epoch = 0u;
    }
  }
  for (int i = tid; i < (kWarps * E + 1) / 2; i += kThreads)   // odd W*E: the last half word too
    reinterpret_cast<uint32_t*>(wcnt)[i] = 0u;
  __syncthreads();

  if (s_tile >= static_cast<uint32_t>(num_tiles)) {
    // a ticket past the grid means the workspace was not zero-filled (or is
    // shared with an overlapping call): touch nothing but the counters
    if (tid == 0) {
      set_status(dev_status, MOE_ERR_WORKSPACE);
      finish_launch(ws.hdr, num_tiles);
    }
    return;
  }
  const int tile = static_cast<int>(s_tile);
  const uint32_t epoch = s_epoch;
  const int s = tile / tiles_per_rank;
  const int c = tile - s * tiles_per_rank;
  const int64_t p0 = int64_t(c) * kTile;
  const int64_t p_end = min(p0 + kTile, pairs_per_rank);
  const int32_t* idx_rank = topk_idx + int64_t(s) * pairs_per_rank;
  int32_t* out_rank = send_idx + int64_t(s) * pairs_per_rank;
  const int64_t seg0 = p0 + int64_t(warp) * kSegment;

  // ---- per-warp stable ranks ------------------------------------------------
  int ev[ROUNDS];
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int64_t p = seg0 + r * 32 + lane;
    ev[r] = (p < p_end) ? __ldg(idx_rank + p) : -1;
  }
  // lane groups of equal experts, all rounds first (independent of each other)
  unsigned grp[ROUNDS];
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int64_t p = seg0 + r * 32 + lane;
    const bool valid = static_cast<unsigned>(ev[r]) < static_cast<unsigned>(E);
    if (p < p_end && !valid) set_status(dev_status, MOE_ERR_EXPERT_ID);
    if (!valid) ev[r] = -1 - lane;   // invalid lanes never group
    grp[r] = __match_any_sync(0xffffffffu, ev[r]);
  }
  // then the running per-warp counters, round by round
  int rk[ROUNDS];
  const unsigned lt = lanemask_lt();
  uint16_t* my_cnt = wcnt + warp * E;
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int e = ev[r];
    const bool valid = e >= 0;
    const int lrank = __popc(grp[r] & lt);
    const int base = valid ? my_cnt[e] : 0;
    __syncwarp();
    if (valid && lrank == 0) my_cnt[e] = static_cast<uint16_t>(base + __popc(grp[r]));
    __syncwarp();
    rk[r] = valid ? base + lrank : -1;
  }
  __syncthreads();

  // ---- warp offsets and tile histogram ---------------------------------------
  for (int e = tid; e < E; e += kThreads) {
    int v[kWarps];
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v[w] = wcnt[w * E + e];
    int run = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      if (kWarps > 1) wcnt[w * E + e] = static_cast<uint16_t>(run);
      run += v[w];
    }
    tagg[e] = run;
    excl[e] = 0;
  }
  __syncthreads();

  // ---- decoupled look-back over the tiles of this source rank ---------------
  if (chained) {
    int32_t* my_vec = (c == 0 ? ws.inc : ws.agg) + int64_t(tile) * E;
    for (int e = tid; e < E; e += kThreads) my_vec[e] = tagg[e];
    __threadfence();
    __syncthreads();
    if (tid == 0)
      st_release_gpu(ws.status + tile, make_status(epoch, c == 0 ? kStateInc : kStateAgg));

    if (c > 0) {
      const int first = tile - c;    // tile 0 of this rank (always publishes INC)
      int hi = tile - 1;             // newest predecessor not yet added
      while (true) {
        // warp 0: lane j watches tile hi - j until it has published something
        if (warp == 0) {
          const int t = hi - lane;
          const bool mine = t >= first;
          uint32_t st = 0;
          bool ok = true;
          for (uint32_t spins = 0;; ++spins) {
            if (mine && st == 0) {
              const uint32_t v = ld_acquire_gpu(ws.status + t);
              if ((v >> 2) == epoch && (v & 3u) != 0) st = v & 3u;
            }
            if (__all_sync(0xffffffffu, !mine || st != 0)) break;
            if (spins >= kSpinLimit) { ok = false; break; }
            __nanosleep(64);
          }
          const unsigned inc = __ballot_sync(0xffffffffu, mine && st == kStateInc);
          const int nvalid = min(32, hi - first + 1);
          if (lane == 0) {   // ok is warp-uniform: the loop exits together
            if (!ok) {
              set_status(dev_status, MOE_ERR_TIMEOUT);
              s_state = 0x40000000u;                        // give up
            } else {
              // the nearest inclusive prefix ends the walk; otherwise all 32
              s_state = inc ? static_cast<uint32_t>(__ffs(inc) - 1) | 0x80000000u
                            : static_cast<uint32_t>(nvalid - 1);
            }
          }
        }
        __syncthreads();
        const uint32_t sv = s_state;
        if (sv & 0x40000000u) break;                      // timed out
        const int last = static_cast<int>(sv & 0x3fffffffu);   // lanes 0..last
        const bool found = (sv & 0x80000000u) != 0;
        // add vectors hi .. hi-last; this thread's (vector, expert) loads are
        // flattened and issued eight at a time so they overlap in flight
        const int slots = (E + kThreads - 1) / kThreads;   // experts per thread
        const int nload = (last + 1) * slots;
        for (int q0 = 0; q0 < nload; q0 += 8) {
          int v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int q = q0 + u;
            const int j = q / slots, e = tid + (q - j * slots) * kThreads;
            v[u] = 0;
            if (q < nload && e < E) {
              const int32_t* src = (found && j == last ? ws.inc : ws.agg) + int64_t(hi - j) * E;
              v[u] = __ldcg(src + e);
            }
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int q = q0 + u;
            const int j = q / slots, e = tid + (q - j * slots) * kThreads;
            if (q < nload && e < E) excl[e] += v[u];
          }
        }
        __syncthreads();   // s_state is rewritten by the next window
        if (found) break;
        hi -= 32;
      }
      // successors whose 32-tile window reaches tile 0 never need this
      // tile's inclusive prefix
      if (c < tiles_per_rank - 1 && tiles_per_rank > 33) {
        int32_t* inc = ws.inc + int64_t(tile) * E;
        for (int e = tid; e < E; e += kThreads) inc[e] = excl[e] + tagg[e];
        __threadfence();
        __syncthreads();
        if (tid == 0) st_release_gpu(ws.status + tile, make_status(epoch, kStateInc));
      }
    }
  }

  // ---- send indices -----------------------------------------------------------
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int64_t p = seg0 + r * 32 + lane;
    if (p < p_end) {
      const int e = ev[r];
      out_rank[p] = rk[r] < 0 ? -1 : excl[e] + (kWarps > 1 ? my_cnt[e] : 0) + rk[r];
    }
  }

  // ---- per-rank totals from the last tile of the rank -----------------------
  if (c == tiles_per_rank - 1) {
    for (int e = tid; e < E; e += kThreads) {
      const int v = excl[e] + tagg[e];
      count[int64_t(s) * E + e] = v;
      tagg[e] = v;
    }
    __syncthreads();
    for (int r = tid; r < R; r += kThreads) {
      int sum = 0;
      for (int j = 0; j < epr; ++j) sum += tagg[r * epr + j];
      rank_send[int64_t(s) * R + r] = sum;
    }
  }

  // ---- the last CTA out advances the epoch and resets the ticket -------------
  if (chained) {
    __syncthreads();
    if (tid == 0) finish_launch(ws.hdr, num_tiles);
  }
}

// Tile geometry from the pairs per rank: (warps, rounds) with tile =
// warps * rounds * 32 pairs.
struct Geometry {
  int warps, rounds;
  int tile() const { return warps * rounds * 32; }
};

// Measured (one launch, L2 flushed, all geometries bit-identical): a tile of
// 2048 pairs as 8 warps x 8 rounds beat 4096-pair tiles (8 x 16) on every
// multi-tile workload (DeepSeek-V3 shape 18.3 -> 16.7 us) -- shorter
// per-warp chains outweigh the longer look-back -- and smaller tiles lost
// again (1024 pairs: 21.3 us); a rank of at most 1024 pairs is one tile of
// 8 warps x 4 rounds (384 ranks x 1024 pairs: 11.0 us, against 22.8 with
// 4096-pair tiles), and a rank of at most 256 pairs one warp.
Geometry geometry_of(const Shape& s) {
  const int64_t per_rank = int64_t(s.bs) * s.k;
  if (per_rank <= 256) return {1, 8};
  if (per_rank <= 1024) return {8, 4};
  return {8, 8};
}

int tiles_per_rank_of(const Shape& s) {
  const int64_t tile = geometry_of(s).tile();
  return static_cast<int>((int64_t(s.bs) * s.k + tile - 1) / tile);
}

size_t smem_bytes(int warps, int E) {
  return static_cast<size_t>(align_up(2 * int64_t(warps) * E, 16) + 8 * int64_t(E));
}

template <int W, int ROUNDS>
cudaError_t launch_t(const Shape& s, const int32_t* topk_idx, int32_t* count,
                     int32_t* rank_send, int32_t* send_idx, void* workspace,
                     int32_t* dev_status, cudaStream_t st) {
  const int tpr = tiles_per_rank_of(s);
  const int num_tiles = s.R * tpr;
  const size_t smem = smem_bytes(W, s.E());
  // opt in above the default 48 KB per block (large E only)
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(layout_kernel<W, ROUNDS>),
                                      smem);
  if (e != cudaSuccess) return e;
  layout_kernel<W, ROUNDS><<<num_tiles, W * 32, smem, st>>>(
      topk_idx, s.R, s.epr, int64_t(s.bs) * s.k, tpr, num_tiles, count,
      rank_send, send_idx, workspace, dev_status);
  return cudaGetLastError();
}

}  // namespace

size_t layout_workspace_bytes(const Shape& s) {
  const int tpr = tiles_per_rank_of(s);
  const int64_t num_tiles = int64_t(s.R) * tpr;
  const int64_t vec = tpr > 1 ? 2 * num_tiles * s.E() * 4 : 0;
  return static_cast<size_t>(64 + align_up(num_tiles * 4, 64) + vec);
}

cudaError_t launch_layout(const Shape& s, const int32_t* topk_idx,
                          int32_t* count, int32_t* rank_send,
                          int32_t* send_idx, void* workspace,
                          int32_t* dev_status, cudaStream_t st) {
  const Geometry g = geometry_of(s);
  if (g.warps == 1)
    return launch_t<1, 8>(s, topk_idx, count, rank_send, send_idx, workspace, dev_status, st);
  if (g.rounds == 4)
    return launch_t<8, 4>(s, topk_idx, count, rank_send, send_idx, workspace, dev_status, st);
  return launch_t<8, 8>(s, topk_idx, count, rank_send, send_idx, workspace, dev_status, st);
}

}  // namespace moe_ep
