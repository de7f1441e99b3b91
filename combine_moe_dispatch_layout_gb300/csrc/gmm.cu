// gmm.cu -- grouped GEMM of the fused deep MoE (UMDK/CAM deep analysis v2,
// sections 4.1 and 4.3: GMM1 and GMM2, INT8 operands with INT32 sums, one weight
// matrix per expert, each expert's rows contiguous in the receive buffer).
//
// sm_103a has no INT8 tensor-core MMA (tcgen05 .kind::i8 is not available on
// this target), so the products run on the bf16 tensor path and stay exact:
//   * an int8 code is exact in bf16, and a product of two codes (|p| <= 2^14)
//     is exact in the fp32 accumulator;
//   * K is split into chunks of 1024: a chunk's partial sums are integers of
//     magnitude <= 1024 * 128 * 128 = 2^24, all exactly representable in fp32,
//     so every accumulation step inside a chunk is exact;
//   * the epilogue converts each chunk's fp32 sums to int32 (exact) and adds
//     the chunks in int32.
// The result is the int32 GEMM bit for bit.
//
// Kernel: persistent CTAs (one per SM) walk 128 x 256 output tiles (the last
// column tile may be ragged: its B rows past the expert are computed from
// the next expert's rows, or zero-filled by TMA, and never stored; tiles of
// one expert together, in blocks of 8 row tiles with the row tile fastest,
// so the expert's weights and rows are reused from L2).  Warp 0 streams 128 x 64 (A) and 256 x 64 (B) bf16 tiles
// into a 4-stage shared-memory ring with TMA (cp.async.bulk.tensor, 128-byte
// swizzle; 192 KB in flight per SM, which the L2 latency needs); warp 1
// allocates all 512 TMEM columns and one elected lane issues tcgen05.mma
// (M = 128, N = 256, K = 16, fp32 accumulate) into one of two 256-column
// accumulators, alternating per K chunk; warps 2-9 drain a finished chunk
// accumulator (tcgen05.ld; a warp reads its TMEM lane quarter, one output row
// per thread, and one half of the columns) into int32 registers while the
// next chunk accumulates, then store the tile's rows.  Every mbarrier wait is
// bounded: a timeout sets MOE_ERR_TIMEOUT and the CTA stops issuing work,
// then waits (bounded again) for the copies, MMAs, commits and stores it
// already issued before it releases TMEM and retires.  A chunk whose K
// blocks were cut short is never handed to the epilogue.  The main-loop
// waits (stage empty / full, accumulator free / final) take their poll
// limit from the launch in a separate test instantiation (POLLS), so that a
// test can make them run out; the production kernel keeps the limit a
// compile-time constant, and the drain waits always use the full bound.
#include <cuda.h>

#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int BM = 128, BN = 256, BK = 64;   // BK bf16 = one 128-byte swizzle row
constexpr int kChunkBlocks = 16;             // 16 x 64 = 1024: exact fp32 partial sums
constexpr int kRasterM = 8;                  // row tiles per raster block (L2 reuse of A)
constexpr uint32_t kTmemCols = 2 * BN;       // two chunk accumulators (all of TMEM)
constexpr int kEpiWarps = 8;                 // 4 TMEM lane quarters x 2 column halves
constexpr int kThreads = 64 + 32 * kEpiWarps;   // TMA warp, MMA warp, epilogue
constexpr int kEpiCols = BN / 2;             // columns per epilogue thread
constexpr uint32_t kTileABytes = BM * BK * 2;
constexpr uint32_t kTileBBytes = BN * BK * 2;
constexpr uint32_t kSpin = kGemmSpin;        // polls per wait (about a second at the least)

// Epilogue stores: each epilogue warp stages 32 rows x 16 columns (2 KB, the
// TMA store box) in shared memory with the 64-byte swizzle and writes it with
// one cp.async.bulk.tensor store.
constexpr int kStoreCols = 16;
constexpr uint32_t kStageBytes = 32 * kStoreCols * 4;

// Dynamic shared memory, from a 1024-byte aligned base: STAGES A tiles,
// STAGES B tiles, the epilogue store buffers, barriers, then the group
// tables.  The block scan that builds the tables borrows the A area before
// the first TMA load.
template <int STAGES>
struct SmemLayout {
  static constexpr uint32_t kOffA = 0;
  static constexpr uint32_t kOffB = kOffA + STAGES * kTileABytes;
  static constexpr uint32_t kOffOut = kOffB + STAGES * kTileBBytes;
  static constexpr uint32_t kOffBar = kOffOut + kEpiWarps * kStageBytes;
  static constexpr uint32_t kOffTables = kOffBar + 256;
  static size_t bytes(int G) {
    return 1024 + kOffTables + size_t(G + 1) * (sizeof(int64_t) + sizeof(int32_t));
  }
};

// ---- tcgen05 / TMA wrappers ---------------------------------------------------

__device__ __forceinline__ void tma_load_2d(uint32_t sdst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(sdst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// shared -> global tile store (clipped at the tensor's bounds), bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t ssrc, int x,
                                             int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(ssrc), "r"(x), "r"(y)
      : "memory");
}

// Shared-memory matrix descriptor: K-major tile, rows of 128 bytes with the
// 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
  uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);   // start address
  d |= uint64_t(1) << 16;                           // leading offset (unused when swizzled)
  d |= uint64_t(1024 >> 4) << 32;                   // stride offset: 8 rows x 128 B
  d |= uint64_t(1) << 46;                           // descriptor version
  d |= uint64_t(2) << 61;                           // 128-byte swizzle
  return d;
}

// Instruction descriptor: bf16 x bf16 -> fp32, both operands K-major.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            (uint32_t(BN >> 3) << 17) | (uint32_t(BM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void prefetch_l1(const void* p) {
  asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// 16 consecutive TMEM columns of this warp's 32 lanes (one row per thread).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]),
        "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- tile bookkeeping ------------------------------------------------------------

// Rows of group g (a negative count is reported and read as 0).
__device__ __forceinline__ int64_t group_count(const int32_t* group_rows, int g,
                                               int32_t* dev_status) {
  const int32_t c = __ldg(group_rows + g);
  if (c < 0 && dev_status) set_status(dev_status, MOE_ERR_INVALID_ARG);
  return c < 0 ? 0 : c;
}

struct Tile {
  int g;          // group (expert)
  int64_t row0;   // first A row of the tile
  int64_t rows;   // valid rows (<= BM)
  int n0;         // first output column
};

__device__ __forceinline__ Tile decode_tile(int64_t t, const int64_t* goff,
                                            const int32_t* tpre, int G, int ntn) {
  int lo = 0, hi = G;                 // largest g with tpre[g] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tpre[mid] <= t) lo = mid; else hi = mid;
  }
  const int g = lo;
  const int64_t cnt = goff[g + 1] - goff[g];
  const int mt = static_cast<int>((cnt + BM - 1) / BM);
  const int local = static_cast<int>(t - tpre[g]);
  // blocks of row tiles: inside a block m is fastest, then n, so the tiles
  // in flight together touch a bounded number of A's row tiles however large
  // the expert is; all blocks have kRasterM row tiles except the last, which
  // takes the remainder too (kRasterM .. 2*kRasterM - 1; an expert of fewer
  // than 2*kRasterM row tiles is one block), so no short block re-reads B
  const int nblk = mt / kRasterM > 0 ? mt / kRasterM : 1;
  const int full = nblk - 1, per_full = kRasterM * ntn;
  const int blk = local / per_full;
  int m, n;
  if (blk < full) {
    const int r = local - blk * per_full;
    m = blk * kRasterM + r % kRasterM;
    n = r / kRasterM;
  } else {
    const int rem = mt - full * kRasterM, r = local - full * per_full;
    m = full * kRasterM + r % rem;
    n = r / rem;
  }
  Tile tl;
  tl.g = g;
  tl.row0 = goff[g] + int64_t(m) * BM;
  const int64_t left = cnt - int64_t(m) * BM;
  tl.rows = left < BM ? left : BM;
  tl.n0 = n * BN;
  return tl;
}

// Epilogue modes.  kOutInt32: c itself.  kOutDequant (the page's "Cast FP32
// -> x weight_scale -> x per_token_scale" after GMM2): y = (fp32(c) *
// col_scale[g][n]) * ts(m), ts(m) the fp32 at row_scale + m *
// row_scale_stride.  kOutSwiGLU (GMM1 with its DeqSwiglu epilogue, section
// 4.8.1; the weights' gate and up rows interleaved, column 2j = gate j,
// 2j + 1 = up j): h[m][j] = swiglu(dequant(c[m][2j]), dequant(c[m][2j+1])),
// N/2 fp32 outputs per row.  Every operation rounds to nearest even.
enum { kOutInt32 = 0, kOutDequant = 1, kOutSwiGLU = 2 };
struct Dequant {
  int mode;
  const float* col_scale;            // [G][N]
  const unsigned char* row_scale;
  int64_t row_scale_stride;          // bytes
};

// One CTA per SM; registers are allocated per SM sub-partition (16 K each),
// and 10 warps put 3 on some of them, so at most 168 registers per thread.
// MODE (kOut*) is a template parameter so each epilogue gets its own
// register allocation.
template <int STAGES, int MODE, bool POLLS>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC,
                    const int32_t* __restrict__ group_rows, int G, int64_t a_rows, int K,
                    int N, int32_t* __restrict__ C, Dequant dq, uint32_t spin_arg,
                    int32_t* dev_status) {
  // the main-loop poll bound: the launch argument only in the test build of
  // the kernel (POLLS); a compile-time constant otherwise
  const uint32_t spin = POLLS ? spin_arg : kSpin;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  using L = SmemLayout<STAGES>;
  constexpr int kStages = STAGES;
  constexpr uint32_t kOffA = L::kOffA, kOffB = L::kOffB;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);
  int64_t* goff = reinterpret_cast<int64_t*>(smem + L::kOffTables);
  int32_t* tpre = reinterpret_cast<int32_t*>(goff + G + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ntn = (N + BN - 1) / BN;

  // ---- group tables: row offsets and tile prefix (block scan over G) ----------
  {
    const int per = (G + kThreads - 1) / kThreads;
    const int g0 = tid * per < G ? tid * per : G, g1 = g0 + per < G ? g0 + per : G;
    int64_t rsum = 0;
    int32_t tsum = 0;
    for (int g = g0; g < g1; ++g) {
      const int64_t c = group_count(group_rows, g, dev_status);
      rsum += c;
      tsum += static_cast<int32_t>((c + BM - 1) / BM) * ntn;
    }
    int64_t* s_r = reinterpret_cast<int64_t*>(smem + kOffA);            // [kThreads]
    int32_t* s_t = reinterpret_cast<int32_t*>(s_r + kThreads);           // [kThreads]
    s_r[tid] = rsum;
    s_t[tid] = tsum;
    __syncthreads();
    if (tid == 0) {
      int64_t r = 0;
      int32_t tt = 0;
      for (int i = 0; i < kThreads; ++i) {
        const int64_t a = s_r[i];
        const int32_t b = s_t[i];
        s_r[i] = r;
        s_t[i] = tt;
        r += a;
        tt += b;
      }
      goff[G] = r;
      tpre[G] = tt;
    }
    __syncthreads();
    int64_t r = s_r[tid];
    int32_t tt = s_t[tid];
    for (int g = g0; g < g1; ++g) {
      goff[g] = r;
      tpre[g] = tt;
      const int64_t c = group_count(group_rows, g, nullptr);
      r += c;
      tt += static_cast<int32_t>((c + BM - 1) / BM) * ntn;
    }
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full + s, 1);
      mbar_init(empty + s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull + b, 1);
      mbar_init(tempty + b, kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {   // TMEM: all 512 columns for this CTA (one CTA per SM)
    __syncwarp();
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t tmem = *tmem_slot;
  const int64_t total_rows = goff[G];
  const int64_t tiles = tpre[G];
  const int nkb = (K + BK - 1) / BK;
  const int nchunks = (nkb + kChunkBlocks - 1) / kChunkBlocks;
  if (total_rows > a_rows) {              // more rows than the A buffer holds
    if (tid == 0) set_status(dev_status, MOE_ERR_CAPACITY);
  } else if (warp == 0) {
    // ---- TMA producer ---------------------------------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, nload = 0;   // nload: stage fills issued
      for (int64_t t = blockIdx.x; t < tiles && !*abort_flag; t += gridDim.x) {
        const Tile tl = decode_tile(t, goff, tpre, G, ntn);
        const int brow = tl.g * N + tl.n0;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(empty + stage, phase ^ 1u, spin)) {
            set_status(dev_status, MOE_ERR_TIMEOUT);
            *abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(full + stage, kTileABytes + kTileBBytes);
          tma_load_2d(smem_addr(smem + kOffA + stage * kTileABytes), &tmA, kb * BK,
                      static_cast<int>(tl.row0), full + stage);
          tma_load_2d(smem_addr(smem + kOffB + stage * kTileBBytes), &tmB, kb * BK, brow,
                      full + stage);
          ++nload;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      // every stage's last MMA read has completed before the CTA retires
      // (a wait that also ends when another role aborts: the MMA issuer then
      // drains its own MMAs)
      for (int s = 0; s < kStages && !*abort_flag; ++s) {
        bool done = false;
        for (uint32_t i = 0; i < kSpin && !done && !*abort_flag; ++i)
          done = mbar_try_wait(empty + stage, phase ^ 1u);
        if (!done && !*abort_flag) {
          set_status(dev_status, MOE_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
      // after a timeout the stages may still be filling: wait (bounded) for
      // the last fill of each stage, fill i being phase i / kStages of
      // full[i % kStages], so no copy lands in shared memory after the CTA
      // has retired
      if (*abort_flag)
        for (uint32_t i = nload > kStages ? nload - kStages : 0; i < nload; ++i)
          mbar_wait_bounded(full + i % kStages, (i / kStages) & 1u, kSpin);
    }
  } else if (warp == 1) {
    // ---- MMA issuer -----------------------------------------------------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, chunk_ctr = 0, ncommit = 0;   // ncommit: stage releases
      bool ok = true;
      for (int64_t t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
        for (int c = 0; ok && c < nchunks; ++c, ++chunk_ctr) {
          const uint32_t b = chunk_ctr & 1u, use = (chunk_ctr >> 1) & 1u;
          if (!mbar_wait_bounded(tempty + b, use ^ 1u, spin) || *abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + b * BN;
          const int kb1 = (c + 1) * kChunkBlocks < nkb ? (c + 1) * kChunkBlocks : nkb;
          for (int kb = c * kChunkBlocks; kb < kb1; ++kb) {
            if (!mbar_wait_bounded(full + stage, phase, spin) || *abort_flag) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = sdesc(smem_addr(smem + kOffA + stage * kTileABytes));
            const uint64_t bd = sdesc(smem_addr(smem + kOffB + stage * kTileBBytes));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)   // +32 bytes along K per step
              mma_bf16(d, ad + 2 * kk, bd + 2 * kk,
                       (kb != c * kChunkBlocks || kk != 0) ? 1u : 0u);
            mma_commit(empty + stage);             // frees the stage when read
            ++ncommit;
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
          }
          if (!ok) break;                          // a cut-short chunk is not final
          mma_commit(tfull + b);                   // the chunk's sums are final
        }
      }
      if (!ok) {
        set_status(dev_status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      if (*abort_flag) {
        // after a timeout, the MMAs already issued finish before TMEM is
        // released: the last stage release (phase k / kStages of
        // empty[k % kStages]) arrives once every earlier MMA of this thread
        // is complete; and the last chunk commit (phase (n-1) / 2 of
        // tfull[(n-1) % 2], n = chunks committed) has landed in shared
        // memory before the CTA can retire
        if (ncommit > 0) {
          const uint32_t k = ncommit - 1;
          if (!mbar_wait_bounded(empty + k % kStages, (k / kStages) & 1u, kSpin))
            set_status(dev_status, MOE_ERR_TIMEOUT);
        }
        if (chunk_ctr > 0) {
          const uint32_t n = chunk_ctr - 1;
          if (!mbar_wait_bounded(tfull + (n & 1u), (n >> 1) & 1u, kSpin))
            set_status(dev_status, MOE_ERR_TIMEOUT);
        }
      }
    }
  } else {
    // ---- epilogue: chunk sums -> int32, tile rows -> C -------------------------
    const int q = warp & 3;                  // TMEM lanes 32q .. 32q+31
    const int half = (warp - 2) >> 2;        // columns half*128 .. half*128+127
    uint32_t chunk_ctr = 0;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
      const Tile tl = decode_tile(t, goff, tpre, G, ntn);
      const int r = q * 32 + lane;
      const int col0 = tl.n0 + half * kEpiCols;
      const int ncols = N - col0;            // a ragged last column tile
      // scales of the dequantising epilogues: pulled into L1 now (no
      // registers held across the chunks), read after the last chunk; lane l
      // reads columns 4l .. 4l+3 of this thread's half
      const float* cs_ptr = MODE != kOutInt32
                                ? dq.col_scale + int64_t(tl.g) * N + col0 + 4 * lane : nullptr;
      const float* ts_ptr = MODE != kOutInt32
                                ? reinterpret_cast<const float*>(
                                      dq.row_scale + (tl.row0 + r) * dq.row_scale_stride)
                                : nullptr;
      if (MODE != kOutInt32) {
        if (4 * lane < ncols) prefetch_l1(cs_ptr);
        if (r < tl.rows) prefetch_l1(ts_ptr);
      }
      int32_t acc[kEpiCols];
#pragma unroll
      for (int j = 0; j < kEpiCols; ++j) acc[j] = 0;
      bool ok = true;
      for (int c = 0; c < nchunks; ++c, ++chunk_ctr) {
        const uint32_t b = chunk_ctr & 1u, use = (chunk_ctr >> 1) & 1u;
        const bool got = mbar_wait_bounded(tfull + b, use, spin) && !*abort_flag;
        if (!__all_sync(0xffffffffu, got)) {   // the warp stays converged
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = tmem + (uint32_t(q * 32) << 16) + b * BN + half * kEpiCols;
#pragma unroll
        for (int cb = 0; cb < kEpiCols / 16; ++cb) {
          uint32_t v[16];
          tmem_ld16(base + cb * 16, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) acc[cb * 16 + j] += __float2int_rn(__uint_as_float(v[j]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty + b);
      }
      if (!ok) {
        if (lane == 0) set_status(dev_status, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      constexpr bool swiglu = MODE == kOutSwiGLU;
      const int nout = swiglu ? N / 2 : N;   // output columns of the matrix
      const int ocol0 = swiglu ? col0 / 2 : col0;
      const int ocols = nout - ocol0;
      constexpr int nvals = swiglu ? kEpiCols / 2 : kEpiCols;   // outputs held per thread
      if (MODE != kOutInt32) {               // dequantise (and SwiGLU) in registers
        const float4 csv = 4 * lane < ncols ? __ldg(reinterpret_cast<const float4*>(cs_ptr))
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
        const float ts = r < tl.rows ? __ldg(ts_ptr) : 0.0f;
#pragma unroll
        for (int j = 0; j < kEpiCols / 4; ++j) {
          const float cv[4] = {__shfl_sync(0xffffffffu, csv.x, j),
                               __shfl_sync(0xffffffffu, csv.y, j),
                               __shfl_sync(0xffffffffu, csv.z, j),
                               __shfl_sync(0xffffffffu, csv.w, j)};
          if (4 * j < ncols) {
            float y[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
              y[i] = __fmul_rn(__fmul_rn(__int2float_rn(acc[4 * j + i]), cv[i]), ts);
            if (swiglu) {                    // (gate, up) pairs -> h, packed to the front
              acc[2 * j] = __float_as_int(swiglu_rn(y[0], y[1]));
              acc[2 * j + 1] = __float_as_int(swiglu_rn(y[2], y[3]));
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) acc[4 * j + i] = __float_as_int(y[i]);
            }
          }
        }
      }
      if (q * 32 + 32 <= tl.rows) {
        // all 32 rows of this warp are the group's: swizzled staging + TMA store
        uint8_t* stg = smem + L::kOffOut + (warp - 2) * kStageBytes;
        const uint32_t sw = (lane >> 1) & 3u;             // 64-byte swizzle of row `lane`
#pragma unroll
        for (int blk = 0; blk < kEpiCols / kStoreCols; ++blk) {
          if (blk * kStoreCols < nvals && blk * kStoreCols < ocols) {
            if (lane == 0) bulk_wait_read<0>();           // the buffer's last store has read it
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 4; ++c)
              *reinterpret_cast<int4*>(stg + lane * 64 + ((c ^ sw) << 4)) =
                  make_int4(acc[blk * 16 + 4 * c], acc[blk * 16 + 4 * c + 1],
                            acc[blk * 16 + 4 * c + 2], acc[blk * 16 + 4 * c + 3]);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmC, smem_addr(stg), ocol0 + blk * kStoreCols,
                           static_cast<int>(tl.row0 + q * 32));
              bulk_commit();
            }
          }
        }
      } else if (r < tl.rows) {              // the group's last rows: plain stores
        int4* dst = reinterpret_cast<int4*>(C + (tl.row0 + r) * int64_t(nout) + ocol0);
#pragma unroll
        for (int j = 0; j < kEpiCols / 4; ++j)
          if (4 * j < nvals && 4 * j < ocols)
            dst[j] = make_int4(acc[4 * j], acc[4 * j + 1], acc[4 * j + 2], acc[4 * j + 3]);
      }
    }
    if (lane == 0) bulk_wait_all<0>();       // every tile store has landed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

// ---- int8 codes -> bf16 ------------------------------------------------------------

__global__ void codes_to_bf16_kernel(const uint8_t* __restrict__ src, int64_t rows,
                                     int64_t stride, int K, uint16_t* __restrict__ dst) {
  const int per_row = K / 8;                       // 8 codes -> 16 bytes of bf16
  const int64_t n = rows * per_row;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row;
    const int c = static_cast<int>(i - r * per_row);
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src + r * stride + 8 * c));
    const uint32_t b[2] = {w.x, w.y};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t word = b[j >> 1] >> (16 * (j & 1));
      const float lo = static_cast<float>(static_cast<int8_t>(word & 0xffu));
      const float hi = static_cast<float>(static_cast<int8_t>((word >> 8) & 0xffu));
      o[j] = narrow_rn<MOE_BF16>(lo) | (narrow_rn<MOE_BF16>(hi) << 16);   // exact
    }
    reinterpret_cast<uint4*>(dst + r * int64_t(K))[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Gate/up interleave of GMM1's weights for the SwiGLU epilogue: output row
// (g, 2j) = input row (g, j) (gate), (g, 2j + 1) = input row (g, I + j) (up),
// converted to bf16; the column scales are permuted the same way.
__global__ void interleave_gate_up_kernel(const uint8_t* __restrict__ w, const float* __restrict__ ws,
                                          int G, int I, int K, uint16_t* __restrict__ wi,
                                          float* __restrict__ wsi) {
  const int per_row = K / 8;
  const int64_t rows = int64_t(G) * 2 * I;
  const int64_t n = rows * per_row;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row;
    const int c = static_cast<int>(i - r * per_row);
    const int64_t g = r / (2 * I);
    const int local = static_cast<int>(r - g * 2 * I);
    const int64_t src = g * 2 * I + ((local & 1) ? I + (local >> 1) : (local >> 1));
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(w + src * K + 8 * c));
    const uint32_t b[2] = {v.x, v.y};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t word = b[j >> 1] >> (16 * (j & 1));
      const float lo = static_cast<float>(static_cast<int8_t>(word & 0xffu));
      const float hi = static_cast<float>(static_cast<int8_t>((word >> 8) & 0xffu));
      o[j] = narrow_rn<MOE_BF16>(lo) | (narrow_rn<MOE_BF16>(hi) << 16);   // exact
    }
    reinterpret_cast<uint4*>(wi + r * int64_t(K))[c] = make_uint4(o[0], o[1], o[2], o[3]);
    if (c == 0) wsi[r] = __ldg(ws + src);
  }
}

// ---- host: tensor maps -------------------------------------------------------------

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t get_encoder(void** fn) {
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  return q == cudaDriverEntryPointSuccess && *fn != nullptr ? cudaSuccess
                                                            : cudaErrorNotSupported;
}

// 32-bit outputs [rows][N]: 32-row x 16-column store boxes, 64-byte swizzle.
cudaError_t encode_out(CUtensorMap* map, void* base, int64_t rows, int N) {
  void* fn = nullptr;
  cudaError_t e = get_encoder(&fn);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[2] = {cuuint64_t(N), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(N) * 4};
  const cuuint32_t box[2] = {cuuint32_t(kStoreCols), 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = reinterpret_cast<EncodeTiled>(fn)(
      map, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, base, dims, strides, box, estr,
      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
      CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_kmajor(CUtensorMap* map, const void* base, int64_t rows, int K,
                          uint32_t box_rows) {
  void* fn = nullptr;
  cudaError_t e = get_encoder(&fn);
  if (e != cudaSuccess) return e;
  const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
  const cuuint32_t box[2] = {cuuint32_t(BK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = reinterpret_cast<EncodeTiled>(fn)(
      map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_codes_to_bf16(const void* src, int64_t rows, int64_t stride, int K,
                                 void* dst, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e != cudaSuccess) return e;
  const int64_t n = rows * (K / 8);
  const int threads = 256;
  const int64_t grid = std::min<int64_t>((n + threads - 1) / threads, int64_t(sms) * 8);
  codes_to_bf16_kernel<<<static_cast<unsigned>(grid), threads, 0, st>>>(
      static_cast<const uint8_t*>(src), rows, stride, K, static_cast<uint16_t*>(dst));
  return cudaGetLastError();
}

int gmm_block_n() { return BN; }

namespace {

template <int STAGES, int MODE, bool POLLS>
cudaError_t launch_polls(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                         const int32_t* group_rows, int G, int64_t a_rows, int K, int N,
                         int32_t* c, const Dequant& dq, uint32_t spin, int32_t* dev_status,
                         int sms, cudaStream_t st) {
  const size_t smem = SmemLayout<STAGES>::bytes(G);
  auto kernel = grouped_gemm_kernel<STAGES, MODE, POLLS>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kernel), smem);
  if (e != cudaSuccess) return e;
  kernel<<<sms, kThreads, smem, st>>>(ma, mb, mc, group_rows, G, a_rows, K, N, c, dq, spin,
                                      dev_status);
  return cudaGetLastError();
}

template <int STAGES, int MODE>
cudaError_t launch_mode(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                        const int32_t* group_rows, int G, int64_t a_rows, int K, int N,
                        int32_t* c, const Dequant& dq, uint32_t spin, int32_t* dev_status,
                        int sms, cudaStream_t st) {
  if (spin == kSpin)
    return launch_polls<STAGES, MODE, false>(ma, mb, mc, group_rows, G, a_rows, K, N, c, dq,
                                             spin, dev_status, sms, st);
  return launch_polls<STAGES, MODE, true>(ma, mb, mc, group_rows, G, a_rows, K, N, c, dq, spin,
                                          dev_status, sms, st);
}

template <int STAGES>
cudaError_t launch_stages(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                          const int32_t* group_rows, int G, int64_t a_rows, int K, int N,
                          int32_t* c, const Dequant& dq, uint32_t spin, int32_t* dev_status,
                          int sms, cudaStream_t st) {
  if (dq.mode == kOutDequant)
    return launch_mode<STAGES, kOutDequant>(ma, mb, mc, group_rows, G, a_rows, K, N, c, dq,
                                            spin, dev_status, sms, st);
  if (dq.mode == kOutSwiGLU)
    return launch_mode<STAGES, kOutSwiGLU>(ma, mb, mc, group_rows, G, a_rows, K, N, c, dq,
                                           spin, dev_status, sms, st);
  return launch_mode<STAGES, kOutInt32>(ma, mb, mc, group_rows, G, a_rows, K, N, c, dq,
                                        spin, dev_status, sms, st);
}

}  // namespace

cudaError_t launch_interleave_gate_up(const void* w, const float* ws, int G, int I, int K,
                                     void* wi, float* wsi, cudaStream_t st) {
  int dev = 0, sms = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e != cudaSuccess) return e;
  const int64_t n = int64_t(G) * 2 * I * (K / 8);
  const int threads = 256;
  const int64_t grid = std::min<int64_t>((n + threads - 1) / threads, int64_t(sms) * 8);
  interleave_gate_up_kernel<<<static_cast<unsigned>(grid), threads, 0, st>>>(
      static_cast<const uint8_t*>(w), ws, G, I, K, static_cast<uint16_t*>(wi), wsi);
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm(const void* a, int64_t a_rows, int K, const void* b, int G,
                                int N, const int32_t* group_rows, void* c, int mode,
                                const float* col_scale, const void* row_scale,
                                int64_t row_scale_stride, int32_t* dev_status,
                                cudaStream_t st, uint32_t main_loop_polls) {
  CUtensorMap ma, mb, mc;
  cudaError_t e = encode_kmajor(&ma, a, a_rows, K, BM);
  if (e == cudaSuccess) e = encode_kmajor(&mb, b, int64_t(G) * N, K, BN);
  if (e == cudaSuccess) e = encode_out(&mc, c, a_rows, mode == kOutSwiGLU ? N / 2 : N);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0, optin = 0;
  e = current_device_sms(&dev, &sms);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  const Dequant dq{mode, col_scale, static_cast<const unsigned char*>(row_scale),
                   row_scale_stride};
  int32_t* out = static_cast<int32_t*>(c);
  // four stages unless the group tables (12 bytes per group) crowd them out
  if (SmemLayout<4>::bytes(G) <= size_t(optin))
    return launch_stages<4>(ma, mb, mc, group_rows, G, a_rows, K, N, out, dq, main_loop_polls,
                            dev_status, sms, st);
  return launch_stages<3>(ma, mb, mc, group_rows, G, a_rows, K, N, out, dq, main_loop_polls,
                          dev_status, sms, st);
}

}  // namespace moe_ep
