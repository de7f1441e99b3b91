// dispatch.cu -- stage 3, dispatch with optional dynamic INT8 quantisation
// (UMDK/CAM deep analysis v2, section 2.5 moe_dispatch_normal_zb and
// QuantProcess).
//
// The page moves each token row through the vector core's unified buffer:
// MTE DMA in, vector quantise, DMA out to each destination's expandXOut.
// The GB300 counterpart of that DMA engine is the TMA bulk-copy unit:
//
//   * a persistent grid walks the tokens; per CTA, x rows arrive in shared
//     memory through cp.async.bulk loads issued one or two tokens ahead
//     (double-buffered stages, mbarrier transaction counts);
//   * INT8 path: compute threads (two 8-element chunks each, kept in
//     registers between the passes) reduce max|x| from shared memory (warp
//     shuffles + one shared step), quantise into a staging row image (codes,
//     zero pad, fp32 1/scale, zero pad), fence the async proxy, and one
//     thread issues the k cp.async.bulk stores of that image to the token's
//     k receive rows -- the k-fold write amplification costs the threads no
//     store instructions;
//   * verbatim path: one warp per CTA; the loaded x row is stored straight
//     from shared memory to the k rows;
//   * the last warp ("producer") resolves the receive rows of the next token
//     (topk_idx -> rank_recv_base / put_offset / send_idx) while the current
//     token is in flight.
//
// Quantisation, element by element: f = fp32(x) (exact); amax = max |f|;
// scale = 127 / (amax + 1e-12f), IEEE add and divide; q = round half to even
// of (f * scale) (one fp32 multiply, then cvt.rni); |q| <= 127, so the
// page's int32 -> int16 -> int8 casts are exact.  1/scale (IEEE divide) goes
// to byte align32(H) of the row, every other byte after the codes is zero.
//
// Expand variant (the fused deep MoE's stage-1 outputs, section 4.3:
// expand_x [M, h] and dynamic_scale [M] as separate arrays): the same codes,
// written as bf16 values (exact) so the tensor-core GEMM reads them directly,
// and 1/scale into a packed fp32 array at the row's index.
#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int kMaxThreads = 1024;
constexpr uint32_t kWaitLimit = 1u << 20;   // mbarrier polls before giving up
constexpr int kSmemBudget = 200 * 1024;     // dynamic smem per CTA, upper bound

// Resolve the k receive rows of token g into rows[] (one warp).
__device__ __forceinline__ void resolve_rows(
    int64_t g, const int32_t* __restrict__ topk_idx,
    const int32_t* __restrict__ send_idx, const int32_t* __restrict__ put_offset,
    const int64_t* __restrict__ rank_recv_base, int R, int bs, int k, int epr,
    int64_t capacity, int64_t* rows, int32_t* dev_status, int lane) {
  const int E = R * epr;
  const int s = static_cast<int>(g / bs);
  for (int kk = lane; kk < k; kk += 32) {
    const int64_t pair = g * k + kk;
    const int e = __ldg(topk_idx + pair);
    const int32_t sidx = __ldg(send_idx + pair);
    int64_t row = -1;
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
      set_status(dev_status, MOE_ERR_EXPERT_ID);
    } else {
      row = __ldg(rank_recv_base + e / epr) + __ldg(put_offset + int64_t(e) * R + s) + sidx;
      if (row < 0 || row >= capacity) {
        set_status(dev_status, MOE_ERR_CAPACITY);
        row = -1;
      }
    }
    rows[kk] = row;
  }
}

struct SmemLayout {
  int x_stride;    // bytes per x stage (16-byte multiple, 128-aligned)
  int o_stride;    // bytes per staging row image
  int bytes;       // total dynamic shared memory
};

// row_bytes: bytes of one output row image (INT8: align32(H) + 32; expand:
// 2H bf16 codes; verbatim: 2H).
__host__ __device__ inline SmemLayout smem_layout(int H, int64_t row_bytes, int stages,
                                                  bool quant) {
  SmemLayout L;
  L.x_stride = static_cast<int>(align_up(int64_t(H) * 2, 128));
  L.o_stride = quant ? static_cast<int>(align_up(row_bytes, 128)) : 0;
  L.bytes = stages * (L.x_stride + L.o_stride) + stages * 8;
  return L;
}

// ---------------------------------------------------------------------------
// INT8 path
// ---------------------------------------------------------------------------
// EXPAND: the codes go out as bf16 values (2H bytes per row) and 1/scale to
// dyn_scale[row]; otherwise the INT8 row image of row_bytes bytes.
// CPT: 8-element chunks per compute thread, held in registers from the max|x|
// pass to the quantising pass (chunks past CPT * compute threads, for very
// wide rows, are read from shared memory again).
template <int DT, int S, bool EXPAND, int CPT>
__global__ void __launch_bounds__(kMaxThreads)
dispatch_quant_kernel(const unsigned char* __restrict__ x,
                      const int32_t* __restrict__ topk_idx,
                      const int32_t* __restrict__ send_idx,
                      const int32_t* __restrict__ put_offset,
                      const int64_t* __restrict__ rank_recv_base, int R, int bs,
                      int k, int epr, int H, int64_t T,
                      unsigned char* __restrict__ recv, int64_t row_bytes,
                      float* __restrict__ dyn_scale, int64_t capacity,
                      int32_t* dev_status) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int64_t s_rows[2][MOE_EP_MAX_TOPK];
  __shared__ float s_wmax[32];
  __shared__ int s_abort;

  const SmemLayout L = smem_layout(H, row_bytes, S, true);
  unsigned char* xbuf = smem;
  unsigned char* obuf = smem + S * L.x_stride;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + S * (L.x_stride + L.o_stride));

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int ncomp = blockDim.x - 32;
  const int ncw = ncomp / 32;
  const bool producer = tid >= ncomp;
  const bool issuer = tid == ncomp;             // lane 0 of the producer warp
  const int nch = H / 8;                        // 8-element chunks
  const uint32_t xbytes = static_cast<uint32_t>(H) * 2u;
  const int h_align = static_cast<int>(align_up(H, 32));
  const int ntail = static_cast<int>((row_bytes - H) / 8);
  const int inv_word = (h_align - H) / 8;
  const int64_t grid = gridDim.x;

  int pend[S];               // issuer: parity of the load in flight per stage
#pragma unroll
  for (int s = 0; s < S; ++s) pend[s] = -1;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&mbar[s], 1);
    fence_mbar_init();
    s_abort = 0;
  }
  __syncthreads();
  if (producer) {
    if (issuer) {
      for (int s = 0; s < S; ++s) {
        const int64_t gs = blockIdx.x + s * grid;
        if (gs < T) {
          mbar_arrive_expect_tx(&mbar[s], xbytes);
          bulk_load(xbuf + s * L.x_stride, x + gs * xbytes, xbytes, &mbar[s]);
          pend[s] = 0;
        }
      }
    }
    resolve_rows(blockIdx.x, topk_idx, send_idx, put_offset, rank_recv_base, R, bs,
                 k, epr, capacity, s_rows[0], dev_status, lane);
  }
  __syncthreads();

  int it = 0;
  float xf[CPT][8];   // this thread's chunks of the current token's x
  for (int64_t g = blockIdx.x; g < T; ++it, g += grid) {
    const int b = it % S;
    const uint32_t parity = static_cast<uint32_t>(it / S) & 1u;
    const unsigned char* xs = xbuf + b * L.x_stride;
    unsigned char* os = obuf + b * L.o_stride;
    if (producer) {
      __syncwarp();   // the issuer is done reading the table refilled here
      const int64_t gn = g + grid;
      if (gn < T)
        resolve_rows(gn, topk_idx, send_idx, put_offset, rank_recv_base, R, bs, k,
                     epr, capacity, s_rows[(it + 1) & 1], dev_status, lane);
      if (issuer) bulk_wait_read<S - 1>();   // staging image b is free again
    } else {
      if (!mbar_wait_bounded(&mbar[b], parity, kWaitLimit)) {
        set_status(dev_status, MOE_ERR_TIMEOUT);
        s_abort = 1;
      }
      float amax = 0.0f;
#pragma unroll
      for (int i = 0; i < CPT; ++i) {
        const int c = tid + i * ncomp;
        if (c < nch) {
          unpack8<DT>(*reinterpret_cast<const uint4*>(xs + c * 16), xf[i]);
#pragma unroll
          for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(xf[i][j]));
        }
      }
      for (int c = tid + CPT * ncomp; c < nch; c += ncomp) {
        float f[8];
        unpack8<DT>(*reinterpret_cast<const uint4*>(xs + c * 16), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
      if (lane == 0) s_wmax[warp] = amax;
    }
    __syncthreads();   // (A) maxima, abort flag and this token's rows visible
    if (s_abort) break;
    if (issuer) pend[b] = -1;   // consumed
    if (!producer) {
      float amax = s_wmax[0];
      for (int w = 1; w < ncw; ++w) amax = fmaxf(amax, s_wmax[w]);
      const float scale = __fdiv_rn(127.0f, __fadd_rn(amax, 1e-12f));
      const float inv = __fdiv_rn(1.0f, scale);
      auto quantise = [&](int c, const float (&f)[8]) {
        if (EXPAND) {   // q as bf16: exact (|q| <= 127 has at most 7 significant bits)
          uint32_t w4[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float q0 = static_cast<float>(__float2int_rn(__fmul_rn(f[2 * j], scale)));
            const float q1 = static_cast<float>(__float2int_rn(__fmul_rn(f[2 * j + 1], scale)));
            w4[j] = (__float_as_uint(q0) >> 16) | (__float_as_uint(q1) & 0xffff0000u);
          }
          *reinterpret_cast<uint4*>(os + c * 16) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        } else {
          uint32_t w2[2] = {0u, 0u};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int q = __float2int_rn(__fmul_rn(f[j], scale));
            w2[j >> 2] |= (static_cast<uint32_t>(q) & 0xffu) << (8 * (j & 3));
          }
          *reinterpret_cast<uint2*>(os + c * 8) = make_uint2(w2[0], w2[1]);
        }
      };
#pragma unroll
      for (int i = 0; i < CPT; ++i)
        if (tid + i * ncomp < nch) quantise(tid + i * ncomp, xf[i]);
      for (int c = tid + CPT * ncomp; c < nch; c += ncomp) {
        float f[8];
        unpack8<DT>(*reinterpret_cast<const uint4*>(xs + c * 16), f);
        quantise(c, f);
      }
      if (EXPAND) {   // 1/scale of this token into each of its k rows' slots
        for (int kk = tid; kk < k; kk += ncomp) {
          const int64_t row = s_rows[it & 1][kk];
          if (row >= 0) dyn_scale[row] = inv;
        }
      } else if (tid < ntail) {   // zero pad to align32(H), fp32 1/scale, zero pad
        *reinterpret_cast<uint2*>(os + H + 8 * tid) =
            make_uint2(tid == inv_word ? __float_as_uint(inv) : 0u, 0u);
      }
      fence_proxy_async_smem();
    }
    __syncthreads();   // (B) the image is complete; x stage b may be refilled
    if (issuer) {
      const int64_t* rows = s_rows[it & 1];
      for (int kk = 0; kk < k; ++kk) {
        const int64_t row = rows[kk];
        if (row >= 0) bulk_store(recv + row * row_bytes, os, static_cast<uint32_t>(row_bytes));
      }
      bulk_commit();
      const int64_t g2 = g + S * grid;
      if (g2 < T) {
        mbar_arrive_expect_tx(&mbar[b], xbytes);
        bulk_load(xbuf + b * L.x_stride, x + g2 * xbytes, xbytes, &mbar[b]);
        pend[b] = static_cast<int>(((it + S) / S) & 1);
        // the row after it starts for L2 now (no stage held; measured: dsv3
        // 372-384 -> 369 us; the verbatim kernel lost with the same prefetch,
        // fp16 208 -> 219 us, so it has none)
        if (g2 + grid < T) bulk_prefetch_l2(x + (g2 + grid) * xbytes, xbytes);
      }
    }
  }

  if (issuer) {
    bulk_wait_all<0>();   // stores done before shared memory goes away
    for (int s = 0; s < S; ++s)   // only after an abort: loads still in flight
      if (pend[s] >= 0 && !mbar_wait_bounded(&mbar[s], pend[s], kWaitLimit))
        set_status(dev_status, MOE_ERR_TIMEOUT);
  }
}

// ---------------------------------------------------------------------------
// verbatim path: one warp per CTA, x rows copied to the k rows by TMA
// ---------------------------------------------------------------------------
template <int S>
__global__ void __launch_bounds__(32)
dispatch_copy_kernel(const unsigned char* __restrict__ x,
                     const int32_t* __restrict__ topk_idx,
                     const int32_t* __restrict__ send_idx,
                     const int32_t* __restrict__ put_offset,
                     const int64_t* __restrict__ rank_recv_base, int R, int bs,
                     int k, int epr, int H, int64_t T,
                     unsigned char* __restrict__ recv, int64_t row_bytes,
                     int64_t capacity, int32_t* dev_status) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int64_t s_rows[MOE_EP_MAX_TOPK];
  const SmemLayout L = smem_layout(H, row_bytes, S, false);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + S * L.x_stride);
  const int lane = threadIdx.x;
  const uint32_t xbytes = static_cast<uint32_t>(H) * 2u;
  const int64_t grid = gridDim.x;
  int pend[2] = {-1, -1};

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&mbar[s], 1);
    fence_mbar_init();
    for (int s = 0; s < S; ++s) {
      const int64_t gs = blockIdx.x + s * grid;
      if (gs < T) {
        mbar_arrive_expect_tx(&mbar[s], xbytes);
        bulk_load(smem + s * L.x_stride, x + gs * xbytes, xbytes, &mbar[s]);
        pend[s] = 0;
      }
    }
  }
  __syncwarp();
  int it = 0;
  for (int64_t g = blockIdx.x; g < T; ++it, g += grid) {
    const int b = it % S;
    resolve_rows(g, topk_idx, send_idx, put_offset, rank_recv_base, R, bs, k, epr,
                 capacity, s_rows, dev_status, lane);
    __syncwarp();
    int abort = 0;
    if (lane == 0) {
      if (!mbar_wait_bounded(&mbar[b], static_cast<uint32_t>(it / S) & 1u, kWaitLimit)) {
        set_status(dev_status, MOE_ERR_TIMEOUT);
        abort = 1;
      } else {
        pend[b] = -1;
        for (int kk = 0; kk < k; ++kk)
          if (s_rows[kk] >= 0)
            bulk_store(recv + s_rows[kk] * row_bytes, smem + b * L.x_stride, xbytes);
        bulk_commit();
        bulk_wait_read<0>();   // stage b is read out; refill it
        const int64_t g2 = g + S * grid;
        if (g2 < T) {
          mbar_arrive_expect_tx(&mbar[b], xbytes);
          bulk_load(smem + b * L.x_stride, x + g2 * xbytes, xbytes, &mbar[b]);
          pend[b] = static_cast<int>(((it + S) / S) & 1);
        }
      }
    }
    if (__shfl_sync(0xffffffffu, abort, 0)) break;
    __syncwarp();   // s_rows is rewritten by the next iteration
  }
  if (lane == 0) {
    bulk_wait_all<0>();
    for (int s = 0; s < S; ++s)
      if (pend[s] >= 0 && !mbar_wait_bounded(&mbar[s], pend[s], kWaitLimit))
        set_status(dev_status, MOE_ERR_TIMEOUT);
  }
}

// ---------------------------------------------------------------------------

template <typename Kernel>
cudaError_t launch_persistent(Kernel kernel, int threads, int smem, int64_t T,
                              int* grid_out) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e == cudaSuccess)
    e = kernel_blocks_per_sm(reinterpret_cast<const void*>(kernel), threads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  *grid_out = static_cast<int>(std::min<int64_t>(T, int64_t(std::max(1, per_sm)) * sms));
  return cudaSuccess;
}

template <int DT, int S, bool EXPAND, int CPT>
cudaError_t launch_quant(const Shape& s, const void* x, const int32_t* topk_idx,
                         const int32_t* send_idx, const int32_t* put_offset,
                         const int64_t* rank_recv_base, void* recv, int64_t row_bytes,
                         float* dyn_scale, int64_t capacity, int32_t* dev_status,
                         cudaStream_t st) {
  const int nch = s.H / 8;
  const int ncomp =
      std::max(32, std::min(kMaxThreads - 32, ((nch + CPT - 1) / CPT + 31) / 32 * 32));
  const int threads = ncomp + 32;
  const int smem = smem_layout(s.H, row_bytes, S, true).bytes;
  int grid = 0;
  cudaError_t e = launch_persistent(dispatch_quant_kernel<DT, S, EXPAND, CPT>, threads, smem,
                                    s.T(), &grid);
  if (e != cudaSuccess) return e;
  dispatch_quant_kernel<DT, S, EXPAND, CPT><<<grid, threads, smem, st>>>(
      static_cast<const unsigned char*>(x), topk_idx, send_idx, put_offset,
      rank_recv_base, s.R, s.bs, s.k, s.epr, s.H, s.T(),
      static_cast<unsigned char*>(recv), row_bytes, dyn_scale, capacity, dev_status);
  return cudaGetLastError();
}

// Two 8-element chunks per compute thread (so H/16 compute threads per
// token, up to 992): measured against four, two was as fast or faster on every
// shape (dsv3 398 -> 374, skew 186 -> 172, maxrank 600 -> 565 us) -- a token's
// critical path (two passes, two block barriers) matters more than CTAs per SM.
constexpr int kCpt = 2;

template <int DT, bool EXPAND>
cudaError_t launch_quant_stages(const Shape& s, const void* x, const int32_t* topk_idx,
                                const int32_t* send_idx, const int32_t* put_offset,
                                const int64_t* rank_recv_base, void* recv,
                                int64_t row_bytes, float* dyn_scale, int64_t capacity,
                                int32_t* dev_status, cudaStream_t st) {
  // two stages (prefetch one token ahead) unless the rows are too wide
  if (smem_layout(s.H, row_bytes, 2, true).bytes <= kSmemBudget)
    return launch_quant<DT, 2, EXPAND, kCpt>(s, x, topk_idx, send_idx, put_offset,
                                             rank_recv_base, recv, row_bytes, dyn_scale,
                                             capacity, dev_status, st);
  return launch_quant<DT, 1, EXPAND, kCpt>(s, x, topk_idx, send_idx, put_offset,
                                           rank_recv_base, recv, row_bytes, dyn_scale,
                                           capacity, dev_status, st);
}

template <int S>
cudaError_t launch_copy(const Shape& s, const void* x, const int32_t* topk_idx,
                        const int32_t* send_idx, const int32_t* put_offset,
                        const int64_t* rank_recv_base, void* recv, int64_t row_bytes,
                        int64_t capacity, int32_t* dev_status, cudaStream_t st) {
  const int smem = smem_layout(s.H, row_bytes, S, false).bytes;
  int grid = 0;
  cudaError_t e = launch_persistent(dispatch_copy_kernel<S>, 32, smem, s.T(), &grid);
  if (e != cudaSuccess) return e;
  dispatch_copy_kernel<S><<<grid, 32, smem, st>>>(
      static_cast<const unsigned char*>(x), topk_idx, send_idx, put_offset,
      rank_recv_base, s.R, s.bs, s.k, s.epr, s.H, s.T(),
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
  if (!quant) {
    // two stages (prefetch one token ahead) unless the rows are too wide
    const bool two = smem_layout(s.H, row_bytes, 2, false).bytes <= kSmemBudget;
    return two ? launch_copy<2>(s, x, topk_idx, send_idx, put_offset, rank_recv_base,
                                recv, row_bytes, capacity_rows, dev_status, st)
               : launch_copy<1>(s, x, topk_idx, send_idx, put_offset, rank_recv_base,
                                recv, row_bytes, capacity_rows, dev_status, st);
  }
  if (s.dtype == MOE_BF16)
    return launch_quant_stages<MOE_BF16, false>(s, x, topk_idx, send_idx, put_offset,
                                                rank_recv_base, recv, row_bytes, nullptr,
                                                capacity_rows, dev_status, st);
  return launch_quant_stages<MOE_FP16, false>(s, x, topk_idx, send_idx, put_offset,
                                              rank_recv_base, recv, row_bytes, nullptr,
                                              capacity_rows, dev_status, st);
}

cudaError_t launch_dispatch_expand(const Shape& s, const void* x, const int32_t* topk_idx,
                                   const int32_t* send_idx, const int32_t* put_offset,
                                   const int64_t* rank_recv_base, void* expand_x,
                                   float* dyn_scale, int64_t capacity_rows,
                                   int32_t* dev_status, cudaStream_t st) {
  if (s.T() == 0) return cudaSuccess;
  const int64_t row_bytes = int64_t(s.H) * 2;
  if (s.dtype == MOE_BF16)
    return launch_quant_stages<MOE_BF16, true>(s, x, topk_idx, send_idx, put_offset,
                                               rank_recv_base, expand_x, row_bytes, dyn_scale,
                                               capacity_rows, dev_status, st);
  return launch_quant_stages<MOE_FP16, true>(s, x, topk_idx, send_idx, put_offset,
                                             rank_recv_base, expand_x, row_bytes, dyn_scale,
                                             capacity_rows, dev_status, st);
}

}  // namespace moe_ep
