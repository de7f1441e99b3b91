// swiglu.cu -- GMM1 epilogue of the fused deep MoE, standalone (UMDK/CAM deep
// analysis v2, section 4.8.1 PerTokenDequantSwiGLU and section 8.7
// int32 sums cast, dequantised, SwiGLU, requantised to INT8).
//
// Row m of the grouped GEMM's int32 accumulator acc [M][2I] becomes one INT8
// row image, in one pass over HBM:
//   v    = fp32(acc) (round to nearest) * weight_scale[col] * token_scale[m]
//   gate = v[j], up = v[I + j]        (left half / right half)
//   h[j] = (gate / (1 + exp(-gate))) * up   (the page's Muls(-1), Exp,
//          Adds(1), Div on the left half; the right half passes through)
//   then the dispatch's dynamic quantisation of h: scale = 127/(amax +
//   1e-12f), q = round-half-even(h * scale), 1/scale at byte align32(I).
// Every step is one fp32 operation rounded to nearest even (explicit _rn
// intrinsics; the unit is built with -fmad=false).  exp is computed by Cody
// and Waite's two-constant range reduction, x = n*ln2 + r with |r| <= ln2/2,
// and the degree-7 Taylor polynomial of e^r in Horner form, scaled by 2^n
// (input clamped to [-87, 88]); the reduction and Horner steps are fused
// multiply-adds.  The CPU oracle evaluates the same textbook method in the
// same order, so results match bit for bit.
//
// Persistent CTAs walk contiguous blocks of rows; each thread owns 8-output
// chunks (two 32-byte loads of the accumulator per chunk), max|h| is reduced with warp
// shuffles and one shared step, and the row image is written with 8-byte
// stores.  HBM-bound: 8I bytes read and align32(I) + 32 written per row.
#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

constexpr int kMaxThreads = 512;
// 8-output chunks per thread: 2 while that fits 512 threads (I <= 8192; more
// warps per SM, measured fastest at I = 2048), else 4 (I <= 16384).

// Where a row's scales come from.  Plain: one weight-scale vector for all
// rows, token scales packed fp32.  Grouped (fused deep MoE): row m belongs to
// the expert g with group_off[g] <= m < group_off[g + 1] and uses
// weight_scale + g * 2I; its token scale is the fp32 at ts_base + m * ts_stride
// (e.g. the 1/scale inside the dispatched row image); rows at or past
// group_off[G] are not written.
struct ScaleSrc {
  const float* weight_scale;
  const int64_t* group_off;   // nullptr: plain
  int G;
  const unsigned char* ts_base;
  int64_t ts_stride;          // bytes
};

// BF16OUT: the codes go out as bf16 values (exact; 2I bytes per row, the
// next GEMM's operand) and 1/scale to out_scale[m]; otherwise the INT8 row
// image of row_bytes bytes.
template <int kCpt, bool BF16OUT>
__global__ void __launch_bounds__(kMaxThreads)
swiglu_quant_kernel(const int32_t* __restrict__ acc, int64_t M, int I, ScaleSrc sc,
                    unsigned char* __restrict__ out, int64_t row_bytes,
                    float* __restrict__ out_scale, float nz) {
  __shared__ float s_wmax[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads / 32;
  const int nch = I / 8;
  const int i_align = static_cast<int>(align_up(I, 32));
  const int ntail = static_cast<int>((row_bytes - I) / 8);
  const int inv_word = (i_align - I) / 8;
  if (sc.group_off) {
    const int64_t rows = __ldg(sc.group_off + sc.G);
    if (rows < M) M = rows;
  }

  // Each CTA takes a contiguous block of rows: neighbouring rows mostly share
  // an expert, so its weight-scale vector stays in L1; the group pointer only
  // moves forward.
  const int64_t per_cta = (M + gridDim.x - 1) / gridDim.x;
  const int64_t m_end = (blockIdx.x + 1) * per_cta < M ? (blockIdx.x + 1) * per_cta : M;
  int grp = 0;
  for (int64_t m = blockIdx.x * per_cta; m < m_end; ++m) {
    const int32_t* row = acc + m * 2 * int64_t(I);
    const float ts = __ldg(reinterpret_cast<const float*>(sc.ts_base + m * sc.ts_stride));
    const float* weight_scale = sc.weight_scale;
    if (sc.group_off) {                  // largest g with group_off[g] <= m
      while (grp + 1 < sc.G && __ldg(sc.group_off + grp + 1) <= m) ++grp;
      weight_scale += int64_t(grp) * 2 * I;
    }
    float h[kCpt][8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kCpt; ++i) {
      const int c = tid + i * nthreads;
      if (c < nch) {
        const uint4 g0 = ld_stream_16(row + 8 * c), g1 = ld_stream_16(row + 8 * c + 4);
        const uint4 u0 = ld_stream_16(row + I + 8 * c), u1 = ld_stream_16(row + I + 8 * c + 4);
        const int32_t gi[8] = {int32_t(g0.x), int32_t(g0.y), int32_t(g0.z), int32_t(g0.w),
                               int32_t(g1.x), int32_t(g1.y), int32_t(g1.z), int32_t(g1.w)};
        const int32_t ui[8] = {int32_t(u0.x), int32_t(u0.y), int32_t(u0.z), int32_t(u0.w),
                               int32_t(u1.x), int32_t(u1.y), int32_t(u1.z), int32_t(u1.w)};
        const float4 wg0 = __ldg(reinterpret_cast<const float4*>(weight_scale + 8 * c));
        const float4 wg1 = __ldg(reinterpret_cast<const float4*>(weight_scale + 8 * c + 4));
        const float4 wu0 = __ldg(reinterpret_cast<const float4*>(weight_scale + I + 8 * c));
        const float4 wu1 = __ldg(reinterpret_cast<const float4*>(weight_scale + I + 8 * c + 4));
        const float wg[8] = {wg0.x, wg0.y, wg0.z, wg0.w, wg1.x, wg1.y, wg1.z, wg1.w};
        const float wu[8] = {wu0.x, wu0.y, wu0.z, wu0.w, wu1.x, wu1.y, wu1.z, wu1.w};
        const float2 ts2 = bcast2(ts);
#pragma unroll
        for (int j = 0; j < 8; j += 2) {   // two outputs per packed operation
          float2 gate = make_float2(__int2float_rn(gi[j]), __int2float_rn(gi[j + 1]));
          gate = mul2_rn(mul2_rn(gate, make_float2(wg[j], wg[j + 1]), nz), ts2, nz);
          float2 up = make_float2(__int2float_rn(ui[j]), __int2float_rn(ui[j + 1]));
          up = mul2_rn(mul2_rn(up, make_float2(wu[j], wu[j + 1]), nz), ts2, nz);
          const float2 hh = swiglu2_rn(gate, up, nz);
          h[i][j] = hh.x;
          h[i][j + 1] = hh.y;
          amax = fmaxf(amax, fabsf(hh.x));
          amax = fmaxf(amax, fabsf(hh.y));
        }
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if (lane == 0) s_wmax[warp] = amax;
    __syncthreads();
    amax = s_wmax[0];
    for (int w = 1; w < nwarps; ++w) amax = fmaxf(amax, s_wmax[w]);
    const float scale = __fdiv_rn(127.0f, __fadd_rn(amax, 1e-12f));
    const float inv = __fdiv_rn(1.0f, scale);
    unsigned char* dst = out + m * row_bytes;
#pragma unroll
    for (int i = 0; i < kCpt; ++i) {
      const int c = tid + i * nthreads;
      if (c < nch) {
        // q = rint(h * scale) in [-127, 127]; after adding kRoundMagic the
        // low byte of the float's bits is q as an int8.
        uint32_t b[8];
        float2 bv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          bv[j] = add2_rn(mul2_rn(make_float2(h[i][2 * j], h[i][2 * j + 1]), bcast2(scale), nz),
                          bcast2(kRoundMagic));
          b[2 * j] = __float_as_uint(bv[j].x);
          b[2 * j + 1] = __float_as_uint(bv[j].y);
        }
        if (BF16OUT) {   // q itself (exact subtraction), then its bf16 bits (exact)
          uint32_t w4[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 q = add2_rn(bv[j], bcast2(-kRoundMagic));
            w4[j] = __byte_perm(__float_as_uint(q.x), __float_as_uint(q.y), 0x7632);
          }
          *reinterpret_cast<uint4*>(dst + 16 * c) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        } else {
          const uint32_t w0 = __byte_perm(__byte_perm(b[0], b[1], 0x0040),
                                          __byte_perm(b[2], b[3], 0x0040), 0x5410);
          const uint32_t w1 = __byte_perm(__byte_perm(b[4], b[5], 0x0040),
                                          __byte_perm(b[6], b[7], 0x0040), 0x5410);
          *reinterpret_cast<uint2*>(dst + 8 * c) = make_uint2(w0, w1);
        }
      }
    }
    if (BF16OUT) {
      if (tid == 0) out_scale[m] = inv;
    } else if (tid < ntail) {
      *reinterpret_cast<uint2*>(dst + I + 8 * tid) =
          make_uint2(tid == inv_word ? __float_as_uint(inv) : 0u, 0u);
    }
    __syncthreads();   // s_wmax is rewritten for the next row
  }
}

// Warp-per-row-block form (I <= kWarpMaxI): each warp takes a contiguous
// block of rows and walks them in 8-output chunks (lane-strided), with the
// next (row, chunk)'s accumulators loaded while the current chunk computes.
// h goes to the warp's shared buffer [I]; max|h| is a warp reduction (no
// block barrier); a second pass over the buffer quantises and stores.
constexpr int kWarpMaxI = 4096;
constexpr int kWarpSmemBudget = 64 * 1024;   // h buffers per CTA

template <bool BF16OUT>
__global__ void __launch_bounds__(256, 3)
swiglu_quant_warp_kernel(const int32_t* __restrict__ acc, int64_t M, int I, ScaleSrc sc,
                         unsigned char* __restrict__ out, int64_t row_bytes,
                         float* __restrict__ out_scale, float nz) {
  extern __shared__ float4 s_hbuf[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
  float* hb = reinterpret_cast<float*>(s_hbuf) + int64_t(warp) * I;
  const int nch = I / 8;
  const int i_align = static_cast<int>(align_up(I, 32));
  const int ntail = static_cast<int>((row_bytes - I) / 8);
  const int inv_word = (i_align - I) / 8;
  if (sc.group_off) {
    const int64_t rows = __ldg(sc.group_off + sc.G);
    if (rows < M) M = rows;
  }
  const int64_t nw = int64_t(gridDim.x) * W;
  const int64_t per = (M + nw - 1) / nw;
  const int64_t m0 = (int64_t(blockIdx.x) * W + warp) * per;
  const int64_t m1 = m0 + per < M ? m0 + per : M;
  if (m0 >= m1) return;                       // no block-level synchronisation below

  // Accumulators of chunk c of row m: gate words g0, g1, up words u0, u1.
  struct Acc { uint4 g0, g1, u0, u1; };
  auto load = [&](int64_t m, int c, Acc& a) {
    const int32_t* row = acc + m * 2 * int64_t(I);
    a.g0 = ld_stream_16(row + 8 * c);
    a.g1 = ld_stream_16(row + 8 * c + 4);
    a.u0 = ld_stream_16(row + I + 8 * c);
    a.u1 = ld_stream_16(row + I + 8 * c + 4);
  };

  int grp = 0;
  int64_t pm = m0;                             // position of `cur`
  int pc = lane;
  Acc cur{}, nxt{};
  if (pc < nch) load(pm, pc, cur);
  for (int64_t m = m0; m < m1; ++m) {
    const float ts = __ldg(reinterpret_cast<const float*>(sc.ts_base + m * sc.ts_stride));
    const float* weight_scale = sc.weight_scale;
    if (sc.group_off) {                        // largest g with group_off[g] <= m
      while (grp + 1 < sc.G && __ldg(sc.group_off + grp + 1) <= m) ++grp;
      weight_scale += int64_t(grp) * 2 * I;
    }
    float amax = 0.0f;
    for (int c = lane; c < nch; c += 32) {
      // Prefetch the lane's next position: the next chunk of this row, else
      // its first chunk of the next row.
      int64_t qm = pm;
      int qc = pc + 32;
      if (qc >= nch) {
        qc = lane;
        ++qm;
      }
      if (qm < m1) load(qm, qc, nxt);
      {   // and the position after that into L2 (no registers held)
        int64_t rm = qm;
        int rc = qc + 32;
        if (rc >= nch) {
          rc = lane;
          ++rm;
        }
        if (rm < m1) {
          const int32_t* row = acc + rm * 2 * int64_t(I);
          prefetch_l2(row + 8 * rc);
          prefetch_l2(row + I + 8 * rc);
        }
      }
      const int32_t gi[8] = {int32_t(cur.g0.x), int32_t(cur.g0.y), int32_t(cur.g0.z),
                             int32_t(cur.g0.w), int32_t(cur.g1.x), int32_t(cur.g1.y),
                             int32_t(cur.g1.z), int32_t(cur.g1.w)};
      const int32_t ui[8] = {int32_t(cur.u0.x), int32_t(cur.u0.y), int32_t(cur.u0.z),
                             int32_t(cur.u0.w), int32_t(cur.u1.x), int32_t(cur.u1.y),
                             int32_t(cur.u1.z), int32_t(cur.u1.w)};
      const float4 wg0 = __ldg(reinterpret_cast<const float4*>(weight_scale + 8 * c));
      const float4 wg1 = __ldg(reinterpret_cast<const float4*>(weight_scale + 8 * c + 4));
      const float4 wu0 = __ldg(reinterpret_cast<const float4*>(weight_scale + I + 8 * c));
      const float4 wu1 = __ldg(reinterpret_cast<const float4*>(weight_scale + I + 8 * c + 4));
      const float wg[8] = {wg0.x, wg0.y, wg0.z, wg0.w, wg1.x, wg1.y, wg1.z, wg1.w};
      const float wu[8] = {wu0.x, wu0.y, wu0.z, wu0.w, wu1.x, wu1.y, wu1.z, wu1.w};
      float h[8];
      const float2 ts2 = bcast2(ts);
#pragma unroll
      for (int j = 0; j < 8; j += 2) {   // two outputs per packed operation
        float2 gate = make_float2(__int2float_rn(gi[j]), __int2float_rn(gi[j + 1]));
        gate = mul2_rn(mul2_rn(gate, make_float2(wg[j], wg[j + 1]), nz), ts2, nz);
        float2 up = make_float2(__int2float_rn(ui[j]), __int2float_rn(ui[j + 1]));
        up = mul2_rn(mul2_rn(up, make_float2(wu[j], wu[j + 1]), nz), ts2, nz);
        const float2 hh = swiglu2_rn(gate, up, nz);
        h[j] = hh.x;
        h[j + 1] = hh.y;
        amax = fmaxf(amax, fabsf(hh.x));
        amax = fmaxf(amax, fabsf(hh.y));
      }
      *reinterpret_cast<float4*>(hb + 8 * c) = make_float4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<float4*>(hb + 8 * c + 4) = make_float4(h[4], h[5], h[6], h[7]);
      pm = qm;
      pc = qc;
      cur = nxt;
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    const float scale = __fdiv_rn(127.0f, __fadd_rn(amax, 1e-12f));
    const float inv = __fdiv_rn(1.0f, scale);
    unsigned char* dst = out + m * row_bytes;
    for (int c = lane; c < nch; c += 32) {
      const float4 h0 = *reinterpret_cast<const float4*>(hb + 8 * c);
      const float4 h1 = *reinterpret_cast<const float4*>(hb + 8 * c + 4);
      const float h[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
      // q = rint(h * scale) in [-127, 127]; after adding kRoundMagic the low
      // byte of the float's bits is q as an int8.
      uint32_t b[8];
      float2 bv[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bv[j] = add2_rn(mul2_rn(make_float2(h[2 * j], h[2 * j + 1]), bcast2(scale), nz),
                        bcast2(kRoundMagic));
        b[2 * j] = __float_as_uint(bv[j].x);
        b[2 * j + 1] = __float_as_uint(bv[j].y);
      }
      if (BF16OUT) {   // q itself (exact subtraction), then its bf16 bits (exact)
        uint32_t w4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 q = add2_rn(bv[j], bcast2(-kRoundMagic));
          w4[j] = __byte_perm(__float_as_uint(q.x), __float_as_uint(q.y), 0x7632);
        }
        *reinterpret_cast<uint4*>(dst + 16 * c) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      } else {
        const uint32_t w0 = __byte_perm(__byte_perm(b[0], b[1], 0x0040),
                                        __byte_perm(b[2], b[3], 0x0040), 0x5410);
        const uint32_t w1 = __byte_perm(__byte_perm(b[4], b[5], 0x0040),
                                        __byte_perm(b[6], b[7], 0x0040), 0x5410);
        *reinterpret_cast<uint2*>(dst + 8 * c) = make_uint2(w0, w1);
      }
    }
    if (BF16OUT) {
      if (lane == 0) out_scale[m] = inv;
    } else if (lane < ntail) {
      *reinterpret_cast<uint2*>(dst + I + 8 * lane) =
          make_uint2(lane == inv_word ? __float_as_uint(inv) : 0u, 0u);
    }
    __syncwarp();                              // hb is rewritten for the next row
  }
}

template <bool BF16OUT>
cudaError_t launch_warp_t(const int32_t* acc, int64_t M, int I, const ScaleSrc& sc, void* out,
                          float* out_scale, cudaStream_t st) {
  const int W = std::max(1, std::min(8, kWarpSmemBudget / (4 * I)));
  const int threads = 32 * W;
  const size_t smem = size_t(W) * I * sizeof(float);
  auto kernel = swiglu_quant_warp_kernel<BF16OUT>;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e == cudaSuccess)
    e = kernel_blocks_per_sm(reinterpret_cast<const void*>(kernel), threads, smem, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t grid =
      std::min<int64_t>((M + W - 1) / W, int64_t(std::max(1, per_sm)) * sms);
  kernel<<<static_cast<unsigned>(grid), threads, smem, st>>>(
      acc, M, I, sc, static_cast<unsigned char*>(out),
      BF16OUT ? int64_t(I) * 2 : align_up(I, 32) + 32, out_scale, -0.0f);
  return cudaGetLastError();
}

template <int kCpt, bool BF16OUT>
cudaError_t launch_t(const int32_t* acc, int64_t M, int I, const ScaleSrc& sc, void* out,
                     float* out_scale, cudaStream_t st) {
  const int nch = I / 8;
  const int threads = std::max(32, std::min(kMaxThreads, ((nch + kCpt - 1) / kCpt + 31) / 32 * 32));
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e == cudaSuccess)
    e = kernel_blocks_per_sm(reinterpret_cast<const void*>(swiglu_quant_kernel<kCpt, BF16OUT>),
                             threads, 0, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(M, int64_t(std::max(1, per_sm)) * sms);
  swiglu_quant_kernel<kCpt, BF16OUT><<<static_cast<unsigned>(grid), threads, 0, st>>>(
      acc, M, I, sc, static_cast<unsigned char*>(out),
      BF16OUT ? int64_t(I) * 2 : align_up(I, 32) + 32, out_scale, -0.0f);
  return cudaGetLastError();
}

// Dynamic INT8 quantisation of fp32 rows (the requant half of the GMM1
// epilogue when the GEMM's own epilogue has produced h): per row, amax =
// max |h|, scale = 127/(amax + 1e-12f), q = rint(h * scale); the codes go out
// as bf16 values (exact) and 1/scale to inv_scale[m].  Rows at or past
// group_off[G] (when given) are not written.
template <int kCpt>
__global__ void __launch_bounds__(kMaxThreads)
quant_rows_bf16_kernel(const float* __restrict__ h, int64_t M, int I,
                       const int64_t* __restrict__ group_off, int G,
                       uint16_t* __restrict__ codes, float* __restrict__ inv_scale) {
  __shared__ float s_wmax[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads / 32;
  const int nch = I / 8;
  if (group_off) {
    const int64_t rows = __ldg(group_off + G);
    if (rows < M) M = rows;
  }
  const int64_t per_cta = (M + gridDim.x - 1) / gridDim.x;
  const int64_t m_end = (blockIdx.x + 1) * per_cta < M ? (blockIdx.x + 1) * per_cta : M;
  for (int64_t m = blockIdx.x * per_cta; m < m_end; ++m) {
    const float* row = h + m * int64_t(I);
    float v[kCpt][8];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kCpt; ++i) {
      const int c = tid + i * nthreads;
      if (c < nch) {
        const uint4 a = ld_stream_16(row + 8 * c), b = ld_stream_16(row + 8 * c + 4);
        const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[i][j] = __uint_as_float(u[j]);
          amax = fmaxf(amax, fabsf(v[i][j]));
        }
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
    if (lane == 0) s_wmax[warp] = amax;
    __syncthreads();
    amax = s_wmax[0];
    for (int w = 1; w < nwarps; ++w) amax = fmaxf(amax, s_wmax[w]);
    const float scale = __fdiv_rn(127.0f, __fadd_rn(amax, 1e-12f));
    const float inv = __fdiv_rn(1.0f, scale);
#pragma unroll
    for (int i = 0; i < kCpt; ++i) {
      const int c = tid + i * nthreads;
      if (c < nch) {
        uint32_t w4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {   // q = rint(h * scale) exactly, then its bf16 bits
          const float q0 = __fsub_rn(__fadd_rn(__fmul_rn(v[i][2 * j], scale), kRoundMagic),
                                     kRoundMagic);
          const float q1 = __fsub_rn(__fadd_rn(__fmul_rn(v[i][2 * j + 1], scale), kRoundMagic),
                                     kRoundMagic);
          w4[j] = __byte_perm(__float_as_uint(q0), __float_as_uint(q1), 0x7632);
        }
        *reinterpret_cast<uint4*>(codes + m * int64_t(I) + 8 * c) =
            make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
    }
    if (tid == 0) inv_scale[m] = inv;
    __syncthreads();   // s_wmax is rewritten for the next row
  }
}

template <int kCpt>
cudaError_t launch_quant_rows_t(const float* h, int64_t M, int I, const int64_t* group_off,
                                int G, void* codes, float* inv_scale, cudaStream_t st) {
  const int nch = I / 8;
  const int threads = std::max(32, std::min(kMaxThreads, ((nch + kCpt - 1) / kCpt + 31) / 32 * 32));
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e == cudaSuccess)
    e = kernel_blocks_per_sm(reinterpret_cast<const void*>(quant_rows_bf16_kernel<kCpt>),
                             threads, 0, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t grid = std::min<int64_t>(M, int64_t(std::max(1, per_sm)) * sms);
  quant_rows_bf16_kernel<kCpt><<<static_cast<unsigned>(grid), threads, 0, st>>>(
      h, M, I, group_off, G, static_cast<uint16_t*>(codes), inv_scale);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_rows_bf16(const float* h, int64_t M, int I, const int64_t* group_off,
                                   int G, void* codes, float* inv_scale, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  return I / 8 <= 2 * kMaxThreads
             ? launch_quant_rows_t<2>(h, M, I, group_off, G, codes, inv_scale, st)
             : launch_quant_rows_t<4>(h, M, I, group_off, G, codes, inv_scale, st);
}

cudaError_t launch_swiglu_quant(const int32_t* acc, int64_t M, int I,
                                const float* weight_scale, const float* token_scale,
                                void* out, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const ScaleSrc sc{weight_scale, nullptr, 1,
                    reinterpret_cast<const unsigned char*>(token_scale), 4};
  if (I <= kWarpMaxI) return launch_warp_t<false>(acc, M, I, sc, out, nullptr, st);
  return I / 8 <= 2 * kMaxThreads ? launch_t<2, false>(acc, M, I, sc, out, nullptr, st)
                                  : launch_t<4, false>(acc, M, I, sc, out, nullptr, st);
}

cudaError_t launch_swiglu_quant_grouped(const int32_t* acc, int64_t M, int I,
                                        const float* weight_scale, const int64_t* group_off,
                                        int G, const void* token_scale,
                                        int64_t token_scale_stride, void* out,
                                        float* out_scale, cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const ScaleSrc sc{weight_scale, group_off, G,
                    static_cast<const unsigned char*>(token_scale), token_scale_stride};
  if (out_scale) {
    if (I <= kWarpMaxI) return launch_warp_t<true>(acc, M, I, sc, out, out_scale, st);
    return I / 8 <= 2 * kMaxThreads ? launch_t<2, true>(acc, M, I, sc, out, out_scale, st)
                                    : launch_t<4, true>(acc, M, I, sc, out, out_scale, st);
  }
  if (I <= kWarpMaxI) return launch_warp_t<false>(acc, M, I, sc, out, nullptr, st);
  return I / 8 <= 2 * kMaxThreads ? launch_t<2, false>(acc, M, I, sc, out, nullptr, st)
                                  : launch_t<4, false>(acc, M, I, sc, out, nullptr, st);
}

}  // namespace moe_ep
