// combine_quant.cu -- stage 4 over INT8 expert outputs: the dequantisation
// that the pipeline diagram (UMDK/CAM deep analysis v2, section 2.1) adds to
// stage 4, on top of section 2.6's ReadBufferAndWeightedSum.
//
// Each expert-output row is a dispatched-style INT8 row image (codes, fp32
// 1/scale at align32(H)).  Every element is dequantised as float(q) *
// (1/scale) (one rounding) before the combine's multiply-then-add
// (__fmul_rn / __fadd_rn, k in order), then rounded to the token dtype.
//
// Per element: a byte permute and a subtraction give the code as a float
// (see code_raw), then two multiplies and an add; these run as packed fp32x2
// operations on pairs of elements (mul2_rn / add2_rn, bit-identical to the
// scalar ones), which halves the arithmetic's instruction count.
//
// Work is split per warp, with no block barrier: a work item is one token,
// or a contiguous part of its hidden dimension when that evens out the last
// round over the grid's warps.  The warp resolves the item's k rows, weights
// and 1/scales into its own shared-memory table, then each lane walks
// 8-code chunks of the item (one 8-byte load per row; all k rows of a chunk
// in one batch when k <= 8, batches of 8 rows otherwise), issuing the next
// (chunk, batch)'s loads before it computes the current one.  Rows are half
// the bytes of bf16 rows.
#include <algorithm>

#include "moe_ep_internal.cuh"

namespace moe_ep {

namespace {

constexpr int kCqWarps = 8;   // warps per CTA, each on its own work item

__device__ __forceinline__ uint2 ld_stream_8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

// The INT8 code in byte i of w as a float, exactly, without the conversion
// pipe (int-to-float runs at a quarter of the FP32 rate, and this kernel
// converts k codes per output): with wb = w ^ 0x80808080 the byte holds
// u = q + 128 in 0..255; a byte permute places it under the exponent of 2^23
// (bits 0x4B0000uu = 2^23 + u, exact), and subtracting 2^23 + 128 leaves q
// (an exact fp32 subtraction of integers below 2^24).
template <int I>
__device__ __forceinline__ float code_raw(uint32_t wb) {
  return __uint_as_float(__byte_perm(wb, 0x4B000000u, 0x7650 + I));
}

// One row of the warp's table: the row's first byte (nullptr for padding or
// a rejected pair), its weight and its 1/scale (both 0 then).
struct __align__(16) RowRef {
  const unsigned char* p;
  float w;
  float inv;
};

// KB: rows per batch.  MULTI = false: KB == k (one batch, no padding).
// MULTI = true: KB = 8, k > 8 split into batches, the last one padded.
// Three CTAs per SM (at most 80 registers); seven rows per batch need a few
// more registers than that without spilling, so that variant runs two.
template <int DT, int KB, bool MULTI>
__global__ void __launch_bounds__(kCqWarps * 32, KB == 7 ? 2 : 3)
combine_quant_kernel(const unsigned char* __restrict__ yq, int64_t y_rows,
                     int64_t row_bytes, const int32_t* __restrict__ topk_idx,
                     const float* __restrict__ weights,
                     const int32_t* __restrict__ send_idx,
                     const int32_t* __restrict__ put_offset,
                     const int64_t* __restrict__ rank_recv_base, int R, int bs,
                     int k, int epr, int H, int64_t T, int parts,
                     uint4* __restrict__ out, int32_t* dev_status, float neg_zero) {
  __shared__ RowRef s_ref[kCqWarps][MOE_EP_MAX_TOPK];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  RowRef* ref = s_ref[warp];
  const int E = R * epr;
  const int nch = H / 8;                         // 8-code chunks per row
  const int64_t h_align = align_up(H, 32);
  const int nb = MULTI ? (k + KB - 1) / KB : 1;
  const int64_t items = T * parts;
  const int64_t nwarps = int64_t(gridDim.x) * kCqWarps;

  for (int64_t item = int64_t(blockIdx.x) * kCqWarps + warp; item < items; item += nwarps) {
    const int64_t g = item / parts;
    const int part = static_cast<int>(item - g * parts);
    const int c0 = static_cast<int>(int64_t(nch) * part / parts);
    const int c1 = static_cast<int>(int64_t(nch) * (part + 1) / parts);
    __syncwarp();                                 // the last item's readers are done
    const int s = static_cast<int>(g / bs);
    for (int kk = lane; kk < nb * KB; kk += 32) {
      RowRef r{nullptr, 0.0f, 0.0f};
      if (kk < k) {
        const int64_t pair = g * k + kk;
        const int e = __ldg(topk_idx + pair);
        const int32_t sidx = __ldg(send_idx + pair);
        const float wt = __ldg(weights + pair);
        if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
          set_status(dev_status, MOE_ERR_EXPERT_ID);
        } else {
          const int64_t row =
              __ldg(rank_recv_base + e / epr) + __ldg(put_offset + int64_t(e) * R + s) + sidx;
          if (row < 0 || row >= y_rows) {
            set_status(dev_status, MOE_ERR_CAPACITY);
          } else {
            r.p = yq + row * row_bytes;
            r.w = wt;
            r.inv = __ldg(reinterpret_cast<const float*>(r.p + h_align));
          }
        }
      }
      ref[kk] = r;
    }
    __syncwarp();

    // A rejected row (p == nullptr) is not loaded; its register keeps older
    // codes, which contribute (q * 0) * 0 = +-0 and leave acc unchanged (acc
    // is never -0: it starts at +0 and a round-to-nearest sum is -0 only
    // when both terms are).
    auto load = [&](int c, int b, uint2 (&v)[KB]) {
#pragma unroll
      for (int j = 0; j < KB; ++j) {
        const unsigned char* p = ref[b * KB + j].p;
        if (p != nullptr) v[j] = ld_stream_8(p + 8 * int64_t(c));
      }
    };
    auto accumulate = [&](int b, const uint2 (&v)[KB], float2 (&acc)[4]) {
#pragma unroll
      for (int j = 0; j < KB; ++j) {
        if (!MULTI || b * KB + j < k) {           // warp-uniform: padding rows skipped
          const float2 wi = *reinterpret_cast<const float2*>(&ref[b * KB + j].w);
          const float2 wk = make_float2(wi.x, wi.x), sk = make_float2(wi.y, wi.y);
          const float2 bias = make_float2(-8388736.0f, -8388736.0f);
          const uint32_t lo = v[j].x ^ 0x80808080u, hi = v[j].y ^ 0x80808080u;
          const float2 q[4] = {add2_rn(make_float2(code_raw<0>(lo), code_raw<1>(lo)), bias),
                               add2_rn(make_float2(code_raw<2>(lo), code_raw<3>(lo)), bias),
                               add2_rn(make_float2(code_raw<0>(hi), code_raw<1>(hi)), bias),
                               add2_rn(make_float2(code_raw<2>(hi), code_raw<3>(hi)), bias)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {   // elements 2e, 2e + 1
            const float2 t = mul2_rn(q[e], sk, neg_zero);              // dequantise
            acc[e] = add2_rn(acc[e], mul2_rn(t, wk, neg_zero));        // Muls, Add
          }
        }
      }
    };
    uint2 va[KB], vb[KB];
#pragma unroll
    for (int j = 0; j < KB; ++j) va[j] = vb[j] = make_uint2(0u, 0u);
    float2 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = make_float2(0.0f, 0.0f);
    auto packed = [&]() {
      const float f[8] = {acc[0].x, acc[0].y, acc[1].x, acc[1].y,
                          acc[2].x, acc[2].y, acc[3].x, acc[3].y};
      return pack8<DT>(f);
    };
    int c = c0 + lane;
    if (!MULTI) {
      // One batch per chunk; two register sets alternate (chunk c + 32 loads
      // while chunk c computes).
      auto finish = [&](int cc) {
        out[g * nch + cc] = packed();
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[j] = make_float2(0.0f, 0.0f);
      };
      // The chunk after that is requested into L2 (no registers held).
      auto prefetch = [&](int cc) {
#pragma unroll
        for (int j = 0; j < KB; ++j) {
          const unsigned char* p = ref[j].p;
          if (p != nullptr) prefetch_l2(p + 8 * int64_t(cc));
        }
      };
      if (c < c1) load(c, 0, va);
      while (c < c1) {
        if (c + 32 < c1) load(c + 32, 0, vb);
        if (c + 64 < c1) prefetch(c + 64);
        accumulate(0, va, acc);
        finish(c);
        c += 32;
        if (c >= c1) break;
        if (c + 32 < c1) load(c + 32, 0, va);
        if (c + 64 < c1) prefetch(c + 64);
        accumulate(0, vb, acc);
        finish(c);
        c += 32;
      }
    } else {
      // (chunk, batch) positions in order: batch fastest, chunks lane-strided.
      int b = 0;
      if (c < c1) load(c, b, va);
      while (c < c1) {
        int cn = c, bn = b + 1;
        if (bn == nb) {
          bn = 0;
          cn = c + 32;
        }
        if (cn < c1) load(cn, bn, vb);
        accumulate(b, va, acc);
        if (bn == 0) {
          out[g * nch + c] = packed();
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[j] = make_float2(0.0f, 0.0f);
        }
        c = cn;
        b = bn;
#pragma unroll
        for (int j = 0; j < KB; ++j) va[j] = vb[j];
      }
    }
  }
}

// Parts per token: the smallest split (1, 2, 4 or 8; each part at least 32
// chunks) whose last round over the grid's warps is at least 97% full, else
// the fullest.
int parts_for(int64_t T, int nch, int64_t warps) {
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= 8; s *= 2) {
    if (s > 1 && nch / s < 32) break;
    const int64_t n = T * s;
    const int64_t rounds = (n + warps - 1) / warps;
    const double eff = double(n) / double(rounds * warps);
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = s;
    }
    if (eff >= 0.97) break;
  }
  return best;
}

template <int DT, int KB, bool MULTI>
cudaError_t launch_quant_t(const Shape& s, const void* yq, int64_t y_rows,
                           const int32_t* topk_idx, const float* weights,
                           const int32_t* send_idx, const int32_t* put_offset,
                           const int64_t* rank_recv_base, void* out,
                           int32_t* dev_status, cudaStream_t st) {
  constexpr int threads = kCqWarps * 32;
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = current_device_sms(&dev, &sms);
  if (e == cudaSuccess)
    e = kernel_blocks_per_sm(reinterpret_cast<const void*>(combine_quant_kernel<DT, KB, MULTI>),
                             threads, 0, &per_sm);
  if (e != cudaSuccess) return e;
  const int64_t max_ctas = int64_t(std::max(1, per_sm)) * sms;
  const int parts = parts_for(s.T(), s.H / 8, max_ctas * kCqWarps);
  const int64_t items = s.T() * parts;
  const int64_t grid = std::min<int64_t>((items + kCqWarps - 1) / kCqWarps, max_ctas);
  combine_quant_kernel<DT, KB, MULTI><<<static_cast<unsigned>(grid), threads, 0, st>>>(
      static_cast<const unsigned char*>(yq), y_rows, align_up(s.H, 32) + 32, topk_idx,
      weights, send_idx, put_offset, rank_recv_base, s.R, s.bs, s.k, s.epr, s.H, s.T(), parts,
      static_cast<uint4*>(out), dev_status, -0.0f);
  return cudaGetLastError();
}

template <int DT>
cudaError_t launch_quant_dt(const Shape& s, const void* yq, int64_t y_rows,
                            const int32_t* topk_idx, const float* weights,
                            const int32_t* send_idx, const int32_t* put_offset,
                            const int64_t* rank_recv_base, void* out, int32_t* dev_status,
                            cudaStream_t st) {
#define MOE_CQ_LAUNCH(KB_, MULTI_)                                                           \
  return launch_quant_t<DT, KB_, MULTI_>(s, yq, y_rows, topk_idx, weights, send_idx,       \
                                         put_offset, rank_recv_base, out, dev_status, st)
  switch (s.k) {
    case 1: MOE_CQ_LAUNCH(1, false);
    case 2: MOE_CQ_LAUNCH(2, false);
    case 3: MOE_CQ_LAUNCH(3, false);
    case 4: MOE_CQ_LAUNCH(4, false);
    case 5: MOE_CQ_LAUNCH(5, false);
    case 6: MOE_CQ_LAUNCH(6, false);
    case 7: MOE_CQ_LAUNCH(7, false);
    case 8: MOE_CQ_LAUNCH(8, false);
    default: MOE_CQ_LAUNCH(8, true);
  }
#undef MOE_CQ_LAUNCH
}

}  // namespace

cudaError_t launch_combine_quant(const Shape& s, const void* yq, int64_t y_rows,
                                 const int32_t* topk_idx, const float* weights,
                                 const int32_t* send_idx, const int32_t* put_offset,
                                 const int64_t* rank_recv_base, void* out,
                                 int32_t* dev_status, cudaStream_t st) {
  if (s.T() == 0) return cudaSuccess;
  if (s.dtype == MOE_BF16)
    return launch_quant_dt<MOE_BF16>(s, yq, y_rows, topk_idx, weights, send_idx,
                                     put_offset, rank_recv_base, out, dev_status, st);
  return launch_quant_dt<MOE_FP16>(s, yq, y_rows, topk_idx, weights, send_idx,
                                   put_offset, rank_recv_base, out, dev_status, st);
}

}  // namespace moe_ep
