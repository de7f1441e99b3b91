// moe_ep_internal.cuh -- device helpers and launcher declarations shared by
// the translation units of libmoe_ep.so (never by the CPU oracle).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_ep.h"

namespace moe_ep {

// ---- small utilities -------------------------------------------------------

__host__ __device__ constexpr int64_t align_up(int64_t v, int64_t a) {
  return (v + a - 1) / a * a;
}

// Records the first error of a launch sequence: 0 -> code, later codes lost.
__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (*reinterpret_cast<volatile int32_t*>(st) == 0) atomicCAS(st, 0, code);
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Streaming 16-byte load that does not allocate in L1 (each x / expert-output
// row is read by exactly one CTA).
// Brings `bytes` (a multiple of 16) from the 16-byte aligned p into L2 with
// one bulk prefetch (no shared memory, no completion to wait for).
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Brings the cache line holding p into L2 (no register, no completion).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint4 ld_stream_16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// ---- bulk asynchronous copies (TMA, no tensor map) and mbarriers -----------
// All addresses 16-byte aligned, sizes multiples of 16 bytes.

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// One bounded poll of phase `parity` (true once that phase has completed).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` at most `limit` polls; false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// global -> shared, completion counted on `bar` (transaction bytes).
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// shared -> global, tracked by bulk groups.
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(ssrc)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N committed groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-bit float <-> fp32.  Widening is exact; narrowing is round to nearest
// even (IEEE), subnormals kept.
template <int DT>
__device__ __forceinline__ float widen(uint32_t bits16);
template <>
__device__ __forceinline__ float widen<MOE_BF16>(uint32_t b) {
  return __uint_as_float(b << 16);
}
template <>
__device__ __forceinline__ float widen<MOE_FP16>(uint32_t b) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
}

template <int DT>
__device__ __forceinline__ uint32_t narrow_rn(float f);
template <>
__device__ __forceinline__ uint32_t narrow_rn<MOE_BF16>(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
template <>
__device__ __forceinline__ uint32_t narrow_rn<MOE_FP16>(float f) {
  return __half_as_ushort(__float2half_rn(f));
}

// The 8 elements of a 16-byte chunk, widened to fp32.
template <int DT>
__device__ __forceinline__ void unpack8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = widen<DT>(w[i] & 0xffffu);
    f[2 * i + 1] = widen<DT>(w[i] >> 16);
  }
}

template <int DT>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = narrow_rn<DT>(f[2 * i]) | (narrow_rn<DT>(f[2 * i + 1]) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---- the SwiGLU step of the GMM1 epilogue (UMDK/CAM deep analysis v2,
// section 4.8.1: Muls(-1), Exp, Adds(1), Div on the gate, times the up value)
// shared by the standalone epilogue kernel and the GEMM's fused epilogue, so
// both evaluate exactly the same operations.

// 1.5 * 2^23: adding it to a float of magnitude below 2^22 rounds that float
// to an integer (ties to even), which then sits in the low mantissa bits.
constexpr float kRoundMagic = 12582912.0f;

// exp by Cody and Waite's two-constant range reduction, x = n ln 2 + r with
// |r| <= ln 2 / 2 (ln 2 = C1 + C2, C1 = 0.693359375 so n*C1 is exact), and
// the degree-7 Taylor polynomial of e^r in Horner form, times 2^n; input
// clamped to [-87, 88].  Every step is one fp32 operation rounded to nearest
// even; the reduction and Horner steps are fused multiply-adds.
// The clamp "if (x > 88) x = 88; if (x < -87) x = -87;" in two instructions:
// min / max with .NaN return NaN when an input is NaN, exactly as the
// comparisons leave a NaN unchanged (plain fminf / fmaxf would return the
// bound), and the bound or x otherwise.
__device__ __forceinline__ float clamp_exp_arg(float x) {
  float y;
  asm("{\n\t.reg .f32 t;\n\tmin.NaN.f32 t, %1, 0f42B00000;\n\t"   // 88
      "max.NaN.f32 %0, t, 0fC2AE0000;\n\t}"                            // -87
      : "=f"(y)
      : "f"(x));
  return y;
}

__device__ __forceinline__ float exp_cody_waite(float x) {
  x = clamp_exp_arg(x);
  const float t = __fmul_rn(x, 1.44269504f);                 // x / ln 2
  const float s = __fadd_rn(t, kRoundMagic);                 // rint(t) in the low bits
  const float n = __fsub_rn(s, kRoundMagic);                 // rint(t), exactly
  float r = __fmaf_rn(-n, 0.693359375f, x);                  // x - n*C1
  r = __fmaf_rn(-n, -2.12194440e-4f, r);                     // - n*C2
  float p = 1.98412698e-4f;                                  // 1/7!
  p = __fmaf_rn(p, r, 1.38888889e-3f);                       // 1/6!
  p = __fmaf_rn(p, r, 8.33333333e-3f);                       // 1/5!
  p = __fmaf_rn(p, r, 4.16666667e-2f);                       // 1/4!
  p = __fmaf_rn(p, r, 1.66666667e-1f);                       // 1/3!
  p = __fmaf_rn(p, r, 0.5f);                                 // 1/2!
  p = __fmaf_rn(p, r, 1.0f);                                 // 1/1!
  p = __fmaf_rn(p, r, 1.0f);                                 // 1/0!
  // n is in -126 .. 127: the low 9 bits of s hold n (two's complement), so
  // (s + 127) << 23 is the bit pattern of 2^n.
  return __fmul_rn(p, __uint_as_float((__float_as_uint(s) + 127u) << 23));
}

// h = (gate / (1 + exp(-gate))) * up, one rounding per operation.
__device__ __forceinline__ float swiglu_rn(float gate, float up) {
  const float e = exp_cody_waite(-gate);
  const float d = __fadd_rn(e, 1.0f);
  const float sg = __fdiv_rn(gate, d);
  return __fmul_rn(sg, up);
}

// ---- packed fp32x2 arithmetic -------------------------------------------------
// Two fp32 operations per instruction (add / fma .rn .f32x2), each half one
// IEEE operation rounded to nearest even, subnormals kept.  The code
// generator merges a packed multiply followed by a packed add into one fused
// multiply-add (one rounding instead of two) even when both carry .rn -- a
// probe measured 824,407 differences in 4 M chained pairs -- so a packed
// product is always written as a fused multiply-add whose addend is -0 taken
// from a kernel argument (`nz`): RN(a*b) + -0 is RN(a*b) bit for bit, signed
// zeros included, and an addend the compiler cannot see as zero leaves it
// nothing to merge.  Every use was checked bit for bit against the scalar
// operations (0 differences in 4 M pairs).
__device__ __forceinline__ float2 fma2_rn(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 pa, pb, pc, pd;\n\t"
      "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\tmov.b64 pc, {%6, %7};\n\t"
      "fma.rn.f32x2 pd, pa, pb, pc;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b, float nz) {
  return fma2_rn(a, b, make_float2(nz, nz));
}
__device__ __forceinline__ float2 add2_rn(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
      "mov.b64 pa, {%2, %3};\n\tmov.b64 pb, {%4, %5};\n\t"
      "add.rn.f32x2 pd, pa, pb;\n\tmov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 bcast2(float v) { return make_float2(v, v); }

// exp_cody_waite on two values at once: the same operations in the same
// order, the floating-point ones packed (results bit-identical).
__device__ __forceinline__ float2 exp_cody_waite2(float2 x, float nz) {
  x.x = clamp_exp_arg(x.x);
  x.y = clamp_exp_arg(x.y);
  const float2 t = mul2_rn(x, bcast2(1.44269504f), nz);            // x / ln 2
  const float2 s = add2_rn(t, bcast2(kRoundMagic));                // rint(t) in the low bits
  const float2 n = add2_rn(s, bcast2(-kRoundMagic));               // rint(t), exactly
  float2 r = fma2_rn(n, bcast2(-0.693359375f), x);                 // x - n*C1
  r = fma2_rn(n, bcast2(2.12194440e-4f), r);                       // - n*C2
  float2 p = fma2_rn(bcast2(1.98412698e-4f), r, bcast2(1.38888889e-3f));
  p = fma2_rn(p, r, bcast2(8.33333333e-3f));
  p = fma2_rn(p, r, bcast2(4.16666667e-2f));
  p = fma2_rn(p, r, bcast2(1.66666667e-1f));
  p = fma2_rn(p, r, bcast2(0.5f));
  p = fma2_rn(p, r, bcast2(1.0f));
  p = fma2_rn(p, r, bcast2(1.0f));
  const float2 two_n = make_float2(__uint_as_float((__float_as_uint(s.x) + 127u) << 23),
                                   __uint_as_float((__float_as_uint(s.y) + 127u) << 23));
  return mul2_rn(p, two_n, nz);
}

// swiglu_rn on two (gate, up) pairs; the divisions stay scalar.
__device__ __forceinline__ float2 swiglu2_rn(float2 gate, float2 up, float nz) {
  const float2 e = exp_cody_waite2(make_float2(-gate.x, -gate.y), nz);
  const float2 d = add2_rn(e, bcast2(1.0f));
  const float2 sg = make_float2(__fdiv_rn(gate.x, d.x), __fdiv_rn(gate.y, d.y));
  return mul2_rn(sg, up, nz);
}

// Combine: resolve the receive rows and gate weights of token g into the
// shared tables rows[k], w[k] (one warp; lane kk handles pair kk).  A bad
// expert id or a row outside [0, y_rows) gives row -1 and a status code.
__device__ __forceinline__ void resolve_token(
    int64_t g, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ weights, const int32_t* __restrict__ send_idx,
    const int32_t* __restrict__ put_offset,
    const int64_t* __restrict__ rank_recv_base, int R, int bs, int k, int epr,
    int64_t y_rows, int64_t* rows, float* w, int32_t* dev_status, int lane) {
  const int E = R * epr;
  const int s = static_cast<int>(g / bs);
  for (int kk = lane; kk < k; kk += 32) {
    const int64_t pair = g * k + kk;
    const int e = __ldg(topk_idx + pair);
    const int32_t sidx = __ldg(send_idx + pair);
    const float wt = __ldg(weights + pair);
    int64_t row = -1;
    if (static_cast<unsigned>(e) >= static_cast<unsigned>(E)) {
      set_status(dev_status, MOE_ERR_EXPERT_ID);
    } else {
      row = __ldg(rank_recv_base + e / epr) + __ldg(put_offset + int64_t(e) * R + s) + sidx;
      if (row < 0 || row >= y_rows) {
        set_status(dev_status, MOE_ERR_CAPACITY);
        row = -1;
      }
    }
    rows[kk] = row;
    w[kk] = wt;
  }
}

// ---- launchers (one per translation unit) ----------------------------------

struct Shape {
  int R, bs, k, epr, H, dtype;
  int E() const { return R * epr; }
  int64_t T() const { return int64_t(R) * bs; }
  int64_t P() const { return T() * k; }
};

// Launch facts (launch_cache.cu): the current device and its SM count, and
// the CTAs of kernel `fn` resident per SM at a block size and dynamic shared
// memory (occupancy cached per kernel, device and size; the >48 KB dynamic
// shared memory attribute is set first when needed).
cudaError_t current_device_sms(int* dev, int* sms);
cudaError_t ensure_dynamic_smem(const void* fn, size_t smem);
cudaError_t kernel_blocks_per_sm(const void* fn, int threads, size_t smem, int* per_sm);

size_t layout_workspace_bytes(const Shape& s);
cudaError_t launch_layout(const Shape& s, const int32_t* topk_idx,
                          int32_t* count, int32_t* rank_send,
                          int32_t* send_idx, void* workspace,
                          int32_t* dev_status, cudaStream_t st);

cudaError_t launch_token_layout(const Shape& s, const int32_t* topk_idx,
                                int32_t* tokens_per_rank, uint8_t* in_rank,
                                int32_t* dev_status, cudaStream_t st);

size_t fused_workspace_bytes(const Shape& s);
cudaError_t launch_fused_dispatch(const Shape& s, const void* x, const int32_t* topk_idx,
                                  bool quant, int32_t* count, int32_t* rank_send,
                                  int32_t* send_idx, int32_t* put_offset,
                                  int32_t* total_recv, int64_t* rank_recv_base,
                                  int32_t* recv_per_expert, int32_t* max_bs, void* recv,
                                  int64_t row_bytes, int64_t capacity, void* workspace,
                                  int32_t* dev_status, cudaStream_t st);

cudaError_t launch_swiglu_quant(const int32_t* acc, int64_t M, int I,
                                const float* weight_scale, const float* token_scale,
                                void* out, cudaStream_t st);

cudaError_t launch_swiglu_quant_grouped(const int32_t* acc, int64_t M, int I,
                                        const float* weight_scale, const int64_t* group_off,
                                        int G, const void* token_scale,
                                        int64_t token_scale_stride, void* out,
                                        float* out_scale, cudaStream_t st);

cudaError_t launch_dispatch_expand(const Shape& s, const void* x, const int32_t* topk_idx,
                                   const int32_t* send_idx, const int32_t* put_offset,
                                   const int64_t* rank_recv_base, void* expand_x,
                                   float* dyn_scale, int64_t capacity_rows,
                                   int32_t* dev_status, cudaStream_t st);

cudaError_t launch_codes_to_bf16(const void* src, int64_t rows, int64_t stride, int K,
                                 void* dst, cudaStream_t st);

int gmm_block_n();

// mode: 0 int32 c, 1 dequantised fp32, 2 SwiGLU of interleaved gate/up pairs.
// main_loop_polls: polls of each main-loop mbarrier wait before it gives up
// (kGemmSpin in every entry point of the header; smaller only in the test
// hook that makes the waits run out).
constexpr uint32_t kGemmSpin = 1u << 20;
cudaError_t launch_grouped_gemm(const void* a, int64_t a_rows, int K, const void* b, int G,
                                int N, const int32_t* group_rows, void* c, int mode,
                                const float* col_scale, const void* row_scale,
                                int64_t row_scale_stride, int32_t* dev_status,
                                cudaStream_t st, uint32_t main_loop_polls = kGemmSpin);

cudaError_t launch_interleave_gate_up(const void* w, const float* ws, int G, int I, int K,
                                     void* wi, float* wsi, cudaStream_t st);

cudaError_t launch_quant_rows_bf16(const float* h, int64_t M, int I, const int64_t* group_off,
                                   int G, void* codes, float* inv_scale, cudaStream_t st);

cudaError_t launch_group_offsets(const int32_t* counts, int G, int64_t* off,
                                 int32_t* dev_status, cudaStream_t st);

cudaError_t launch_deq_combine(const Shape& s, const int32_t* acc2, int64_t y_rows,
                               const float* weight_scale, const void* row_scale,
                               int64_t row_scale_stride, const int32_t* topk_idx,
                               const float* weights, const int32_t* send_idx,
                               const int32_t* put_offset, const int64_t* rank_recv_base,
                               void* out, int32_t* dev_status, cudaStream_t st);

cudaError_t launch_combine_f32(const Shape& s, const float* y, int64_t y_rows,
                               const int32_t* topk_idx, const float* weights,
                               const int32_t* send_idx, const int32_t* put_offset,
                               const int64_t* rank_recv_base, void* out, int32_t* dev_status,
                               cudaStream_t st);

cudaError_t launch_notify(const Shape& s, const int32_t* count,
                          int32_t* put_offset, int32_t* total_recv,
                          int64_t* rank_recv_base, int32_t* recv_per_expert,
                          int32_t* max_bs, cudaStream_t st);

cudaError_t launch_dispatch(const Shape& s, const void* x,
                            const int32_t* topk_idx, const int32_t* send_idx,
                            const int32_t* put_offset,
                            const int64_t* rank_recv_base, bool quant,
                            void* recv, int64_t row_bytes,
                            int64_t capacity_rows, int32_t* dev_status,
                            cudaStream_t st);

cudaError_t launch_combine_quant(const Shape& s, const void* yq, int64_t y_rows,
                                 const int32_t* topk_idx, const float* weights,
                                 const int32_t* send_idx, const int32_t* put_offset,
                                 const int64_t* rank_recv_base, void* out,
                                 int32_t* dev_status, cudaStream_t st);

cudaError_t launch_combine(const Shape& s, const void* y, int64_t y_rows,
                           const int32_t* topk_idx, const float* weights,
                           const int32_t* send_idx, const int32_t* put_offset,
                           const int64_t* rank_recv_base, void* out,
                           int32_t* dev_status, cudaStream_t st);

}  // namespace moe_ep
