// api.cu -- extern "C" entry points of libmoe_ep.so (declared in
// include/moe_ep.h): argument validation, then one launch per stage.
// Every check here is a host-side check; nothing touches the GPU before the
// arguments have been accepted.
#include <climits>
#include <cstdint>

#include "moe_ep_internal.cuh"

namespace {

using moe_ep::Shape;

bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Shape limits of include/moe_ep.h.
bool valid_shape(const moe_shape* sh, Shape* out) {
  if (sh == nullptr) return false;
  const int64_t R = sh->R, bs = sh->bs, k = sh->k, epr = sh->experts_per_rank,
                H = sh->H;
  if (R < 1 || R > MOE_EP_MAX_RANKS) return false;
  if (epr < 1 || R * epr > MOE_EP_MAX_EXPERTS) return false;
  if (k < 1 || k > MOE_EP_MAX_TOPK || k > R * epr) return false;
  if (bs < 0 || R * bs * k >= (int64_t(1) << 31)) return false;
  if (H < 8 || H > MOE_EP_MAX_HIDDEN || H % 8 != 0) return false;
  if (sh->dtype != MOE_BF16 && sh->dtype != MOE_FP16) return false;
  *out = Shape{int(R), int(bs), int(k), int(epr), int(H), int(sh->dtype)};
  return true;
}

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

extern "C" {

const char* moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_EXPERT_ID: return "expert id out of range";
    case MOE_ERR_CAPACITY: return "row outside the receive buffer";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_WORKSPACE: return "layout workspace not zero-filled or shared by overlapping calls";
    default: return "unknown status";
  }
}

int64_t moe_recv_row_bytes(const moe_shape* shape, int quant) {
  Shape s;
  if (!valid_shape(shape, &s)) return -1;
  return quant ? moe_ep::align_up(s.H, 32) + 32 : int64_t(s.H) * 2;
}

size_t moe_layout_workspace_bytes(const moe_shape* shape) {
  Shape s;
  if (!valid_shape(shape, &s)) return 0;
  return moe_ep::layout_workspace_bytes(s);
}

moe_status moe_dispatch_layout(const moe_shape* shape, const int32_t* topk_idx,
                               int32_t* count, int32_t* rank_send,
                               int32_t* send_idx, void* workspace,
                               int32_t* dev_status, void* stream) {
  Shape s;
  if (!valid_shape(shape, &s)) return MOE_ERR_INVALID_ARG;
  if (!count || !rank_send || !dev_status) return MOE_ERR_INVALID_ARG;
  if (!aligned(count, 4) || !aligned(rank_send, 4) || !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (s.P() == 0) {
    cudaError_t e = cudaMemsetAsync(count, 0, sizeof(int32_t) * size_t(s.R) * s.E(), st);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(rank_send, 0, sizeof(int32_t) * size_t(s.R) * s.R, st);
    return from_cuda(e);
  }
  if (!topk_idx || !send_idx || !workspace) return MOE_ERR_INVALID_ARG;
  if (!aligned(topk_idx, 4) || !aligned(send_idx, 4) || !aligned(workspace, 16))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_layout(s, topk_idx, count, rank_send, send_idx,
                                         workspace, dev_status, st));
}

moe_status moe_token_layout(const moe_shape* shape, const int32_t* topk_idx,
                            int32_t* tokens_per_rank, uint8_t* in_rank,
                            int32_t* dev_status, void* stream) {
  Shape s;
  if (!valid_shape(shape, &s)) return MOE_ERR_INVALID_ARG;
  if (!tokens_per_rank || !dev_status || !aligned(tokens_per_rank, 4) ||
      !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  if (s.T() > 0 && (!topk_idx || !in_rank || !aligned(topk_idx, 4) || !aligned(in_rank, 4)))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_token_layout(s, topk_idx, tokens_per_rank, in_rank,
                                               dev_status, static_cast<cudaStream_t>(stream)));
}

moe_status moe_notify_dispatch(const moe_shape* shape, const int32_t* count,
                               int32_t* put_offset, int32_t* total_recv,
                               int64_t* rank_recv_base,
                               int32_t* recv_per_expert, int32_t* max_bs,
                               int32_t* dev_status, void* stream) {
  Shape s;
  if (!valid_shape(shape, &s)) return MOE_ERR_INVALID_ARG;
  if (!count || !put_offset || !total_recv || !rank_recv_base ||
      !recv_per_expert || !max_bs || !dev_status)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(count, 4) || !aligned(put_offset, 4) || !aligned(total_recv, 4) ||
      !aligned(rank_recv_base, 8) || !aligned(recv_per_expert, 4) ||
      !aligned(max_bs, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_notify(s, count, put_offset, total_recv,
                                         rank_recv_base, recv_per_expert,
                                         max_bs, static_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch(const moe_shape* shape, const void* x,
                        const int32_t* topk_idx, const int32_t* send_idx,
                        const int32_t* put_offset,
                        const int64_t* rank_recv_base, int quant, void* recv,
                        int64_t recv_capacity_rows, int32_t* dev_status,
                        void* stream) {
  Shape s;
  if (!valid_shape(shape, &s)) return MOE_ERR_INVALID_ARG;
  if (recv_capacity_rows < 0 || !dev_status) return MOE_ERR_INVALID_ARG;
  if (s.T() == 0) return MOE_OK;
  if (!x || !topk_idx || !send_idx || !put_offset || !rank_recv_base ||
      (!recv && recv_capacity_rows > 0))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(topk_idx, 4) ||
      !aligned(send_idx, 4) || !aligned(put_offset, 4) ||
      !aligned(rank_recv_base, 8) || !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  const int64_t row_bytes = quant ? moe_ep::align_up(s.H, 32) + 32 : int64_t(s.H) * 2;
  return from_cuda(moe_ep::launch_dispatch(
      s, x, topk_idx, send_idx, put_offset, rank_recv_base, quant != 0, recv,
      row_bytes, recv_capacity_rows, dev_status, static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine(const moe_shape* shape, const void* expert_out,
                       int64_t expert_out_rows, const int32_t* topk_idx,
                       const float* topk_weights, const int32_t* send_idx,
                       const int32_t* put_offset,
                       const int64_t* rank_recv_base, void* out,
                       int32_t* dev_status, void* stream) {
  Shape s;
  if (!valid_shape(shape, &s)) return MOE_ERR_INVALID_ARG;
  if (expert_out_rows < 0 || !dev_status) return MOE_ERR_INVALID_ARG;
  if (s.T() == 0) return MOE_OK;
  if ((!expert_out && expert_out_rows > 0) || !topk_idx || !topk_weights ||
      !send_idx || !put_offset || !rank_recv_base || !out)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(expert_out, 16) || !aligned(out, 16) || !aligned(topk_idx, 4) ||
      !aligned(topk_weights, 4) || !aligned(send_idx, 4) ||
      !aligned(put_offset, 4) || !aligned(rank_recv_base, 8) ||
      !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_combine(s, expert_out, expert_out_rows,
                                          topk_idx, topk_weights, send_idx,
                                          put_offset, rank_recv_base, out,
                                          dev_status, static_cast<cudaStream_t>(stream)));
}

moe_status moe_swiglu_quant(const int32_t* acc, int64_t M, int32_t I,
                            const float* weight_scale, const float* token_scale,
                            void* out, int32_t* dev_status, void* stream) {
  if (M < 0 || I < 8 || I > 16384 || I % 8 != 0 || !dev_status) return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if (!acc || !weight_scale || !token_scale || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(acc, 16) || !aligned(weight_scale, 16) || !aligned(token_scale, 4) ||
      !aligned(out, 16) || !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_swiglu_quant(acc, M, I, weight_scale, token_scale, out,
                                               static_cast<cudaStream_t>(stream)));
}

size_t moe_fused_workspace_bytes(const moe_shape* shape) {
  Shape s;
  if (!valid_shape(shape, &s)) return 0;
  return moe_ep::fused_workspace_bytes(s);
}

moe_status moe_dispatch_fused(const moe_shape* shape, const void* x,
                              const int32_t* topk_idx, int quant, int32_t* count,
                              int32_t* rank_send, int32_t* send_idx,
                              int32_t* put_offset, int32_t* total_recv,
                              int64_t* rank_recv_base, int32_t* recv_per_expert,
                              int32_t* max_bs, void* recv,
                              int64_t recv_capacity_rows, void* workspace,
                              int32_t* dev_status, void* stream) {
  Shape s;
  if (!valid_shape(shape, &s)) return MOE_ERR_INVALID_ARG;
  if (recv_capacity_rows < 0 || !count || !rank_send || !put_offset || !total_recv ||
      !rank_recv_base || !recv_per_expert || !max_bs || !workspace || !dev_status)
    return MOE_ERR_INVALID_ARG;
  if (s.T() > 0 && (!x || !topk_idx || !send_idx || (!recv && recv_capacity_rows > 0)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(workspace, 16) ||
      !aligned(topk_idx, 4) || !aligned(count, 4) || !aligned(rank_send, 4) ||
      !aligned(send_idx, 4) || !aligned(put_offset, 4) || !aligned(total_recv, 4) ||
      !aligned(rank_recv_base, 8) || !aligned(recv_per_expert, 4) ||
      !aligned(max_bs, 4) || !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  const int64_t row_bytes = quant ? moe_ep::align_up(s.H, 32) + 32 : int64_t(s.H) * 2;
  return from_cuda(moe_ep::launch_fused_dispatch(
      s, x, topk_idx, quant != 0, count, rank_send, send_idx, put_offset, total_recv,
      rank_recv_base, recv_per_expert, max_bs, recv, row_bytes, recv_capacity_rows,
      workspace, dev_status, static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_quant(const moe_shape* shape, const void* expert_out_q,
                             int64_t expert_out_rows, const int32_t* topk_idx,
                             const float* topk_weights, const int32_t* send_idx,
                             const int32_t* put_offset,
                             const int64_t* rank_recv_base, void* out,
                             int32_t* dev_status, void* stream) {
  Shape s;
  if (!valid_shape(shape, &s)) return MOE_ERR_INVALID_ARG;
  if (expert_out_rows < 0 || !dev_status) return MOE_ERR_INVALID_ARG;
  if (s.T() == 0) return MOE_OK;
  if ((!expert_out_q && expert_out_rows > 0) || !topk_idx || !topk_weights ||
      !send_idx || !put_offset || !rank_recv_base || !out)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(expert_out_q, 16) || !aligned(out, 16) || !aligned(topk_idx, 4) ||
      !aligned(topk_weights, 4) || !aligned(send_idx, 4) ||
      !aligned(put_offset, 4) || !aligned(rank_recv_base, 8) ||
      !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_combine_quant(
      s, expert_out_q, expert_out_rows, topk_idx, topk_weights, send_idx, put_offset,
      rank_recv_base, out, dev_status, static_cast<cudaStream_t>(stream)));
}

moe_status moe_swiglu_quant_grouped(const int32_t* acc, int64_t M, int32_t I,
                                    const float* weight_scale, const int64_t* group_off,
                                    int32_t G, const void* token_scale,
                                    int64_t token_scale_stride, void* out,
                                    int32_t* dev_status, void* stream) {
  if (M < 0 || I < 8 || I > 16384 || I % 8 != 0 || G < 1 || G > MOE_EP_MAX_EXPERTS ||
      token_scale_stride < 4 || token_scale_stride % 4 != 0 || !dev_status)
    return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if (!acc || !weight_scale || !group_off || !token_scale || !out) return MOE_ERR_INVALID_ARG;
  if (!aligned(acc, 16) || !aligned(weight_scale, 16) || !aligned(group_off, 8) ||
      !aligned(token_scale, 4) || !aligned(out, 16) || !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_swiglu_quant_grouped(
      acc, M, I, weight_scale, group_off, G, token_scale, token_scale_stride, out, nullptr,
      static_cast<cudaStream_t>(stream)));
}

moe_status moe_swiglu_quant_grouped_bf16(const int32_t* acc, int64_t M, int32_t I,
                                         const float* weight_scale, const int64_t* group_off,
                                         int32_t G, const void* token_scale,
                                         int64_t token_scale_stride, void* codes,
                                         float* inv_scale, int32_t* dev_status,
                                         void* stream) {
  if (M < 0 || I < 8 || I > 16384 || I % 8 != 0 || G < 1 || G > MOE_EP_MAX_EXPERTS ||
      token_scale_stride < 4 || token_scale_stride % 4 != 0 || !dev_status)
    return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if (!acc || !weight_scale || !group_off || !token_scale || !codes || !inv_scale)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(acc, 16) || !aligned(weight_scale, 16) || !aligned(group_off, 8) ||
      !aligned(token_scale, 4) || !aligned(codes, 16) || !aligned(inv_scale, 4) ||
      !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_swiglu_quant_grouped(
      acc, M, I, weight_scale, group_off, G, token_scale, token_scale_stride, codes,
      inv_scale, static_cast<cudaStream_t>(stream)));
}

moe_status moe_dispatch_expand(const moe_shape* shape, const void* x,
                               const int32_t* topk_idx, const int32_t* send_idx,
                               const int32_t* put_offset, const int64_t* rank_recv_base,
                               void* expand_x, float* dynamic_scale,
                               int64_t capacity_rows, int32_t* dev_status, void* stream) {
  Shape s;
  if (!valid_shape(shape, &s)) return MOE_ERR_INVALID_ARG;
  if (capacity_rows < 0 || !dev_status) return MOE_ERR_INVALID_ARG;
  if (s.T() == 0) return MOE_OK;
  if (!x || !topk_idx || !send_idx || !put_offset || !rank_recv_base ||
      (capacity_rows > 0 && (!expand_x || !dynamic_scale)))
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(expand_x, 16) || !aligned(dynamic_scale, 4) ||
      !aligned(topk_idx, 4) || !aligned(send_idx, 4) || !aligned(put_offset, 4) ||
      !aligned(rank_recv_base, 8) || !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_dispatch_expand(
      s, x, topk_idx, send_idx, put_offset, rank_recv_base, expand_x, dynamic_scale,
      capacity_rows, dev_status, static_cast<cudaStream_t>(stream)));
}

moe_status moe_codes_to_bf16(const void* codes, int64_t rows, int64_t row_stride, int32_t K,
                             void* out, void* stream) {
  if (rows < 0 || K < 8 || K > MOE_EP_MAX_HIDDEN || K % 8 != 0 || row_stride < K ||
      row_stride % 8 != 0)
    return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!codes || !out || !aligned(codes, 8) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_codes_to_bf16(codes, rows, row_stride, K, out,
                                                static_cast<cudaStream_t>(stream)));
}

int32_t moe_gmm_block_n(void) { return moe_ep::gmm_block_n(); }

moe_status moe_grouped_gemm_i8(const void* a, int64_t a_rows, int32_t K, const void* w,
                               int32_t G, int32_t N, const int32_t* group_rows, int32_t* c,
                               int32_t* dev_status, void* stream) {
  const int64_t bn = moe_ep::gmm_block_n();
  if (a_rows < 0 || a_rows > INT32_MAX || K < 8 || K > MOE_EP_MAX_HIDDEN || K % 8 != 0 ||
      G < 1 || G > MOE_EP_MAX_EXPERTS || N < 8 || N > MOE_EP_MAX_HIDDEN || N % 8 != 0 ||
      !dev_status)
    return MOE_ERR_INVALID_ARG;
  if (a_rows == 0) return MOE_OK;   // no rows: nothing to compute
  if ((a_rows / 128 + G) * ((N + bn - 1) / bn) > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (!a || !w || !group_rows || !c) return MOE_ERR_INVALID_ARG;
  if (!aligned(a, 16) || !aligned(w, 16) || !aligned(group_rows, 4) || !aligned(c, 16) ||
      !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_grouped_gemm(a, a_rows, K, w, G, N, group_rows, c, 0,
                                               nullptr, nullptr, 0, dev_status,
                                               static_cast<cudaStream_t>(stream)));
}

// Test hook, deliberately not declared in moe_ep.h: moe_grouped_gemm_i8 with
// the pipeline's main-loop waits limited to `main_loop_polls` polls (0 makes
// the first wait of every working CTA give up), so that a test can drive the
// kernel's timeout path -- MOE_ERR_TIMEOUT in *dev_status, no further work
// issued, every copy, MMA, commit and store already in flight drained under
// the full bound before TMEM is released -- without a fault or a hang.
extern "C" moe_status moe_test_grouped_gemm_i8_polls(const void* a, int64_t a_rows, int32_t K,
                                                     const void* w, int32_t G, int32_t N,
                                                     const int32_t* group_rows, int32_t* c,
                                                     uint32_t main_loop_polls,
                                                     int32_t* dev_status, void* stream) {
  const int64_t bn = moe_ep::gmm_block_n();
  if (a_rows < 1 || a_rows > INT32_MAX || K < 8 || K > MOE_EP_MAX_HIDDEN || K % 8 != 0 ||
      G < 1 || G > MOE_EP_MAX_EXPERTS || N < 8 || N > MOE_EP_MAX_HIDDEN || N % 8 != 0 ||
      !dev_status || !a || !w || !group_rows || !c)
    return MOE_ERR_INVALID_ARG;
  if ((a_rows / 128 + G) * ((N + bn - 1) / bn) > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (!aligned(a, 16) || !aligned(w, 16) || !aligned(group_rows, 4) || !aligned(c, 16) ||
      !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_grouped_gemm(a, a_rows, K, w, G, N, group_rows, c, 0,
                                               nullptr, nullptr, 0, dev_status,
                                               static_cast<cudaStream_t>(stream),
                                               main_loop_polls));
}

moe_status moe_grouped_gemm_i8_dequant(const void* a, int64_t a_rows, int32_t K,
                                       const void* w, int32_t G, int32_t N,
                                       const int32_t* group_rows, const float* col_scale,
                                       const void* row_scale, int64_t row_scale_stride,
                                       float* y, int32_t* dev_status, void* stream) {
  const int64_t bn = moe_ep::gmm_block_n();
  if (a_rows < 0 || a_rows > INT32_MAX || K < 8 || K > MOE_EP_MAX_HIDDEN || K % 8 != 0 ||
      G < 1 || G > MOE_EP_MAX_EXPERTS || N < 8 || N > MOE_EP_MAX_HIDDEN || N % 8 != 0 ||
      row_scale_stride < 4 || row_scale_stride % 4 != 0 || !dev_status)
    return MOE_ERR_INVALID_ARG;
  if (a_rows == 0) return MOE_OK;
  if ((a_rows / 128 + G) * ((N + bn - 1) / bn) > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (!a || !w || !group_rows || !col_scale || !row_scale || !y) return MOE_ERR_INVALID_ARG;
  if (!aligned(a, 16) || !aligned(w, 16) || !aligned(group_rows, 4) ||
      !aligned(col_scale, 16) || !aligned(row_scale, 4) || !aligned(y, 16) ||
      !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_grouped_gemm(a, a_rows, K, w, G, N, group_rows, y, 1,
                                               col_scale, row_scale, row_scale_stride,
                                               dev_status,
                                               static_cast<cudaStream_t>(stream)));
}

moe_status moe_grouped_gemm_i8_swiglu(const void* a, int64_t a_rows, int32_t K,
                                      const void* w_interleaved, int32_t G, int32_t I,
                                      const int32_t* group_rows,
                                      const float* col_scale_interleaved,
                                      const void* row_scale, int64_t row_scale_stride,
                                      float* h, int32_t* dev_status, void* stream) {
  const int64_t bn = moe_ep::gmm_block_n();
  const int64_t N = 2 * int64_t(I);
  if (a_rows < 0 || a_rows > INT32_MAX || K < 8 || K > MOE_EP_MAX_HIDDEN || K % 8 != 0 ||
      G < 1 || G > MOE_EP_MAX_EXPERTS || I < 8 || N > MOE_EP_MAX_HIDDEN || I % 8 != 0 ||
      row_scale_stride < 4 || row_scale_stride % 4 != 0 || !dev_status)
    return MOE_ERR_INVALID_ARG;
  if (a_rows == 0) return MOE_OK;
  if ((a_rows / 128 + G) * ((N + bn - 1) / bn) > INT32_MAX) return MOE_ERR_INVALID_ARG;
  if (!a || !w_interleaved || !group_rows || !col_scale_interleaved || !row_scale || !h)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(a, 16) || !aligned(w_interleaved, 16) || !aligned(group_rows, 4) ||
      !aligned(col_scale_interleaved, 16) || !aligned(row_scale, 4) || !aligned(h, 16) ||
      !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_grouped_gemm(
      a, a_rows, K, w_interleaved, G, static_cast<int>(N), group_rows, h, 2,
      col_scale_interleaved, row_scale, row_scale_stride, dev_status,
      static_cast<cudaStream_t>(stream)));
}

moe_status moe_interleave_gate_up(const void* w1, const float* ws1, int32_t G, int32_t I,
                                  int32_t K, void* w1_interleaved,
                                  float* ws1_interleaved, void* stream) {
  if (G < 1 || G > MOE_EP_MAX_EXPERTS || I < 8 || 2 * int64_t(I) > MOE_EP_MAX_HIDDEN ||
      I % 8 != 0 || K < 8 || K > MOE_EP_MAX_HIDDEN || K % 8 != 0)
    return MOE_ERR_INVALID_ARG;
  if (!w1 || !ws1 || !w1_interleaved || !ws1_interleaved || !aligned(w1, 8) ||
      !aligned(ws1, 4) || !aligned(w1_interleaved, 16) || !aligned(ws1_interleaved, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_interleave_gate_up(w1, ws1, G, I, K, w1_interleaved,
                                                     ws1_interleaved,
                                                     static_cast<cudaStream_t>(stream)));
}

moe_status moe_quant_rows_bf16(const float* h, int64_t M, int32_t I, const int64_t* group_off,
                               int32_t G, void* codes, float* inv_scale, void* stream) {
  if (M < 0 || I < 8 || I > 16384 || I % 8 != 0 || (group_off && (G < 1 || G > MOE_EP_MAX_EXPERTS)))
    return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if (!h || !codes || !inv_scale || !aligned(h, 16) || !aligned(codes, 16) ||
      !aligned(inv_scale, 4) || !aligned(group_off, 8))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_quant_rows_bf16(h, M, I, group_off, G, codes, inv_scale,
                                                  static_cast<cudaStream_t>(stream)));
}

moe_status moe_combine_f32(const moe_shape* shape, const float* expert_out,
                           int64_t expert_out_rows, const int32_t* topk_idx,
                           const float* topk_weights, const int32_t* send_idx,
                           const int32_t* put_offset, const int64_t* rank_recv_base,
                           void* out, int32_t* dev_status, void* stream) {
  Shape s;
  if (!valid_shape(shape, &s)) return MOE_ERR_INVALID_ARG;
  if (expert_out_rows < 0 || !dev_status) return MOE_ERR_INVALID_ARG;
  if (s.T() == 0) return MOE_OK;
  if ((!expert_out && expert_out_rows > 0) || !topk_idx || !topk_weights || !send_idx ||
      !put_offset || !rank_recv_base || !out)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(expert_out, 16) || !aligned(out, 16) || !aligned(topk_idx, 4) ||
      !aligned(topk_weights, 4) || !aligned(send_idx, 4) || !aligned(put_offset, 4) ||
      !aligned(rank_recv_base, 8) || !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_combine_f32(s, expert_out, expert_out_rows, topk_idx,
                                              topk_weights, send_idx, put_offset,
                                              rank_recv_base, out, dev_status,
                                              static_cast<cudaStream_t>(stream)));
}

moe_status moe_group_offsets(const int32_t* group_rows, int32_t G, int64_t* group_off,
                             int32_t* dev_status, void* stream) {
  if (G < 1 || G > MOE_EP_MAX_EXPERTS || !group_rows || !group_off || !dev_status ||
      !aligned(group_rows, 4) || !aligned(group_off, 8) || !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_group_offsets(group_rows, G, group_off, dev_status,
                                                static_cast<cudaStream_t>(stream)));
}

moe_status moe_deq_combine(const moe_shape* shape, const int32_t* expert_acc,
                           int64_t expert_rows, const float* weight_scale,
                           const void* row_scale, int64_t row_scale_stride,
                           const int32_t* topk_idx, const float* topk_weights,
                           const int32_t* send_idx, const int32_t* put_offset,
                           const int64_t* rank_recv_base, void* out, int32_t* dev_status,
                           void* stream) {
  Shape s;
  if (!valid_shape(shape, &s)) return MOE_ERR_INVALID_ARG;
  if (expert_rows < 0 || row_scale_stride < 4 || row_scale_stride % 4 != 0 || !dev_status)
    return MOE_ERR_INVALID_ARG;
  if (s.T() == 0) return MOE_OK;
  if ((expert_rows > 0 && (!expert_acc || !row_scale)) || !weight_scale || !topk_idx ||
      !topk_weights || !send_idx || !put_offset || !rank_recv_base || !out)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(expert_acc, 16) || !aligned(weight_scale, 16) || !aligned(row_scale, 4) ||
      !aligned(out, 16) || !aligned(topk_idx, 4) || !aligned(topk_weights, 4) ||
      !aligned(send_idx, 4) || !aligned(put_offset, 4) || !aligned(rank_recv_base, 8) ||
      !aligned(dev_status, 4))
    return MOE_ERR_INVALID_ARG;
  return from_cuda(moe_ep::launch_deq_combine(
      s, expert_acc, expert_rows, weight_scale, row_scale, row_scale_stride, topk_idx,
      topk_weights, send_idx, put_offset, rank_recv_base, out, dev_status,
      static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
