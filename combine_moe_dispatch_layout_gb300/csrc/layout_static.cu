// layout_static.cu -- moe_dispatch_layout_static: the dispatch layout with
// its scratch memory in a fixed, library-owned device array instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// The scratch is one file-scope __device__ array of MOE_EP_STATIC_LAYOUT_WS_BYTES
// bytes; every GPU that loads the library holds it until the process exits.
// Host code never uses the array's name as an address: on the first call on
// each device (with that device current) cudaGetSymbolAddress gives the
// device address, which is cached per device and passed to the kernel.
#include <mutex>

#include "moe_ep_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_layout_scratch[MOE_EP_STATIC_LAYOUT_WS_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_layout_scratch on the current device (set-up on the
// first call per device).
cudaError_t scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_layout_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" moe_status moe_dispatch_layout_static(
    const moe_shape* shape, const int32_t* topk_idx, int32_t* count,
    int32_t* rank_send, int32_t* send_idx, int32_t* dev_status, void* stream) {
  const size_t need = moe_layout_workspace_bytes(shape);   // 0: invalid shape
  if (need > MOE_EP_STATIC_LAYOUT_WS_BYTES) return MOE_ERR_INVALID_ARG;
  // the regular entry point's pointer checks, before this one's own CUDA
  // calls (host-checkable errors return before any CUDA call)
  auto misaligned4 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 3u) != 0; };
  if (!count || !rank_send || !dev_status || misaligned4(count) || misaligned4(rank_send) ||
      misaligned4(dev_status))
    return MOE_ERR_INVALID_ARG;
  if (need > 0 && int64_t(shape->R) * shape->bs * shape->k > 0 &&
      (!topk_idx || !send_idx || misaligned4(topk_idx) || misaligned4(send_idx)))
    return MOE_ERR_INVALID_ARG;
  if (need == 0)   // let the regular entry point report the invalid shape
    return moe_dispatch_layout(shape, topk_idx, count, rank_send, send_idx,
                               nullptr, dev_status, stream);
  void* scratch = nullptr;
  if (scratch_on_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
  // The array keeps whatever the previous call left in it; the part this
  // call uses is cleared first, on the caller's stream, so it starts at zero.
  if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return moe_dispatch_layout(shape, topk_idx, count, rank_send, send_idx,
                             scratch, dev_status, stream);
}
