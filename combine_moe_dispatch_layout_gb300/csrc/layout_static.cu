// layout_static.cu -- moe_dispatch_layout_static: the dispatch layout with
// its scratch memory in a fixed, library-owned device array instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// The scratch is one file-scope static __device__ array of
// MOE_EP_STATIC_LAYOUT_WS_BYTES bytes; every GPU that loads the library holds
// it until the process exits.  Host code never uses the array's name as an
// address: every call, with the stream's device current, asks
// cudaGetSymbolAddress for the array's device address on that device and
// passes it to the kernel.  The first call on a device is the set-up: that
// lookup also loads the library's module onto the device.  Later lookups
// are cheap, and not caching the address keeps a call made after
// cudaDeviceReset (which unloads the module and frees the array) from
// writing through a stale pointer.
#include "moe_ep_internal.cuh"

static __device__ __align__(256) unsigned char g_layout_scratch[MOE_EP_STATIC_LAYOUT_WS_BYTES];

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
  if (cudaGetSymbolAddress(&scratch, g_layout_scratch) != cudaSuccess || scratch == nullptr)
    return MOE_ERR_CUDA;
  // Ordinary calls would not need this clear: the layout kernel's per-launch
  // epoch leaves the workspace ready for the next launch of any shape, and
  // the array starts zero-filled.  It is here so that a call that follows
  // one that stopped early (a wait that timed out) or that overlapped
  // another call on the GPU starts from a clean workspace all the same.
  // Keep it.
  if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOE_ERR_CUDA;
  return moe_dispatch_layout(shape, topk_idx, count, rank_send, send_idx,
                             scratch, dev_status, stream);
}
