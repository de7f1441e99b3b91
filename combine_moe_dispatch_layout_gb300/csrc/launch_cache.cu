// launch_cache.cu -- per-device launch facts, looked up once.
//
// The persistent kernels size their grids from the SM count and from how
// many CTAs of the kernel fit on an SM.  The occupancy query costs
// microseconds of host time per launch, as long as a small problem's whole
// kernel, so its answer is remembered per (kernel, device, block size,
// dynamic shared memory), and the SM count per device.  Both are properties
// of the device and the compiled kernel: caching them changes no result.
// The dynamic shared memory limit above the default 48 KB per block (static
// plus dynamic) is a per-context function attribute, which a device reset
// clears, so it is set on every launch that needs it (a cheap call) rather
// than remembered; the kernel's static size it depends on is looked up once.
#include <mutex>
#include <vector>

#include "moe_ep_internal.cuh"

namespace moe_ep {
namespace {

struct OccEntry {
  const void* fn;
  int dev, threads;
  size_t smem;
  int per_sm;
};

constexpr int kMaxDevs = 64;

struct StaticEntry {
  const void* fn;
  size_t bytes;
};

std::mutex g_mu;
std::vector<OccEntry> g_occ;
std::vector<StaticEntry> g_static;
int g_sms[kMaxDevs] = {};

}  // namespace

cudaError_t current_device_sms(int* dev, int* sms) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  if (*dev >= 0 && *dev < kMaxDevs) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_sms[*dev] > 0) {
      *sms = g_sms[*dev];
      return cudaSuccess;
    }
  }
  e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev);
  if (e == cudaSuccess && *dev >= 0 && *dev < kMaxDevs && *sms > 0) {
    std::lock_guard<std::mutex> lock(g_mu);
    g_sms[*dev] = *sms;
  }
  return e;
}

// Static shared memory of a kernel (a property of the compiled function,
// looked up once).
cudaError_t static_smem(const void* fn, size_t* bytes) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (const StaticEntry& e : g_static)
      if (e.fn == fn) {
        *bytes = e.bytes;
        return cudaSuccess;
      }
  }
  cudaFuncAttributes a;
  const cudaError_t e = cudaFuncGetAttributes(&a, fn);
  if (e != cudaSuccess) return e;
  *bytes = a.sharedSizeBytes;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_static.size() < 4096) g_static.push_back({fn, a.sharedSizeBytes});
  return cudaSuccess;
}

cudaError_t ensure_dynamic_smem(const void* fn, size_t smem) {
  if (smem == 0) return cudaSuccess;
  size_t stat = 0;
  cudaError_t e = static_smem(fn, &stat);
  if (e != cudaSuccess) return e;
  // the default per-block limit (48 KB) covers static plus dynamic memory
  if (smem + stat <= 48 * 1024) return cudaSuccess;
  return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(smem));
}

cudaError_t kernel_blocks_per_sm(const void* fn, int threads, size_t smem, int* per_sm) {
  cudaError_t e = ensure_dynamic_smem(fn, smem);
  if (e != cudaSuccess) return e;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (const OccEntry& o : g_occ)
      if (o.fn == fn && o.dev == dev && o.threads == threads && o.smem == smem) {
        *per_sm = o.per_sm;
        return cudaSuccess;
      }
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, fn, threads, smem);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_occ.size() < 4096) g_occ.push_back({fn, dev, threads, smem, *per_sm});
  return cudaSuccess;
}

}  // namespace moe_ep
