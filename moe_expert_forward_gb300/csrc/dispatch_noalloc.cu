// mm_moe_dispatch_noalloc: the routing step (a1) for callers that cannot hand
// the library any scratch memory.  The per-CTA expert counts that
// mm_moe_dispatch keeps in caller scratch live here in a fixed file-scope
// device array instead, so this entry point performs no allocation at all.
#include <mutex>

#include "internal.h"

namespace mm {
namespace {

// Per-CTA expert counts [CTAs][E] of one call.  Every GPU that loads the
// library holds these 256 KiB until the process exits.
constexpr int64_t kNoallocScratchInts = 64 * 1024;
static __device__ __align__(256) int32_t g_dispatch_scratch[kNoallocScratchInts];

constexpr int kMaxDevices = 64;
int32_t* g_scratch_addr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

// Device address of g_dispatch_scratch on the current device, looked up once per device.
cudaError_t scratch_for_current_device(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace mm

extern "C" int mm_moe_dispatch_noalloc(const int32_t* topk_idx, int T, int K, int E, int block_m, int32_t* cnt,
                                       int32_t* blk_off, int32_t* slot, int32_t* src, int64_t src_capacity,
                                       int32_t* status, void* stream) {
  using namespace mm;
  if (T < 0 || K <= 0 || E <= 0 || K > kMaxK || K > E || E > kMaxE) return MM_MOE_ERR_INVALID_ARG;
  if (static_cast<int64_t>(T) * K > (int64_t(1) << 30)) return MM_MOE_ERR_INVALID_ARG;
  if (block_m < 16 || block_m > 256 || block_m % 16) return MM_MOE_ERR_INVALID_ARG;
  if (!cnt || !blk_off || !status || (T > 0 && (!topk_idx || !slot || !src))) return MM_MOE_ERR_INVALID_ARG;
  const int64_t pairs = static_cast<int64_t>(T) * K;
  const int64_t live = pairs < E ? pairs : E;
  if (src_capacity < pairs + live * (block_m - 1)) return MM_MOE_ERR_INVALID_ARG;
  const DevInfo& d = dev_info();
  if (!(d.cc_major == 10 && d.cc_minor == 3)) return MM_MOE_ERR_UNSUPPORTED;
  // The fixed array bounds the CTA count at kNoallocScratchInts / E (at least
  // 64 for E <= 1024), as a small caller scratch does for mm_moe_dispatch; the
  // slots do not depend on the CTA count, so every valid shape fits.
  if (E > kNoallocScratchInts) return MM_MOE_ERR_WORKSPACE_TOO_SMALL;
  int32_t* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return MM_MOE_ERR_CUDA;
  // The count kernel rewrites all CTAs x E entries it uses before the assign
  // kernel reads them, so nothing in the array has to be cleared between calls.
  const cudaError_t e = launch_dispatch(topk_idx, T, K, E, block_m, cnt, blk_off, slot, src, status, scratch,
                                        kNoallocScratchInts, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MM_MOE_OK : MM_MOE_ERR_CUDA;
}
