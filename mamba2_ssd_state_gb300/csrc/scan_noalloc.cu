// scan_noalloc.cu -- the library-owned scratch behind ssd_chunk_scan_static_ws.
//
// A caller that cannot allocate device memory at call time still gets the split scan:
// its workspace comes from one statically sized device array that is part of this
// library's image, so no allocator runs on the call path.  The array is one buffer per
// device shared by every call on that device: calls that overlap in time race on it.
#include <mutex>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

// 16 MiB: a split of one 16384-token sequence on 24 heads of 64 channels needs 11 MiB.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

// Nothing in it needs to start at zero: the scan writes every word of it that the
// fix-up pass reads, before that pass reads it.
static __device__ __align__(256) unsigned char g_scan_scratch[kStaticScratchBytes];

}  // namespace

size_t scan_static_scratch_bytes() { return kStaticScratchBytes; }

// Device address of the scratch on the current device, looked up on the first call for
// that device (the lookup may load this library's module onto the device) and cached.
void* scan_static_scratch() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scan_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace ssd
