// gdn_status.cu -- the per-device status word kernels raise errors into.
//
// A kernel that meets an input only the device can see (a state index outside
// the pool, malformed cu_seqlens) ORs a bit into this word and skips the
// offending sequence instead of touching memory out of bounds.
// gdn_read_device_status() reads and clears it.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "gdn_internal.h"

namespace {
__device__ unsigned g_status_word;

constexpr int kMaxDevices = 64;
unsigned* g_addr[kMaxDevices] = {};
std::mutex g_mu;
std::atomic<uint64_t> g_launches{0};
}  // namespace

extern "C" uint64_t gdn_launch_count(void) { return g_launches.load(); }

namespace gdn {

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

unsigned* status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
      cudaGetLastError();  // clear the non-sticky error so a later call's check does not see it
      return nullptr;
    }
    g_addr[dev] = static_cast<unsigned*>(p);
  }
  return g_addr[dev];
}

}  // namespace gdn
