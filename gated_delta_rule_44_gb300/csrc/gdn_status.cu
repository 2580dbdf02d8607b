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
#include <string>

#include "../../include/gdn.h"
#include "gdn_internal.h"
#include "tcgen05.cuh"

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

namespace {

// One thread waits, with the library's bounded wait, on an mbarrier that
// nothing ever arrives on; when the budget runs out it records the timeout in
// the status word, exactly as the kernels do when one of their waits gives
// up.  Nothing else is issued, so nothing is in flight when it returns.
__global__ void wait_timeout_kernel(unsigned* status, long long budget) {
  __shared__ uint64_t mbar;
  const uint32_t mb = gdn::umma::smem_u32(&mbar);
  gdn::umma::mbar_init(mb, 1);
  gdn::umma::fence_mbar_init();
  if (!gdn::umma::mbar_wait(mb, 0, budget)) atomicOr(status, gdn::kStatusTimeout);
}

}  // namespace

extern "C" int gdn_check_wait_timeout(long long budget_cycles, void* stream) {
  if (budget_cycles <= 0 || budget_cycles > 2000000000LL)
    return gdn::report_error(GDN_ERR_INVALID_ARGUMENT,
                             "budget_cycles must be in (0, 2e9] (about one second)");
  unsigned* w = gdn::status_word();
  if (w == nullptr) return gdn::report_error(GDN_ERR_CUDA, "device status word unavailable");
  wait_timeout_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(w, budget_cycles);
  gdn::note_launch();
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return gdn::report_error(GDN_ERR_CUDA,
                             (std::string("gdn_check_wait_timeout: ") + cudaGetErrorString(e)).c_str());
  return gdn::report_error(GDN_OK, "");
}
