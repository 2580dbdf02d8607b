// gdn_noalloc.cu -- gdn_prefill_varlen for callers that cannot allocate
// device memory.
//
// The chunked prefill needs a scratch buffer (gdn_prefill_workspace_bytes).
// Some callers cannot provide one: a plug-in running inside a host runtime
// that owns all device memory and hands plug-ins no allocator, or a
// latency-critical serving loop that must never call cudaMalloc (it can
// synchronise the device and fail under memory pressure at the worst time).
// gdn_prefill_varlen_noalloc serves them from a fixed scratch array that is
// part of this library's device image: it calls no cudaMalloc, cudaFree or
// other allocating routine.
//
// The array is a file-scope static __device__ variable, so every GPU that
// loads this library's module holds kNoAllocScratchBytes of device memory for
// it until the process exits.  Under CUDA's default lazy module loading the
// module, and with it the 64 MiB, is committed on the first call on each
// device, when cudaGetSymbolAddress needs it; that set-up can fail (for
// instance when the device is out of memory), and then the call returns
// GDN_ERR_CUDA with the CUDA error in gdn_last_error_message().  Host code
// cannot use the array's name as a device address (in host code it is only a
// stand-in), so that first call, with the device current, resolves the real
// address once and caches it; it should therefore come before any stream
// capture.  Every call shares the one array: calls whose
// GPU work overlaps (different streams, or several host threads) race on it.
// Nothing in it has to start at zero: the prefill writes every scratch byte it
// reads within the same call, so the previous call's contents never matter.
#include <cuda_runtime.h>

#include <mutex>

#include <string>

#include "../../include/gdn.h"
#include "gdn_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;  // 64 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

}  // namespace

extern "C" int gdn_prefill_varlen_noalloc(const gdn_prefill_args* args, void* stream) {
  if (args == nullptr) return gdn_prefill_varlen(args, stream);  // reports the NULL args
  int dev = 0;
  const cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) {
    cudaGetLastError();
    return gdn::report_error(
        GDN_ERR_CUDA, (std::string("noalloc: no current device: ") + cudaGetErrorString(de)).c_str());
  }
  if (dev < 0 || dev >= kMaxDevices)
    return gdn::report_error(GDN_ERR_CUDA, ("noalloc: device ordinal " + std::to_string(dev) +
                                            " beyond the " + std::to_string(kMaxDevices) +
                                            " this library tracks").c_str());
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {  // once per device, with that device current
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
      if (e != cudaSuccess) {
        cudaGetLastError();  // clear it: a later launch check must not pick it up
        return gdn::report_error(GDN_ERR_CUDA,
                                 (std::string("noalloc scratch address lookup failed: ") +
                                  cudaGetErrorString(e)).c_str());
      }
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  // Same call with the static scratch as its workspace.  When the sizes need
  // more than kNoAllocScratchBytes, gdn_prefill_varlen's own workspace check
  // rejects the call (GDN_ERR_INVALID_ARGUMENT, "... workspace needs N bytes,
  // got 67108864") before anything is launched.
  gdn_prefill_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = kNoAllocScratchBytes;
  return gdn_prefill_varlen(&a, stream);
}
