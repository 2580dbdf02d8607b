// gdn_chunked.cu -- chunked (C = 64) WY/UT-form prefill on tcgen05 tensor cores.
#include <cuda_runtime.h>

#include "gdn_internal.h"

namespace gdn {

bool chunked_supported(int, int, bool) { return false; }

size_t chunked_workspace_bytes(int64_t, int64_t, int64_t, int64_t, int64_t) { return 0; }

cudaError_t launch_chunked(const ChunkedLaunch&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gdn
