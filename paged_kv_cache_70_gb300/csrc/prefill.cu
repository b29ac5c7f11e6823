// prefill.cu -- causal varlen prefill over a paged cache (placeholder).
#include "common.cuh"
#include "launch.h"

namespace pkv {

size_t prefill_workspace_bytes(int32_t, int32_t, int) { return 0; }

cudaError_t launch_prefill(const DeviceInfo&, const void*, const void*, const void*,
                           const int32_t*, const int32_t*, int32_t, int32_t, int32_t,
                           const int32_t*, int32_t, int, float, void*, void*, int, int, int, int,
                           int64_t, unsigned int*, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace pkv
