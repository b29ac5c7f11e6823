// decode_noalloc.cu -- paged_decode_noalloc: paged decode whose split-KV
// scratch lives in a fixed, file-scope device array instead of a buffer the
// caller provides.
//
// Some callers cannot allocate device memory for the library: a plugin whose
// host framework owns every device allocation and offers no workspace hook, or
// a serving loop that must not call cudaMalloc because it can synchronise the
// device and stall the other streams.  This entry point needs no workspace and
// allocates nothing itself.  The scratch is PKV_NOALLOC_SCRATCH_BYTES of
// device memory that every GPU which loads this library holds until the
// process exits.  All calls share it, so calls that overlap on the GPU race:
// the caller must order them (one stream, or events between streams).  The
// kernels write every scratch byte they later read, so nothing needs clearing
// between calls.
//
// The first call on a device resolves the array's device address.  The
// library is built without relocatable device code, so under lazy module
// loading (the CUDA default) that lookup is also what loads this file's module
// and backs the array, which can allocate and synchronise.  Callers that must
// avoid that inside their serving loop make one call with batch 0 at set-up
// time (or run with CUDA_MODULE_LOADING=EAGER).  The cached address is not
// refreshed after cudaDeviceReset; a process that resets a device must not use
// the library on it afterwards.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace pkv {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDev];

// Device address of g_decode_scratch on the current device, looked up once per
// device.  In host code the symbol is only a host-side stand-in, so the kernels
// must be given this address, never the symbol itself.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}
}  // namespace

}  // namespace pkv

extern "C" int paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_table, int32_t max_blocks_per_seq,
                                    const int32_t* cache_seqlens, int32_t batch, float scale,
                                    void* out, const pkv_geom* geom, cudaStream_t stream) {
    // the same argument checks as paged_decode (api.cu)
    const int st = pkv::check_geom(geom);
    if (st != PKV_OK) return st;
    if (batch < 0 || max_blocks_per_seq < 0) return PKV_ERR_INVALID;
    // batch 0 does the per-device set-up only (a warm-up call: see pagedkv.h)
    void* scratch = nullptr;
    if (batch == 0) return pkv::scratch_address(&scratch) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
    if (!q || !k_cache || !v_cache || !block_table || !cache_seqlens || !out)
        return PKV_ERR_INVALID;
    if (!pkv::aligned(q, 16) || !pkv::aligned(k_cache, 16) || !pkv::aligned(v_cache, 16) ||
        !pkv::aligned(out, 16))
        return PKV_ERR_INVALID;
    pkv::DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    pkv::DecodePlan plan;
    if (!pkv::plan_decode(dev, batch, geom->num_heads, geom->num_kv_heads, geom->head_dim,
                          geom->block_size, pkv::elt_size(geom->dtype), &plan))
        return PKV_ERR_UNSUPPORTED;
    if (plan.ws_bytes > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
    if (pkv::scratch_address(&scratch) != cudaSuccess) return PKV_ERR_CUDA;
    cudaError_t e = pkv::launch_decode(plan, q, k_cache, v_cache, block_table, max_blocks_per_seq,
                                       cache_seqlens, batch, scale, out, scratch,
                                       geom->num_heads, geom->num_kv_heads, geom->head_dim,
                                       geom->block_size, geom->num_blocks, geom->dtype, dev.err,
                                       stream);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
