// api.cu -- the extern "C" entry points of libpagedkv (declared in
// include/pagedkv.h): argument validation, per-device state (SM count,
// shared-memory limit, error word) and dispatch to the kernel launchers.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace pkv {

// One error word per device (each device holds its own copy of this variable).
__device__ unsigned int g_error_word = 0;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_have[kMaxDevices];
DeviceInfo g_info[kMaxDevices];
}  // namespace

cudaError_t current_device_info(DeviceInfo* info) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_have[dev]) {
        DeviceInfo d{};
        d.device = dev;
        e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        int smem = 0;
        e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e != cudaSuccess) return e;
        d.max_smem_optin = (size_t)smem;
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_error_word);
        if (e != cudaSuccess) return e;
        d.err = static_cast<unsigned int*>(p);
        g_info[dev] = d;
        g_have[dev] = true;
    }
    *info = g_info[dev];
    return cudaSuccess;
}

int check_geom(const pkv_geom* g) {
    if (!g) return PKV_ERR_INVALID;
    if (g->num_heads <= 0 || g->num_kv_heads <= 0 || g->head_dim <= 0 || g->block_size <= 0 ||
        g->num_blocks < 0)
        return PKV_ERR_INVALID;
    if (g->num_heads % g->num_kv_heads) return PKV_ERR_INVALID;
    if (!elt_size(g->dtype)) return PKV_ERR_INVALID;
    // slot ids are int32
    if ((double)g->num_blocks * g->block_size > 2147483647.0) return PKV_ERR_UNSUPPORTED;
    return PKV_OK;
}

}  // namespace pkv

using pkv::DeviceInfo;
using pkv::aligned;
using pkv::check_geom;
using pkv::elt_size;

namespace {

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

}  // namespace

extern "C" {

int paged_build_slot_mapping(const int32_t* block_table, int32_t max_blocks_per_seq,
                             int32_t num_seqs, const int32_t* token_seq,
                             const int32_t* token_pos, int64_t num_tokens, int32_t block_size,
                             int32_t* slot_mapping, cudaStream_t stream) {
    if (num_tokens < 0 || block_size <= 0 || max_blocks_per_seq < 0 || num_seqs < 0)
        return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!token_seq || !token_pos || !slot_mapping) return PKV_ERR_INVALID;
    if (num_seqs > 0 && max_blocks_per_seq > 0 && !block_table) return PKV_ERR_INVALID;
    DeviceInfo dev;
    cudaError_t e = pkv::current_device_info(&dev);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    return cuda_status(pkv::launch_build_slot_mapping(block_table, max_blocks_per_seq, num_seqs,
                                                      token_seq, token_pos, num_tokens,
                                                      block_size, slot_mapping, dev.err, stream));
}

int paged_kv_write(const void* k, const void* v, int32_t kv_dtype, const int32_t* slot_mapping,
                   int64_t num_tokens, void* k_cache, void* v_cache, const pkv_geom* geom,
                   cudaStream_t stream) {
    int st = check_geom(geom);
    if (st != PKV_OK) return st;
    if (!elt_size(kv_dtype) || num_tokens < 0) return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const int64_t kv_dim = (int64_t)geom->num_kv_heads * geom->head_dim;
    const int64_t num_slots = geom->num_blocks * geom->block_size;
    return cuda_status(pkv::launch_kv_write(k, v, kv_dtype, slot_mapping, num_tokens, k_cache,
                                            v_cache, geom->dtype, kv_dim, num_slots, dev.err,
                                            stream));
}

int paged_kv_write_positions(const void* k, const void* v, int32_t kv_dtype,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             int32_t num_seqs, const int32_t* token_seq,
                             const int32_t* token_pos, int64_t num_tokens,
                             int32_t* slot_mapping_out, void* k_cache, void* v_cache,
                             const pkv_geom* geom, cudaStream_t stream) {
    int st = check_geom(geom);
    if (st != PKV_OK) return st;
    if (!elt_size(kv_dtype) || num_tokens < 0 || max_blocks_per_seq < 0 || num_seqs < 0)
        return PKV_ERR_INVALID;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !token_seq || !token_pos || !k_cache || !v_cache) return PKV_ERR_INVALID;
    if (num_seqs > 0 && max_blocks_per_seq > 0 && !block_table) return PKV_ERR_INVALID;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const int64_t kv_dim = (int64_t)geom->num_kv_heads * geom->head_dim;
    const int64_t num_slots = geom->num_blocks * geom->block_size;
    return cuda_status(pkv::launch_kv_write_positions(
        k, v, kv_dtype, block_table, max_blocks_per_seq, num_seqs, token_seq, token_pos,
        num_tokens, geom->block_size, slot_mapping_out, k_cache, v_cache, geom->dtype, kv_dim,
        num_slots, dev.err, stream));
}

static size_t align256(size_t x) { return (x + 255) / 256 * 256; }

static pkv::PrefixLaunch prefix_pass(const DeviceInfo& dev, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* table,
                                     int32_t max_blocks, int32_t batch, const int32_t* group_cu,
                                     const int32_t* group_plen, int32_t n_groups,
                                     int32_t max_group_size, float scale, void* x_out,
                                     float* x_lse, const pkv_geom* g, bool pdl);

// bf16 decode with a GQA group of 4 or more: every sequence's keys go through
// the tensor-core pass as a group of one, in chunks of keys, about one
// (sequence, KV head, chunk) item per SM, and the combine merges the chunks
// (no split launch).  With 4 or more query heads per KV head the split runs
// short of issue slots on the CUDA cores; with 2 it streams faster than the
// tensor-core pass.  Returns the chunks per sequence, 0 when the CUDA-core
// split takes the decode.
constexpr int kMaxTcChunks = 32;
static int tc_chunks(const DeviceInfo& dev, int32_t batch, const pkv_geom* g) {
    const int G = g->num_heads / g->num_kv_heads;
    if (g->dtype != PKV_BF16 || G < 4 || 128 % G) return 0;
    if (g->head_dim != 128 && g->head_dim != 64) return 0;
    const int B = g->block_size;
    if (!(B >= 128 ? B % 128 == 0 : (B >= 8 && 128 % B == 0))) return 0;
    const int64_t units = (int64_t)batch * g->num_kv_heads;
    if (units <= 0) return 0;
    const int64_t kc = ((int64_t)dev.num_sms + units - 1) / units;
    return (int)std::min<int64_t>(std::max<int64_t>(kc, 1), kMaxTcChunks);
}
// the chunks' partials: [kc, batch, hq, d] bf16 outputs, [kc, batch, hq] log2-sum-exp
static size_t tc_extra_bytes(int kc, int32_t batch, const pkv_geom* g) {
    return align256((size_t)kc * batch * g->num_heads * g->head_dim * 2) +
           align256((size_t)kc * batch * g->num_heads * 4);
}

// the decode through the tensor-core pass (tc_chunks > 0), with or without
// the append
static int tc_decode(const DeviceInfo& dev, const pkv::DecodePlan& plan, int kc, const void* q,
                     const void* k_cache, const void* v_cache, const int32_t* block_table,
                     int32_t max_blocks, const int32_t* cache_seqlens, int32_t batch,
                     float scale, void* out, void* workspace, const pkv_geom* geom,
                     const pkv::DecodeAppend* ap, cudaStream_t stream) {
    unsigned char* x_out = static_cast<unsigned char*>(workspace) + plan.ws_bytes;
    float* x_lse = reinterpret_cast<float*>(
        x_out + align256((size_t)kc * batch * geom->num_heads * geom->head_dim * 2));
    pkv::PrefixLaunch pp = prefix_pass(dev, q, k_cache, v_cache, block_table, max_blocks, batch,
                                       nullptr, nullptr, batch, 1, scale, x_out, x_lse, geom,
                                       false);
    const int64_t cap = (int64_t)max_blocks * geom->block_size;
    int64_t per = (cap + kc - 1) / kc;
    per = (per + 127) / 128 * 128;
    pp.kchunks = kc;
    pp.seqlens = cache_seqlens;
    pp.chunk_keys = (int32_t)std::min<int64_t>(std::max<int64_t>(per, 128), 1 << 30);
    cudaError_t e = pkv::launch_prefix(dev, pp, stream);
    if (e == cudaErrorNotSupported)  // the pass does not take this pool (nothing was
                                     // launched): the split alone does the decode
        return cuda_status(pkv::launch_decode(plan, q, k_cache, v_cache, block_table, max_blocks,
                                              cache_seqlens, batch, scale, out, workspace,
                                              geom->num_heads, geom->num_kv_heads,
                                              geom->head_dim, geom->block_size,
                                              geom->num_blocks, geom->dtype, dev.err, stream,
                                              nullptr, ap, nullptr));
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    pkv::SharedPrefix sp{nullptr, nullptr, 0, x_out, x_lse, kc};
    pkv::DecodeChain ch{true, true};
    return cuda_status(pkv::launch_decode(plan, q, k_cache, v_cache, block_table, max_blocks,
                                          cache_seqlens, batch, scale, out, workspace,
                                          geom->num_heads, geom->num_kv_heads, geom->head_dim,
                                          geom->block_size, geom->num_blocks, geom->dtype,
                                          dev.err, stream, &sp, ap, &ch));
}

size_t paged_decode_workspace_size(int32_t batch, const pkv_geom* geom) {
    if (check_geom(geom) != PKV_OK || batch < 0) return 0;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return 0;
    pkv::DecodePlan plan;
    if (!pkv::plan_decode(dev, batch, geom->num_heads, geom->num_kv_heads, geom->head_dim,
                          geom->block_size, elt_size(geom->dtype), &plan))
        return 0;
    const int kc = tc_chunks(dev, batch, geom);
    return plan.ws_bytes + (kc ? tc_extra_bytes(kc, batch, geom) : 0);
}

int paged_decode(const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_table, int32_t max_blocks_per_seq,
                 const int32_t* cache_seqlens, int32_t batch, float scale, void* out,
                 void* workspace, size_t workspace_bytes, const pkv_geom* geom,
                 cudaStream_t stream) {
    int st = check_geom(geom);
    if (st != PKV_OK) return st;
    if (batch < 0 || max_blocks_per_seq < 0) return PKV_ERR_INVALID;
    if (batch == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_table || !cache_seqlens || !out)
        return PKV_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return PKV_ERR_INVALID;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    pkv::DecodePlan plan;
    if (!pkv::plan_decode(dev, batch, geom->num_heads, geom->num_kv_heads, geom->head_dim,
                          geom->block_size, elt_size(geom->dtype), &plan))
        return PKV_ERR_UNSUPPORTED;
    const int kc = tc_chunks(dev, batch, geom);
    const size_t need = plan.ws_bytes + (kc ? tc_extra_bytes(kc, batch, geom) : 0);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
        return PKV_ERR_WORKSPACE;
    if (kc)
        return tc_decode(dev, plan, kc, q, k_cache, v_cache, block_table, max_blocks_per_seq,
                         cache_seqlens, batch, scale, out, workspace, geom, nullptr, stream);
    return cuda_status(pkv::launch_decode(plan, q, k_cache, v_cache, block_table,
                                          max_blocks_per_seq, cache_seqlens, batch, scale, out,
                                          workspace, geom->num_heads, geom->num_kv_heads,
                                          geom->head_dim, geom->block_size, geom->num_blocks,
                                          geom->dtype, dev.err, stream));
}

int paged_decode_append(const void* q, const void* k_new, const void* v_new, void* k_cache,
                        void* v_cache, const int32_t* block_table, int32_t max_blocks_per_seq,
                        const int32_t* cache_seqlens, int32_t batch, float scale, void* out,
                        void* workspace, size_t workspace_bytes, const pkv_geom* geom,
                        cudaStream_t stream) {
    int st = check_geom(geom);
    if (st != PKV_OK) return st;
    if (batch < 0 || max_blocks_per_seq < 0) return PKV_ERR_INVALID;
    if (batch == 0) return PKV_OK;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !block_table || !cache_seqlens || !out)
        return PKV_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(k_new, 16) || !aligned(v_new, 16))
        return PKV_ERR_INVALID;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    pkv::DecodePlan plan;
    if (!pkv::plan_decode(dev, batch, geom->num_heads, geom->num_kv_heads, geom->head_dim,
                          geom->block_size, elt_size(geom->dtype), &plan))
        return PKV_ERR_UNSUPPORTED;
    const int kc = tc_chunks(dev, batch, geom);
    const size_t need = plan.ws_bytes + (kc ? tc_extra_bytes(kc, batch, geom) : 0);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
        return PKV_ERR_WORKSPACE;
    pkv::DecodeAppend ap{k_new, v_new, k_cache, v_cache};
    if (kc)
        return tc_decode(dev, plan, kc, q, k_cache, v_cache, block_table, max_blocks_per_seq,
                         cache_seqlens, batch, scale, out, workspace, geom, &ap, stream);
    return cuda_status(pkv::launch_decode(plan, q, k_cache, v_cache, block_table,
                                          max_blocks_per_seq, cache_seqlens, batch, scale, out,
                                          workspace, geom->num_heads, geom->num_kv_heads,
                                          geom->head_dim, geom->block_size, geom->num_blocks,
                                          geom->dtype, dev.err, stream, nullptr, &ap));
}

size_t paged_varlen_prefill_workspace_size(int32_t batch, int32_t max_seqlen_q,
                                           const pkv_geom* geom) {
    if (check_geom(geom) != PKV_OK || batch < 0 || max_seqlen_q < 0) return 0;
    return pkv::prefill_workspace_bytes(batch, max_seqlen_q, geom->num_heads);
}

int paged_varlen_prefill(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                         int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t* block_table,
                         int32_t max_blocks_per_seq, int32_t causal, float scale, void* out,
                         void* workspace, size_t workspace_bytes, const pkv_geom* geom,
                         cudaStream_t stream) {
    int st = check_geom(geom);
    if (st != PKV_OK) return st;
    if (batch < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || max_blocks_per_seq < 0)
        return PKV_ERR_INVALID;
    if (batch == 0 || max_seqlen_q == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !cu_seqlens_q || !cu_seqlens_k || !out)
        return PKV_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return PKV_ERR_INVALID;
    if (geom->dtype != PKV_BF16 || (geom->head_dim != 128 && geom->head_dim != 64))
        return PKV_ERR_UNSUPPORTED;
    const size_t need = pkv::prefill_workspace_bytes(batch, max_seqlen_q, geom->num_heads);
    if (need && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
        return PKV_ERR_WORKSPACE;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    cudaError_t e = pkv::launch_prefill(
        dev, q, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, batch, max_seqlen_q, max_seqlen_k,
        block_table, max_blocks_per_seq, causal, scale, out, workspace, geom->num_heads,
        geom->num_kv_heads, geom->head_dim, geom->block_size, geom->num_blocks, dev.err, stream);
    if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
    return cuda_status(e);
}

// the prefix keys of a group are split into at most this many chunks (work
// items for the SMs); each chunk leaves its own partial per (sequence, head)
constexpr int kMaxPrefixChunks = 8;

static size_t shared_prefix_extra_bytes(int32_t batch, const pkv_geom* g) {
    return align256((size_t)kMaxPrefixChunks * batch * g->num_heads * g->head_dim * 2) +
           align256((size_t)kMaxPrefixChunks * batch * g->num_heads * 4);
}

// Workspace of a grouped decode: the split's pieces, then the prefix partials.
static size_t grouped_ws_bytes(const pkv::DecodePlan& plan, int32_t batch, const pkv_geom* g) {
    return plan.ws_bytes + shared_prefix_extra_bytes(batch, g);
}

size_t paged_decode_shared_prefix_workspace_size(int32_t batch, const pkv_geom* geom) {
    if (check_geom(geom) != PKV_OK || batch < 0) return 0;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return 0;
    pkv::DecodePlan plan;
    if (!pkv::plan_decode(dev, batch, geom->num_heads, geom->num_kv_heads, geom->head_dim,
                          geom->block_size, elt_size(geom->dtype), &plan))
        return 0;
    return grouped_ws_bytes(plan, batch, geom);
}

// The shared-prefix pass of a grouped decode: one work item per (group, KV
// head, key chunk, block of 128 / G members); the keys are cut into enough
// chunks for the items to cover the SMs once.
static pkv::PrefixLaunch prefix_pass(const DeviceInfo& dev, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* table,
                                     int32_t max_blocks, int32_t batch, const int32_t* group_cu,
                                     const int32_t* group_plen, int32_t n_groups,
                                     int32_t max_group_size, float scale, void* x_out,
                                     float* x_lse, const pkv_geom* g, bool pdl) {
    const int G = g->num_heads / g->num_kv_heads;
    const int per_blk = G <= 128 ? 128 / G : 1;
    const int units = n_groups * g->num_kv_heads * ((max_group_size + per_blk - 1) / per_blk);
    int kchunks = units > 0 ? dev.num_sms / units : 1;
    kchunks = kchunks < 1 ? 1 : (kchunks > kMaxPrefixChunks ? kMaxPrefixChunks : kchunks);
    pkv::PrefixLaunch p{};
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.table = table;
    p.group_cu = group_cu;
    p.group_plen = group_plen;
    p.x_out = x_out;
    p.x_lse = x_lse;
    p.err = dev.err;
    p.num_blocks = g->num_blocks;
    p.scale = scale;
    p.max_blocks = max_blocks;
    p.batch = batch;
    p.hq = g->num_heads;
    p.hkv = g->num_kv_heads;
    p.hd = g->head_dim;
    p.block_size = g->block_size;
    p.n_groups = n_groups;
    p.max_group_size = max_group_size;
    p.kchunks = kchunks;
    p.pdl = pdl;
    return p;
}

int paged_decode_shared_prefix(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int32_t max_blocks_per_seq,
                               const int32_t* cache_seqlens, int32_t batch,
                               const int32_t* group_cu, const int32_t* group_prefix_len,
                               int32_t n_groups, int32_t max_group_size, float scale, void* out,
                               void* workspace, size_t workspace_bytes, const pkv_geom* geom,
                               cudaStream_t stream) {
    int st = check_geom(geom);
    if (st != PKV_OK) return st;
    if (batch < 0 || max_blocks_per_seq < 0 || n_groups < 0 || max_group_size < 0)
        return PKV_ERR_INVALID;
    if (batch == 0) return PKV_OK;
    if (n_groups == 0 || max_group_size == 0) return PKV_ERR_INVALID;
    if (!q || !k_cache || !v_cache || !block_table || !cache_seqlens || !out || !group_cu ||
        !group_prefix_len)
        return PKV_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return PKV_ERR_INVALID;
    if (geom->dtype != PKV_BF16 || (geom->head_dim != 128 && geom->head_dim != 64))
        return PKV_ERR_UNSUPPORTED;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    pkv::DecodePlan plan;
    if (!pkv::plan_decode(dev, batch, geom->num_heads, geom->num_kv_heads, geom->head_dim,
                          geom->block_size, elt_size(geom->dtype), &plan))
        return PKV_ERR_UNSUPPORTED;
    const size_t need = grouped_ws_bytes(plan, batch, geom);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return PKV_ERR_WORKSPACE;
    unsigned char* x_out = static_cast<unsigned char*>(workspace) + plan.ws_bytes;
    float* x_lse = reinterpret_cast<float*>(
        x_out + align256((size_t)kMaxPrefixChunks * batch * geom->num_heads * geom->head_dim * 2));
    // 1. the prefix of every group, once: attention of the group's queries
    //    over its first group_prefix_len[g] keys, read through the block-table
    //    row of the group's first sequence (tensor cores)
    const pkv::PrefixLaunch pp = prefix_pass(dev, q, k_cache, v_cache, block_table,
                                             max_blocks_per_seq, batch, group_cu,
                                             group_prefix_len, n_groups, max_group_size, scale,
                                             x_out, x_lse, geom, false);
    const int kchunks = pp.kchunks;
    cudaError_t e = pkv::launch_prefix(dev, pp, stream);
    if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    // 2. each sequence's own keys after the prefix, merged with the prefix state.
    //    The split needs nothing from the prefix pass (only the combine does),
    //    so it starts while the prefix pass runs and holds its grid open until
    //    that kernel completes; the prefix pass itself started after all earlier
    //    work on the stream.
    pkv::SharedPrefix sp{group_cu, group_prefix_len, n_groups, x_out, x_lse, kchunks};
    pkv::DecodeChain ch{true};
    return cuda_status(pkv::launch_decode(plan, q, k_cache, v_cache, block_table,
                                          max_blocks_per_seq, cache_seqlens, batch, scale, out,
                                          workspace, geom->num_heads, geom->num_kv_heads,
                                          geom->head_dim, geom->block_size, geom->num_blocks,
                                          geom->dtype, dev.err, stream, &sp, nullptr, &ch));
}

// The mixed step's workspace: the grouped decode's, then 256 bytes for the
// one-launch form's counters.
size_t paged_mixed_step_workspace_size(int32_t decode_batch, const pkv_geom* geom) {
    if (check_geom(geom) != PKV_OK || decode_batch < 0) return 0;
    if (decode_batch == 0) return 256;
    const size_t g = paged_decode_shared_prefix_workspace_size(decode_batch, geom);
    return g ? g + 256 : 0;
}

int paged_mixed_step(const pkv_mixed_step* s, void* k_cache, void* v_cache, void* workspace,
                     size_t workspace_bytes, const pkv_geom* geom, cudaStream_t stream) {
    int st = check_geom(geom);
    if (st != PKV_OK) return st;
    if (!s || !k_cache || !v_cache) return PKV_ERR_INVALID;
    if (s->prefill_new_tokens < 0 || s->prefill_batch < 0 || s->decode_batch < 0 ||
        s->n_groups < 0)
        return PKV_ERR_INVALID;
    const bool pf = s->prefill_batch > 0 && s->max_seqlen_q > 0;
    const bool dec = s->decode_batch > 0;
    const bool grp = dec && s->n_groups > 0;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16)) return PKV_ERR_INVALID;
    if ((pf || grp) &&
        (geom->dtype != PKV_BF16 || (geom->head_dim != 128 && geom->head_dim != 64)))
        return PKV_ERR_UNSUPPORTED;
    if (s->prefill_new_tokens > 0 &&
        (!s->prefill_k_new || !s->prefill_v_new || !s->prefill_slots))
        return PKV_ERR_INVALID;
    if (pf && (!s->prefill_q || !s->cu_seqlens_q || !s->cu_seqlens_k || !s->prefill_table ||
               !s->prefill_out || !aligned(s->prefill_q, 16) || !aligned(s->prefill_out, 16)))
        return PKV_ERR_INVALID;
    if (dec && (!s->decode_q || !s->decode_k_new || !s->decode_v_new || !s->decode_table ||
                !s->decode_seqlens || !s->decode_out || !aligned(s->decode_q, 16) ||
                !aligned(s->decode_out, 16) || !aligned(s->decode_k_new, 16) ||
                !aligned(s->decode_v_new, 16)))
        return PKV_ERR_INVALID;
    if (grp && (!s->group_cu || !s->group_prefix_len || s->max_group_size <= 0))
        return PKV_ERR_INVALID;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    pkv::DecodePlan plan;
    if (dec) {
        if (!pkv::plan_decode(dev, s->decode_batch, geom->num_heads, geom->num_kv_heads,
                              geom->head_dim, geom->block_size, elt_size(geom->dtype), &plan))
            return PKV_ERR_UNSUPPORTED;
        const size_t need = grouped_ws_bytes(plan, s->decode_batch, geom);
        if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
            return PKV_ERR_WORKSPACE;
    }
    const int64_t kv_dim = (int64_t)geom->num_kv_heads * geom->head_dim;
    // 1. the prefill requests' new rows
    if (s->prefill_new_tokens > 0) {
        cudaError_t e = pkv::launch_kv_write(s->prefill_k_new, s->prefill_v_new, geom->dtype,
                                             s->prefill_slots, s->prefill_new_tokens, k_cache,
                                             v_cache, geom->dtype, kv_dim,
                                             geom->num_blocks * geom->block_size, dev.err, stream);
        if (e != cudaSuccess) return PKV_ERR_CUDA;
    }
    // 2. the tensor-core work: the causal varlen prefill and, when the decode
    //    is grouped, the shared-prefix pass, in one launch (the prefix items
    //    start at once; the prefill items wait for the write)
    pkv::SharedPrefix sp{};
    pkv::PrefixLaunch pp{};
    if (grp) {
        unsigned char* x_out = static_cast<unsigned char*>(workspace) + plan.ws_bytes;
        float* x_lse = reinterpret_cast<float*>(
            x_out + align256((size_t)kMaxPrefixChunks * s->decode_batch * geom->num_heads *
                             geom->head_dim * 2));
        pp = prefix_pass(dev, s->decode_q, k_cache, v_cache, s->decode_table, s->decode_max_blocks,
                         s->decode_batch, s->group_cu, s->group_prefix_len, s->n_groups,
                         s->max_group_size, s->scale, x_out, x_lse, geom, true);
        sp = pkv::SharedPrefix{s->group_cu, s->group_prefix_len, s->n_groups, x_out, x_lse,
                               pp.kchunks};
    }
    cudaError_t e = cudaSuccess;
    if (pf && grp) {
        e = pkv::launch_prefill_with_prefix(
            dev, s->prefill_q, k_cache, v_cache, s->cu_seqlens_q, s->cu_seqlens_k,
            s->prefill_batch, s->max_seqlen_q, s->prefill_table, s->prefill_max_blocks, s->scale,
            s->prefill_out, geom->num_heads, geom->num_kv_heads, geom->head_dim,
            geom->block_size, geom->num_blocks, dev.err, pp, stream);
    } else if (pf) {
        e = pkv::launch_prefill(dev, s->prefill_q, k_cache, v_cache, s->cu_seqlens_q,
                                s->cu_seqlens_k, s->prefill_batch, s->max_seqlen_q,
                                s->max_seqlen_k, s->prefill_table, s->prefill_max_blocks, 1,
                                s->scale, s->prefill_out, nullptr, geom->num_heads,
                                geom->num_kv_heads, geom->head_dim, geom->block_size,
                                geom->num_blocks, dev.err, stream);
    } else if (grp) {
        e = pkv::launch_prefix(dev, pp, stream);
    }
    if (e == cudaErrorNotSupported) return PKV_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    const bool chained = pf || grp;  // a kernel of this call precedes the decode
    if (!dec) return PKV_OK;
    // 3. decode with the append, merged with the shared prefixes when grouped
    pkv::DecodeAppend ap{s->decode_k_new, s->decode_v_new, k_cache, v_cache};
    pkv::DecodeChain ch{chained};
    return cuda_status(pkv::launch_decode(
        plan, s->decode_q, k_cache, v_cache, s->decode_table, s->decode_max_blocks,
        s->decode_seqlens, s->decode_batch, s->scale, s->decode_out, workspace, geom->num_heads,
        geom->num_kv_heads, geom->head_dim, geom->block_size, geom->num_blocks, geom->dtype,
        dev.err, stream, grp ? &sp : nullptr, &ap, &ch));
}

int paged_mixed_step_one_launch(const pkv_mixed_step* s, void* k_cache, void* v_cache,
                                void* workspace, size_t workspace_bytes, const pkv_geom* geom,
                                cudaStream_t stream) {
    // the one-launch form takes full steps of its shape; anything else (or an
    // invalid step, which paged_mixed_step reports) goes the chained way
    const int st_g = check_geom(geom);
    if (st_g != PKV_OK || !s || !k_cache || !v_cache) return paged_mixed_step(s, k_cache, v_cache,
                                                                              workspace,
                                                                              workspace_bytes,
                                                                              geom, stream);
    const bool full = s->prefill_batch > 0 && s->max_seqlen_q > 0 && s->decode_batch > 0 &&
                      s->n_groups > 0 && s->prefill_new_tokens > 0;
    if (!full || geom->dtype != PKV_BF16 || geom->num_heads != 2 * geom->num_kv_heads)
        return paged_mixed_step(s, k_cache, v_cache, workspace, workspace_bytes, geom, stream);
    if (!s->prefill_k_new || !s->prefill_v_new || !s->prefill_slots || !s->prefill_q ||
        !s->cu_seqlens_q || !s->cu_seqlens_k || !s->prefill_table || !s->prefill_out ||
        !s->decode_q || !s->decode_k_new || !s->decode_v_new || !s->decode_table ||
        !s->decode_seqlens || !s->decode_out || !s->group_cu || !s->group_prefix_len ||
        s->max_group_size <= 0)
        return paged_mixed_step(s, k_cache, v_cache, workspace, workspace_bytes, geom, stream);
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(s->prefill_q, 16) ||
        !aligned(s->prefill_out, 16) || !aligned(s->decode_q, 16) ||
        !aligned(s->decode_out, 16) || !aligned(s->decode_k_new, 16) ||
        !aligned(s->decode_v_new, 16) || !aligned(s->prefill_k_new, 16) ||
        !aligned(s->prefill_v_new, 16))
        return PKV_ERR_INVALID;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    pkv::DecodePlan plan;
    if (!pkv::plan_decode(dev, s->decode_batch, geom->num_heads, geom->num_kv_heads,
                          geom->head_dim, geom->block_size, elt_size(geom->dtype), &plan))
        return PKV_ERR_UNSUPPORTED;
    const size_t grouped = grouped_ws_bytes(plan, s->decode_batch, geom);
    if (!workspace || workspace_bytes < grouped + 256 || !aligned(workspace, 256))
        return PKV_ERR_WORKSPACE;
    unsigned char* x_out = static_cast<unsigned char*>(workspace) + plan.ws_bytes;
    float* x_lse = reinterpret_cast<float*>(
        x_out + align256((size_t)kMaxPrefixChunks * s->decode_batch * geom->num_heads *
                         geom->head_dim * 2));
    pkv::StepOneLaunch st{};
    st.prefix = prefix_pass(dev, s->decode_q, k_cache, v_cache, s->decode_table,
                            s->decode_max_blocks, s->decode_batch, s->group_cu,
                            s->group_prefix_len, s->n_groups, s->max_group_size, s->scale,
                            x_out, x_lse, geom, false);
    st.plan = plan;
    st.pf_k_new = s->prefill_k_new;
    st.pf_v_new = s->prefill_v_new;
    st.pf_slots = s->prefill_slots;
    st.pf_new_tokens = s->prefill_new_tokens;
    st.pf_q = s->prefill_q;
    st.cu_q = s->cu_seqlens_q;
    st.cu_k = s->cu_seqlens_k;
    st.pf_batch = s->prefill_batch;
    st.max_seqlen_q = s->max_seqlen_q;
    st.pf_max_blocks = s->prefill_max_blocks;
    st.pf_table = s->prefill_table;
    st.pf_out = s->prefill_out;
    st.dec_k_new = s->decode_k_new;
    st.dec_v_new = s->decode_v_new;
    st.dec_seqlens = s->decode_seqlens;
    st.dec_out = s->decode_out;
    st.k_cache = k_cache;
    st.v_cache = v_cache;
    st.workspace = workspace;
    st.counters = reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(workspace) + grouped);
    st.scale = s->scale;
    st.hq = geom->num_heads;
    st.hkv = geom->num_kv_heads;
    st.block_size = geom->block_size;
    st.dtype = geom->dtype;
    st.num_blocks = geom->num_blocks;
    const cudaError_t e = pkv::launch_step_one(dev, st, stream);
    if (e == cudaErrorNotSupported)  // nothing was launched: the chained form
        return paged_mixed_step(s, k_cache, v_cache, workspace, workspace_bytes, geom, stream);
    return cuda_status(e);
}

int paged_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst,
                      int32_t n_pairs, const pkv_geom* geom, cudaStream_t stream) {
    int st = check_geom(geom);
    if (st != PKV_OK) return st;
    if (n_pairs < 0 || n_pairs > 65535) return n_pairs < 0 ? PKV_ERR_INVALID : PKV_ERR_UNSUPPORTED;
    if (n_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !src || !dst) return PKV_ERR_INVALID;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    const int64_t block_bytes = (int64_t)geom->block_size * geom->num_kv_heads * geom->head_dim *
                                elt_size(geom->dtype);
    return cuda_status(pkv::launch_copy_blocks(k_cache, v_cache, src, dst, n_pairs, block_bytes,
                                               geom->num_blocks, dev.err, stream));
}

int paged_error_flags(uint32_t* flags, int32_t clear) {
    if (!flags) return PKV_ERR_INVALID;
    DeviceInfo dev;
    if (pkv::current_device_info(&dev) != cudaSuccess) return PKV_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpy(&v, dev.err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (clear) {
        const unsigned int zero = 0;
        if (cudaMemcpy(dev.err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return PKV_ERR_CUDA;
    }
    *flags = v;
    return PKV_OK;
}

const char* paged_status_string(int status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case PKV_ERR_WORKSPACE: return "workspace missing or too small";
        case PKV_ERR_CUDA: return "CUDA error";
        case PKV_ERR_NO_SPACE: return "not enough free blocks";
        default: return "unknown status";
    }
}

}  // extern "C"
