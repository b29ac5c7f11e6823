// launch.h -- internal host-side launchers of libpagedkv's kernels.  The C ABI
// layer (api.cu) validates arguments before calling any of these; each returns
// the cudaError_t of its launch(es).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

// Launch `kern` as a programmatic dependent of the kernel before it on
// `stream`: it may be scheduled while that kernel finishes, and must execute
// griddepcontrol.wait before it touches memory that kernel (or any earlier
// work) may produce.  After any other kind of predecessor this is an ordinary
// stream-ordered launch.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// First statement of such kernels: let the next kernel launch early, then wait
// for this one's inputs.
#define PKV_DEPENDENT_PROLOGUE()                                  \
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); \
    asm volatile("griddepcontrol.wait;" ::: "memory")

// ---- argument checks shared by the entry points -----------------------------
inline bool aligned(const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// bytes per element of a pkv_dtype, 0 for an unknown code
inline int elt_size(int dtype) { return dtype == PKV_F32 ? 4 : (dtype == PKV_BF16 ? 2 : 0); }

// Geometry checks common to every call taking a pkv_geom (api.cu): PKV_OK,
// PKV_ERR_INVALID (null, non-positive sizes, Hq % Hkv != 0, unknown dtype) or
// PKV_ERR_UNSUPPORTED (more than 2^31 - 1 slots: slot ids are int32).
int check_geom(const pkv_geom* g);

struct DeviceInfo {
    int device;
    int num_sms;
    size_t max_smem_optin;
    unsigned int* err;  // device address of this device's error word
};

// Looks up (once per device) the SM count, shared-memory limit and the error
// word's device address of the current device.
cudaError_t current_device_info(DeviceInfo* info);

cudaError_t launch_build_slot_mapping(const int32_t* block_table, int32_t max_blocks,
                                      int32_t num_seqs, const int32_t* token_seq,
                                      const int32_t* token_pos, int64_t num_tokens,
                                      int32_t block_size, int32_t* slot_mapping,
                                      unsigned int* err, cudaStream_t stream);

cudaError_t launch_kv_write(const void* k, const void* v, int src_dtype, const int32_t* slots,
                            int64_t num_tokens, void* k_cache, void* v_cache, int cache_dtype,
                            int64_t kv_dim, int64_t num_slots, unsigned int* err,
                            cudaStream_t stream);

// The slot build and the write in one launch (slots_out may be null).
cudaError_t launch_kv_write_positions(const void* k, const void* v, int src_dtype,
                                      const int32_t* block_table, int32_t max_blocks,
                                      int32_t num_seqs, const int32_t* token_seq,
                                      const int32_t* token_pos, int64_t num_tokens,
                                      int32_t block_size, int32_t* slots_out, void* k_cache,
                                      void* v_cache, int cache_dtype, int64_t kv_dim,
                                      int64_t num_slots, unsigned int* err, cudaStream_t stream);

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src,
                               const int32_t* dst, int32_t n_pairs, int64_t block_bytes,
                               int64_t num_blocks, unsigned int* err, cudaStream_t stream);

// ---- decode -----------------------------------------------------------------
struct DecodePlan {
    int heads_per_cta;   // KV heads one CTA handles (HC)
    int gsplit;          // consumer warps per KV head and row (each with Hq/Hkv/gsplit query heads)
    int head_groups;     // grid.y = Hkv / HC
    int ctas;            // grid.x (CTAs along the key axis)
    int rows_per_tile;   // R: keys per pipeline stage (divides block_size)
    int stages;          // pipeline depth
    size_t smem_bytes;   // dynamic shared memory per CTA
    size_t ws_bytes;     // workspace bytes needed
};

constexpr int kDecodeMaxBatch = 4096;

// Shared-prefix decode: groups of consecutive sequences share a prefix whose
// attention (normalised output and log2-sum-exp per sequence and head) was
// computed separately; the decode covers the keys after it and merges.
struct SharedPrefix {
    const int32_t* group_cu;    // [n_groups + 1]
    const int32_t* group_plen;  // [n_groups]
    int32_t n_groups;
    const void* x_out;          // [x_chunks, batch, hq, d] bf16
    const float* x_lse;         // [x_chunks, batch, hq]
    int32_t x_chunks;           // prefix partials per (sequence, head)
};

// In-place append: the new token of every sequence ([batch, hkv, d], the
// cache dtype) is attended to as key cache_seqlens[b] and written there.
struct DecodeAppend {
    const void* k_new;
    const void* v_new;
    void* k_cache;
    void* v_cache;
};

// Launch options of the decode pair: the split kernel as a programmatic
// dependent of the previous kernel (which it does not read), completing only
// after that kernel has (so the combine, which waits for the split, sees it).
struct DecodeChain {
    bool pdl_split;
    bool no_split;  // the prefix chunks hold every key: the combine alone follows them
};

// Returns false when the geometry is not supported.
bool plan_decode(const DeviceInfo& dev, int32_t batch, int hq, int hkv, int d, int block_size,
                 int elt, DecodePlan* plan);


cudaError_t launch_decode(const DecodePlan& plan, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* block_table, int32_t max_blocks,
                          const int32_t* cache_seqlens, int32_t batch, float scale, void* out,
                          void* workspace, int hq, int hkv, int d, int block_size,
                          int64_t num_blocks, int dtype, unsigned int* err, cudaStream_t stream,
                          const SharedPrefix* shared = nullptr,
                          const DecodeAppend* append = nullptr,
                          const DecodeChain* chain = nullptr);

// ---- shared-prefix pass (prefill.cu) -------------------------------------------
// For every group of consecutive sequences sharing their first group_plen[g]
// keys: attention of all the group's queries over those keys (in kchunks key
// chunks), written as normalised bf16 rows x_out [kchunks, batch, hq, hd] and
// log2-sum-exp x_lse [kchunks, batch, hq] for the decode's merge.
struct PrefixLaunch {
    const void* q;              // [batch, hq, hd] bf16
    const void* k_cache;
    const void* v_cache;
    const int32_t* table;       // [batch, max_blocks]; a group reads its first member's row
    const int32_t* group_cu;    // [n_groups + 1]; null: every sequence is a group of one
    const int32_t* group_plen;  // [n_groups]
    const int32_t* seqlens;     // groups of one: their prefix is the whole pieces of seqlens[g]
    void* x_out;
    float* x_lse;
    unsigned int* err;
    int64_t num_blocks;
    float scale;
    int32_t max_blocks, batch, hq, hkv, hd, block_size, n_groups, max_group_size, kchunks;
    int32_t chunk_keys;         // > 0: keys per chunk (a multiple of 128), else prefix / kchunks
    bool pdl;                   // launch as a programmatic dependent of the previous kernel
};

cudaError_t launch_prefix(const DeviceInfo& dev, const PrefixLaunch& p, cudaStream_t stream);

// The continuous-batching step in one launch (step.cu): the prefill rows'
// write, the prefix items and the causal prefill items, the decode split and
// the combine with the append, as CTAs of one grid ordered by block index and
// tied by counters.  bf16, head_dim 128, 2 query heads per KV head, one
// KV-head group per split CTA; cudaErrorNotSupported otherwise (before any
// launch).
struct StepOneLaunch {
    PrefixLaunch prefix;        // the decode groups' shared-prefix pass (q, table, groups)
    DecodePlan plan;            // the decode split's plan
    const void* pf_k_new;       // [pf_new_tokens, Hkv, d] bf16
    const void* pf_v_new;
    const int32_t* pf_slots;    // [pf_new_tokens]
    int64_t pf_new_tokens;
    const void* pf_q;           // [total_q, Hq, d]
    const int32_t* cu_q;
    const int32_t* cu_k;
    int32_t pf_batch, max_seqlen_q, pf_max_blocks;
    const int32_t* pf_table;
    void* pf_out;
    const void* dec_k_new;      // [decode batch, Hkv, d]
    const void* dec_v_new;
    const int32_t* dec_seqlens;
    void* dec_out;
    void* k_cache;
    void* v_cache;
    void* workspace;            // the decode split's workspace (plan.ws_bytes, then the prefix partials)
    unsigned int* counters;     // 4 words of device memory
    float scale;
    int hq, hkv, block_size, dtype;
    int64_t num_blocks;
};
cudaError_t launch_step_one(const DeviceInfo& dev, const StepOneLaunch& st, cudaStream_t stream);

// A causal varlen prefill (the arguments of launch_prefill) and a
// shared-prefix pass in ONE launch: the prefill's items wait for the kernel
// before them, the prefix items start at once, and the SMs take either kind
// as they free up.
cudaError_t launch_prefill_with_prefix(const DeviceInfo& dev, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* cu_q,
                                       const int32_t* cu_k, int32_t batch, int32_t max_seqlen_q,
                                       const int32_t* block_table, int32_t max_blocks,
                                       float scale, void* out, int hq, int hkv, int d,
                                       int block_size, int64_t num_blocks, unsigned int* err,
                                       const PrefixLaunch& p, cudaStream_t stream);

// ---- prefill ----------------------------------------------------------------
size_t prefill_workspace_bytes(int32_t batch, int32_t max_seqlen_q, int hq);

cudaError_t launch_prefill(const DeviceInfo& dev, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* cu_q, const int32_t* cu_k,
                           int32_t batch, int32_t max_seqlen_q, int32_t max_seqlen_k,
                           const int32_t* block_table, int32_t max_blocks, int causal,
                           float scale, void* out, void* workspace, int hq, int hkv, int d,
                           int block_size, int64_t num_blocks, unsigned int* err,
                           cudaStream_t stream);

}  // namespace pkv
