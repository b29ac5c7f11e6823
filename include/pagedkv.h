/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache attention library
 * (libpagedkv.so).
 *
 * The library implements the data-parallel hot path of paged attention:
 *   - the slot_mapping KV-cache write (new K/V rows scattered into the paged
 *     pool, negative slots skipped);
 *   - one-query-per-sequence decode that reads K/V through a block table and
 *     merges blocks with the online-softmax rule (split over the keys of long
 *     sequences, partial states merged by the same rule);
 *   - causal varlen prefill over cu_seqlens_q / cu_seqlens_k that reads the
 *     paged prior context (prefix cache / chunked prefill) on the tensor cores.
 *
 * Sources: "11. Paged attention 与 online softmax" (dilfish.github.io), §11.1
 * block table and offset equation, §11.2 boxed merge equation;
 * "从零开始写Qwen3（六）PagedAttention" (mlqm.cn), sections "fast-attn 库的使用"
 * (the varlen / kvcache call shapes and their parameters) and "自己来实现一个"
 * (the slot_mapping write kernel); "Sayfalı dikkat" (Hugging Face transformers
 * docs), varlen path (cu_seq_lens) and decode path (block_table, cache_seqlens).
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory.  Every pointer argument is a DEVICE pointer unless stated otherwise
 * (pkv_geom is read on the host).  The caller owns every buffer; the library
 * allocates no device memory.  Calls are asynchronous on `stream` and never
 * synchronise the host, except paged_error_flags.
 * Ordering.  Work enqueued on `stream` before a call completes before the
 * call reads anything, and work enqueued after it sees all of its results,
 * as for any stream-ordered launch.  The library's kernels are launched as
 * programmatic dependents of the kernel before them and let the next kernel
 * launch early (programmatic dependent launch).  This matters only to a
 * caller kernel that is itself launched after a call with the
 * programmatic-stream-serialization attribute: it may start before the call's
 * kernels finish, and must execute griddepcontrol.wait
 * (cudaGridDependencySynchronize) before it reads their results.
 * Layouts (row-major, contiguous):
 *   K/V pools  [num_blocks, block_size, num_kv_heads, head_dim]; the element
 *              offset of logical position p of a sequence whose block-table row
 *              is t is (t[p / B] * B + p % B) * kvDim, kvDim = Hkv * head_dim.
 *   block_table [rows, max_blocks_per_seq] int32; entries past a sequence's
 *              length are never read and may hold -1.
 *   q / out    decode [batch, Hq, head_dim]; prefill [total_q, Hq, head_dim].
 *   index arrays are int32.
 * GQA: query head h reads KV head h / (Hq / Hkv).
 * dtype: q, out and both pools share pkv_geom.dtype.
 * Return codes: PKV_OK, or a negative PKV_ERR_* (no work is enqueued then).
 * Device-side checks: an out-of-range block id, slot or sequence length found
 * while a kernel runs is skipped (never dereferenced) and recorded in a
 * per-device error word read by paged_error_flags.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types */
typedef enum pkv_dtype { PKV_F32 = 0, PKV_BF16 = 1 } pkv_dtype;

/* status codes */
#define PKV_OK 0
#define PKV_ERR_INVALID (-1)     /* null pointer, bad size, Hq % Hkv != 0, misaligned */
#define PKV_ERR_UNSUPPORTED (-2) /* valid but not implemented (dtype/head_dim/GQA combo) */
#define PKV_ERR_WORKSPACE (-3)   /* workspace missing or smaller than the *_workspace_size */
#define PKV_ERR_CUDA (-4)        /* a CUDA runtime call or kernel launch failed */
#define PKV_ERR_NO_SPACE (-5)    /* block manager: not enough free blocks (nothing changed) */

/* device error-word bits (paged_error_flags) */
#define PKV_FLAG_BAD_BLOCK (1u << 0)   /* block-table entry outside [0, num_blocks) */
#define PKV_FLAG_BAD_SLOT (1u << 1)    /* slot_mapping entry >= num_blocks * block_size */
#define PKV_FLAG_BAD_LENGTH (1u << 2)  /* length < 0 or beyond max_blocks_per_seq * B */
#define PKV_FLAG_BAD_SEQ (1u << 3)     /* token sequence index >= num_seqs */
#define PKV_FLAG_TIMEOUT (1u << 4)     /* a pipeline wait gave up (kernel returned early) */

/* Geometry of one paged pool (one layer's K pool and V pool). */
typedef struct pkv_geom {
    int32_t num_heads;    /* Hq, query heads */
    int32_t num_kv_heads; /* Hkv, KV heads; Hq % Hkv == 0 */
    int32_t head_dim;     /* d */
    int32_t block_size;   /* B, tokens per physical block (page) */
    int64_t num_blocks;   /* physical blocks in each pool */
    int32_t dtype;        /* pkv_dtype of q, out and the pools */
} pkv_geom;

/*
 * paged_build_slot_mapping -- address translation for the new tokens of a step.
 * ("11. Paged attention 与 online softmax" §11.1: logical block p / B, slot
 * p mod B, phys = table[p / B]; "自己来实现一个": the per-token index is
 * computed once and reused by every layer.)
 *   slot_mapping[n] = block_table[s][p / B] * B + p % B with s = token_seq[n],
 *   p = token_pos[n]; token_seq[n] < 0 marks a padding row -> -1.
 *   block_table [num_seqs, max_blocks_per_seq]; token_seq, token_pos,
 *   slot_mapping [num_tokens].  Out-of-range s, p or table entries give -1 and
 *   set PKV_FLAG_BAD_SEQ / _BAD_LENGTH / _BAD_BLOCK.
 */
int paged_build_slot_mapping(const int32_t* block_table, int32_t max_blocks_per_seq,
                             int32_t num_seqs, const int32_t* token_seq,
                             const int32_t* token_pos, int64_t num_tokens, int32_t block_size,
                             int32_t* slot_mapping, cudaStream_t stream);

/*
 * paged_kv_write -- the slot_mapping cache write ("自己来实现一个",
 * _update_paged_kv_cache_kernel).  For every token n with s = slot_mapping[n]
 * >= 0: k_cache[s*kvDim + j] = cast(k[n*kvDim + j]) and likewise for v,
 * j < kvDim; s < 0 writes nothing.  k, v [num_tokens, Hkv, d] of kv_dtype; the
 * pools of geom->dtype.  fp32 -> bf16 rounds to nearest even; equal dtypes
 * copy bits.  Duplicate non-negative slots are a caller error (the surviving
 * row is unspecified).  s >= num_blocks*B is skipped and sets PKV_FLAG_BAD_SLOT.
 */
int paged_kv_write(const void* k, const void* v, int32_t kv_dtype, const int32_t* slot_mapping,
                   int64_t num_tokens, void* k_cache, void* v_cache, const pkv_geom* geom,
                   cudaStream_t stream);

/*
 * paged_kv_write_positions -- paged_build_slot_mapping and paged_kv_write in
 * one launch: token n's slot is block_table[s][p / B] * B + p % B with
 * s = token_seq[n], p = token_pos[n] ("11. Paged attention 与 online softmax"
 * §11.1; "自己来实现一个" computes it once per step for every layer), and its
 * K and V rows are written there as paged_kv_write does.  The slots are also
 * stored in slot_mapping_out [num_tokens] when it is not NULL, so that the
 * other layers of the step can call paged_kv_write with them.  token_seq[n] < 0
 * marks a padding row (slot -1, nothing written).  Out-of-range s, p or table
 * entries give slot -1 (nothing written) and set PKV_FLAG_BAD_SEQ /
 * _BAD_LENGTH / _BAD_BLOCK; a slot >= num_blocks * B sets PKV_FLAG_BAD_SLOT.
 * Arguments as for the two calls it replaces.
 */
int paged_kv_write_positions(const void* k, const void* v, int32_t kv_dtype,
                             const int32_t* block_table, int32_t max_blocks_per_seq,
                             int32_t num_seqs, const int32_t* token_seq,
                             const int32_t* token_pos, int64_t num_tokens,
                             int32_t* slot_mapping_out, void* k_cache, void* v_cache,
                             const pkv_geom* geom, cudaStream_t stream);

/*
 * paged_decode_workspace_size -- bytes of device scratch paged_decode needs for
 * `batch` sequences on the CURRENT device (the split plan depends on its SM
 * count).  Returns 0 for invalid arguments.  There is no max_seqlen_k
 * argument: the keys of all sequences are cut into one share per CTA, so the
 * scratch holds (CTAs + batch) partial states whatever the lengths are, and
 * the lengths themselves are device data the host need not know.  On the
 * tensor-core path (below) it adds c partial states per (sequence, query
 * head), c = min(32, ceil(SMs / (batch * Hkv))).
 */
size_t paged_decode_workspace_size(int32_t batch, const pkv_geom* geom);

/*
 * paged_decode -- paged attention of one query token per sequence ("Sayfalı
 * dikkat" decode path; "11. Paged attention 与 online softmax" §11.1-§11.2).
 * Sequence b attends over exactly cache_seqlens[b] keys (positions 0 ..
 * cache_seqlens[b]-1, read through block_table row b), i.e. the new token's
 * K/V must already have been written with paged_kv_write.
 *   out[b,h,:] = sum_j softmax_j(scale * q[b,h,:] . k_j) v_j  over those keys,
 *   0 when cache_seqlens[b] == 0.
 * The keys of all sequences are cut into shares, one per CTA (equal once each
 * sequence start is counted as one tile of keys); each CTA keeps the (m, l, o)
 * online-softmax state of its share and a second kernel merges the shares of
 * each sequence with the same rule and normalises.
 * Tensor-core path: bf16 with G = Hq/Hkv >= 4 (and dividing 128), and block
 * sizes the shared-prefix pass takes (multiples of 128, or divisors of 128 of
 * at least 8).  There the keys of each sequence are attended on the tensor
 * cores in c chunks of ceil(max_blocks_per_seq * B / c) keys rounded up to
 * 128, one work item per (sequence, KV head, chunk) with the G query heads as
 * rows of one MMA tile (keys past the length in the last page are masked, and
 * their V rows zeroed in shared memory); the same second kernel merges the
 * chunks' states (two launches, no split).
 * Supported: head_dim 64 or 128; fp32 or bf16; G = Hq/Hkv in {1, 2, 4, 8, 16,
 * 32} (from 8 up, G/4 warps per KV head, 4 query heads each, share its K/V
 * tiles); with s = 8 / max(1, G/4) KV heads per CTA, Hkv divides s or is a
 * multiple of s; any block_size >= 1; batch <= 4096.
 * Like its workspace-size call it takes no max_seqlen_k: nothing in the launch
 * depends on the longest sequence.
 * workspace: device scratch of at least paged_decode_workspace_size(batch, geom)
 * bytes, 256-byte aligned, contents irrelevant on entry; it must not be used by
 * another call that runs concurrently.
 */
int paged_decode(const void* q, const void* k_cache, const void* v_cache,
                 const int32_t* block_table, int32_t max_blocks_per_seq,
                 const int32_t* cache_seqlens, int32_t batch, float scale, void* out,
                 void* workspace, size_t workspace_bytes, const pkv_geom* geom,
                 cudaStream_t stream);

/*
 * paged_decode_append -- paged_decode with the in-place append of the new
 * token ("Sayfalı dikkat" decode path: the flash_attn_with_kvcache call takes
 * the new k and v, writes them into the cache and attends over them together
 * with the cached keys).  cache_seqlens[b] counts the keys cached BEFORE this
 * step.  For every sequence b:
 *   - k_new[b], v_new[b] ([batch, Hkv, d], the cache dtype) are written at
 *     position cache_seqlens[b] (slot = block_table[b][L / B] * B + L % B);
 *   - out[b,h] = attention of q[b,h] over the cache_seqlens[b] cached keys
 *     and the new key (cache_seqlens[b] + 1 keys in all).
 * The caller advances cache_seqlens afterwards.  The new key is scored from
 * k_new directly (not read back from the cache) and written after the cached
 * keys have been read.  Supported, workspace and errors as paged_decode (same
 * workspace size); a position past max_blocks_per_seq * B or a bad table
 * entry skips that write and sets PKV_FLAG_BAD_LENGTH / _BAD_BLOCK.
 */
int paged_decode_append(const void* q, const void* k_new, const void* v_new, void* k_cache,
                        void* v_cache, const int32_t* block_table, int32_t max_blocks_per_seq,
                        const int32_t* cache_seqlens, int32_t batch, float scale, void* out,
                        void* workspace, size_t workspace_bytes, const pkv_geom* geom,
                        cudaStream_t stream);

/*
 * paged_varlen_prefill_workspace_size -- bytes of device scratch
 * paged_varlen_prefill needs (0 when it needs none).  Returns 0 for invalid
 * arguments as well.
 */
size_t paged_varlen_prefill_workspace_size(int32_t batch, int32_t max_seqlen_q,
                                           const pkv_geom* geom);

/*
 * paged_varlen_prefill -- causal varlen prefill over a paged cache
 * ("从零开始写Qwen3（六）PagedAttention", "fast-attn 库的使用": prefix cache and
 * chunked prefill read the cache through block_table; "Sayfalı dikkat" varlen
 * path).  Request r owns query rows [cu_seqlens_q[r], cu_seqlens_q[r+1]) of q
 * and keys 0 .. k_len-1, k_len = cu_seqlens_k[r+1] - cu_seqlens_k[r], read
 * through block_table row r (the new tokens' K/V must already be written).
 * With causal != 0 query i of a request with q_len queries sees key j iff
 * j <= i + k_len - q_len (bottom-right alignment: the queries are the last
 * q_len positions); a row that sees no key outputs 0.
 * max_seqlen_q / max_seqlen_k are host-side upper bounds of the per-request
 * lengths (they size the launch).  q, out [total_q, Hq, d].
 * Contiguous mode ("从零开始写Qwen3（六）PagedAttention", "一个小细节": without
 * a prefix cache the varlen call reads packed K/V): block_table == NULL makes
 * k_cache / v_cache packed arrays [rows, Hkv, d] with rows = geom->num_blocks
 * * geom->block_size (any factorisation, e.g. block_size 1), and request r's
 * keys are rows cu_seqlens_k[r] .. cu_seqlens_k[r+1]-1; max_blocks_per_seq is
 * ignored.  Keys past row `rows` are flagged PKV_FLAG_BAD_LENGTH.
 * Supported: bf16, head_dim 64 or 128, Hq/Hkv in {1, 2, 4, 8, ...}; paged
 * mode: a block_size that is a multiple of 128 or divides 128 and is >= 8.
 */
int paged_varlen_prefill(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int32_t batch,
                         int32_t max_seqlen_q, int32_t max_seqlen_k, const int32_t* block_table,
                         int32_t max_blocks_per_seq, int32_t causal, float scale, void* out,
                         void* workspace, size_t workspace_bytes, const pkv_geom* geom,
                         cudaStream_t stream);

/*
 * paged_decode_shared_prefix -- paged_decode for batches whose sequences come
 * in groups that share the physical blocks of a common prefix ("11. Paged
 * attention 与 online softmax" §11.3 block sharing; the prefix cache of
 * "结合nanovllm的FlashAttention和PagedAttention主要原理概述" 题目6), reading each
 * shared block once per group instead of once per sequence.
 *   group_cu [n_groups + 1] (device): group g is sequences group_cu[g] ..
 *   group_cu[g+1]-1 of the batch (group_cu[0] = 0, group_cu[n_groups] =
 *   batch: the batch is ordered by group; a sequence sharing nothing is a
 *   group of one with prefix 0).  group_prefix_len [n_groups] (device): the
 *   leading keys every sequence of group g holds in the same physical blocks,
 *   a multiple of block_size and at most each member's cache_seqlens; the
 *   prefix blocks are read through the table row of the group's first
 *   sequence.  max_group_size: a host-side bound of the group sizes.
 * The result is paged_decode's (same arguments and layouts otherwise): the
 * prefix part is the attention of the group's queries over the prefix keys
 * (one pass over them, on the tensor cores), the rest the decode of each
 * sequence's own keys, merged with §11.2's boxed rule.
 * Supported: bf16, head_dim 64 or 128, Hq/Hkv and Hkv as for paged_decode,
 * block_size a multiple of 128 or a divisor of 128 (>= 8).
 * workspace: at least
 * paged_decode_shared_prefix_workspace_size(batch, geom) bytes, 256-byte
 * aligned.  A prefix length that is negative, longer than a member's keys or
 * not a multiple of block_size sets PKV_FLAG_BAD_LENGTH.
 */
size_t paged_decode_shared_prefix_workspace_size(int32_t batch, const pkv_geom* geom);
int paged_decode_shared_prefix(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int32_t max_blocks_per_seq,
                               const int32_t* cache_seqlens, int32_t batch,
                               const int32_t* group_cu, const int32_t* group_prefix_len,
                               int32_t n_groups, int32_t max_group_size, float scale, void* out,
                               void* workspace, size_t workspace_bytes, const pkv_geom* geom,
                               cudaStream_t stream);

/*
 * paged_mixed_step -- one continuous-batching step in one call: prefill
 * requests and decode sequences over the same pools ("从零开始写Qwen3（六）
 * PagedAttention", "fast-attn 库的使用": the varlen call for prefill, the
 * kvcache call for decode; "11. Paged attention 与 online softmax" §11.3 for
 * groups sharing a prefix).  In order on `stream`:
 *   1. the prefill requests' new K/V rows are written at prefill_slots
 *      (paged_kv_write; negative slots skipped);
 *   2. causal varlen prefill of the prefill requests (paged_varlen_prefill);
 *   3. decode of the decode sequences with the in-place append
 *      (paged_decode_append), through the shared-prefix path when n_groups > 0
 *      (paged_decode_shared_prefix semantics).
 * Parts with a zero count are skipped.  The decode kernels are launched as
 * programmatic dependents of the prefill kernel, which they do not read: they
 * start on SMs the prefill leaves free instead of after it.  Arguments mean
 * what they mean in the single calls; all pointers in the struct are DEVICE
 * pointers.  Supported as the single calls; with a prefill part or groups:
 * bf16 and head_dim 64 or 128.  workspace: at least
 * paged_mixed_step_workspace_size(decode_batch, geom) bytes, 256-byte aligned.
 */
typedef struct pkv_mixed_step {
    /* prefill requests */
    const void* prefill_k_new;   /* [prefill_new_tokens, Hkv, d] */
    const void* prefill_v_new;
    const int32_t* prefill_slots; /* [prefill_new_tokens] */
    int64_t prefill_new_tokens;
    const void* prefill_q;        /* [total_q, Hq, d] */
    const int32_t* cu_seqlens_q;  /* [prefill_batch + 1] */
    const int32_t* cu_seqlens_k;
    int32_t prefill_batch;
    int32_t max_seqlen_q;
    int32_t max_seqlen_k;
    const int32_t* prefill_table; /* [prefill_batch, prefill_max_blocks] */
    int32_t prefill_max_blocks;
    void* prefill_out;            /* [total_q, Hq, d] */
    /* decode sequences (in-place append) */
    const void* decode_q;         /* [decode_batch, Hq, d] */
    const void* decode_k_new;     /* [decode_batch, Hkv, d] */
    const void* decode_v_new;
    const int32_t* decode_table;  /* [decode_batch, decode_max_blocks] */
    int32_t decode_max_blocks;
    const int32_t* decode_seqlens; /* keys cached before the step */
    int32_t decode_batch;
    const int32_t* group_cu;      /* [n_groups + 1], or NULL with n_groups 0 */
    const int32_t* group_prefix_len;
    int32_t n_groups;
    int32_t max_group_size;
    void* decode_out;             /* [decode_batch, Hq, d] */
    float scale;
} pkv_mixed_step;

size_t paged_mixed_step_workspace_size(int32_t decode_batch, const pkv_geom* geom);
int paged_mixed_step(const pkv_mixed_step* step, void* k_cache, void* v_cache, void* workspace,
                     size_t workspace_bytes, const pkv_geom* geom, cudaStream_t stream);

/*
 * paged_mixed_step_one_launch -- paged_mixed_step's result from ONE kernel
 * launch (plus a 16-byte memset of its counters): the prefill rows' write, the
 * shared-prefix and causal-prefill work items on the tensor cores, the decode
 * split and the combine with the append run as CTAs of one grid, in that
 * order of block index; a CTA that needs earlier results (a prefill item the
 * write, a combine CTA the prefix items and the split) waits until their
 * counters are complete (time-limited: PKV_FLAG_TIMEOUT).  Same arguments,
 * workspace and errors as paged_mixed_step.  It takes full steps (prefill
 * rows, prefill requests and grouped decode sequences) in bf16, head_dim 128,
 * with 2 query heads per KV head and at most 8 KV heads; any other step is done
 * by paged_mixed_step.  paged_mixed_step is faster on GB300 (each phase keeps
 * its own CTA shape there); this form is for callers that need a single
 * kernel launch.
 */
int paged_mixed_step_one_launch(const pkv_mixed_step* step, void* k_cache, void* v_cache,
                                void* workspace, size_t workspace_bytes, const pkv_geom* geom,
                                cudaStream_t stream);

/*
 * paged_decode_noalloc -- paged_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart: this is a deployment variant of
 * paged_decode that takes no workspace.
 * Some callers cannot hand the library a scratch buffer: a plugin whose host
 * framework owns every device allocation and offers no workspace hook, or a
 * serving loop that must not call cudaMalloc because it can synchronise the
 * device and stall other streams.  This call allocates nothing (no cudaMalloc,
 * no cudaFree, no allocating library routine); its split-KV scratch is a fixed
 * device array of PKV_NOALLOC_SCRATCH_BYTES inside the library, which every
 * GPU that loads the library holds until the process exits.
 *   - Same arguments, layouts, results and support matrix as paged_decode,
 *     minus workspace / workspace_bytes.  It always takes the CUDA-core split
 *     (never paged_decode's tensor-core path), whose scratch is the array.
 *   - Returns PKV_ERR_WORKSPACE when the split needs more scratch than the
 *     array holds.  That scratch is about
 *     (SMs + batch) * Hq * (head_dim + 2) * 4 bytes, so the limit is
 *     batch <= PKV_NOALLOC_SCRATCH_BYTES / (Hq * (head_dim + 2) * 4) - SMs:
 *     about 850 sequences for Hq=16, head_dim=128 on a 152-SM GPU.
 *   - All calls share the one array, and it keeps the previous call's contents
 *     (nothing in it needs to start at zero).  Calls that overlap on the GPU
 *     race on it: order them on one stream or with events.
 *   - Set-up: the first call on each device looks up the array's device
 *     address (cudaGetSymbolAddress) with that device current.  Under lazy
 *     module loading (the CUDA default) that lookup also loads the module that
 *     holds the array, which may allocate and synchronise.  A call with
 *     batch 0 does this set-up alone (and nothing else): make it once per
 *     device at initialisation, before any stream capture, or run with
 *     CUDA_MODULE_LOADING=EAGER.  The looked-up address is cached; after
 *     cudaDeviceReset the library must not be used on that device again.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (8u << 20)
int paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_table, int32_t max_blocks_per_seq,
                         const int32_t* cache_seqlens, int32_t batch, float scale, void* out,
                         const pkv_geom* geom, cudaStream_t stream);

/*
 * paged_error_flags -- read (and with clear != 0, reset) the device error word
 * of the current device: an OR of PKV_FLAG_* bits set by kernels since the
 * last clear.  *flags (host pointer) receives the word.
 * This call SYNCHRONISES with the device (it copies the word to the host with
 * cudaMemcpy), unlike every other call here: use it between steps, not on a
 * latency-critical path.  It replaces a plain int-returning "last error"
 * call: the word is a set of independent flag bits, so it is returned through
 * a pointer beside the status, and reading without clearing is possible.
 */
int paged_error_flags(uint32_t* flags, int32_t clear);

/*
 * Block manager (host side) and block copies -- "11. Paged attention 与 online
 * softmax" §11.3 (block sharing, copy-on-write, reference counts and the free
 * stack) and "结合nanovllm的FlashAttention和PagedAttention主要原理概述" 题目6
 * (prefix cache: chained block hashes, a hit shares the block, release in
 * reverse block order).
 *
 * A pkv_block_manager owns the bookkeeping of one pool of num_blocks blocks of
 * block_size tokens and the sequences that hold them; it makes no CUDA call and
 * is not thread-safe (callers serialise).  Every pointer of the paged_bm_*
 * calls is a HOST pointer.
 *   - refs[b] = the number of sequence block tables that contain block b; a
 *     block with refs 0 is on the free stack (top = block 0 at creation; a
 *     released block is pushed on top, allocation pops the top).
 *   - Only full blocks are shared by lookup.  The cache key of block i of a
 *     token sequence is (the physical block of block i-1, or -1; the block's
 *     block_size token ids), compared in full: two sequences share their
 *     leading full blocks exactly as far as their tokens agree.
 *   - PKV_ERR_NO_SPACE leaves the manager unchanged.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* a manager of num_blocks (< 2^31) blocks of block_size (>= 1) tokens */
int paged_bm_create(int64_t num_blocks, int32_t block_size, pkv_block_manager** out);
int paged_bm_destroy(pkv_block_manager* bm);

/* New sequence holding tokens[0 .. n_tokens): its leading full blocks that are
 * cached are shared (refs +1), the rest are allocated (refs 1) and the full
 * ones cached.  *seq_out: the sequence id; *cached_tokens_out (may be NULL):
 * tokens in shared blocks, i.e. tokens whose K/V are already in the pool. */
int paged_bm_allocate(pkv_block_manager* bm, const int64_t* tokens, int64_t n_tokens,
                      int64_t* seq_out, int64_t* cached_tokens_out);

/* New sequence with the same tokens and blocks as `seq` (every block refs +1). */
int paged_bm_fork(pkv_block_manager* bm, int64_t seq, int64_t* child_out);

/* One more token for `seq`.  A full last block gets a new block after it; a
 * partial last block that is shared (refs > 1) is replaced by a new block the
 * sequence owns and *cow_src_out / *cow_dst_out name the block whose contents
 * must be copied first (paged_copy_blocks) -- otherwise both are -1.  A block
 * that the token fills enters the cache. */
int paged_bm_append(pkv_block_manager* bm, int64_t seq, int64_t token, int32_t* cow_src_out,
                    int32_t* cow_dst_out);

/* Release a sequence: its blocks in reverse order, refs -1 each; a block at 0
 * leaves the cache and is pushed on the free stack. */
int paged_bm_free(pkv_block_manager* bm, int64_t seq);

/* The sequence's block table (host int32 array of `capacity` entries);
 * *n_blocks_out receives its length (also when capacity is too small, which
 * returns PKV_ERR_INVALID). */
int paged_bm_block_table(const pkv_block_manager* bm, int64_t seq, int32_t* table_out,
                         int32_t capacity, int32_t* n_blocks_out);
int paged_bm_seq_len(const pkv_block_manager* bm, int64_t seq, int64_t* len_out);
int paged_bm_ref_count(const pkv_block_manager* bm, int32_t block, int32_t* ref_out);

/* The free stack, bottom first, into stack_out[capacity] (NULL: count only);
 * *n_out receives the number of free blocks. */
int paged_bm_free_blocks(const pkv_block_manager* bm, int32_t* stack_out, int64_t capacity,
                         int64_t* n_out);

/*
 * paged_copy_blocks -- the copies a copy-on-write needs (§11.3: the old
 * contents go into the new block before the write).  For i < n_pairs, block
 * dst[i] of both pools becomes a bitwise copy of block src[i] (block_size *
 * kvDim elements of geom->dtype).  src, dst: DEVICE int32 arrays; a dst block
 * must not also be a src block or appear twice (the result is unspecified
 * then).  An id outside [0, num_blocks) skips the pair and sets
 * PKV_FLAG_BAD_BLOCK.
 */
int paged_copy_blocks(void* k_cache, void* v_cache, const int32_t* src, const int32_t* dst,
                      int32_t n_pairs, const pkv_geom* geom, cudaStream_t stream);

/* paged_status_string -- static text for a PKV_* status code. */
const char* paged_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
