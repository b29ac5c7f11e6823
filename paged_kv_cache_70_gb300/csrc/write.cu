// write.cu -- slot_mapping construction and the paged KV-cache write.
//
// "从零开始写Qwen3（六）PagedAttention", section "自己来实现一个": the slot of
// every new token is computed once per step (shared by all layers), then each
// token's K and V rows are copied to cache[slot * kvDim ...] with a cast to the
// cache dtype; a negative slot is skipped.  Addressing follows
// "11. Paged attention 与 online softmax" §11.1 (slot = table[p/B]*B + p%B).
//
// GB300 layout of the write: one warp per token row; each lane moves 16-byte
// vectors of the K row and of the V row (2 KiB rows for Hkv=8, d=128, bf16), so
// a warp issues fully coalesced 512-byte transactions.  The kernel is HBM-bound
// (2 * kvDim * elt bytes read and written per token).
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace pkv {

// The slot of token n: table[s][p / B] * B + p % B for s = token_seq[n],
// p = token_pos[n]; -1 for a padding row (s < 0) or an out-of-range s, p or
// table entry (flagged).
struct TokenSlots {
    const int32_t* table;
    int32_t max_blocks;
    int32_t num_seqs;
    const int32_t* token_seq;
    const int32_t* token_pos;
    int32_t block_size;
};

__device__ __forceinline__ int32_t token_slot(const TokenSlots& t, int64_t n, unsigned int* err) {
    const int32_t s = t.token_seq[n];
    const int32_t p = t.token_pos[n];
    if (s < 0) return -1;
    if (s >= t.num_seqs) {
        flag_error(err, PKV_FLAG_BAD_SEQ);
        return -1;
    }
    if (p < 0 || p / t.block_size >= t.max_blocks) {
        flag_error(err, PKV_FLAG_BAD_LENGTH);
        return -1;
    }
    const int32_t phys = t.table[(int64_t)s * t.max_blocks + p / t.block_size];
    if (phys < 0) {
        flag_error(err, PKV_FLAG_BAD_BLOCK);
        return -1;
    }
    return phys * t.block_size + p % t.block_size;
}

__global__ void build_slot_mapping_kernel(const TokenSlots t, int64_t num_tokens,
                                          int32_t* __restrict__ slots, unsigned int* err) {
    PKV_DEPENDENT_PROLOGUE();
    int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= num_tokens) return;
    slots[n] = token_slot(t, n, err);
}

cudaError_t launch_build_slot_mapping(const int32_t* block_table, int32_t max_blocks,
                                      int32_t num_seqs, const int32_t* token_seq,
                                      const int32_t* token_pos, int64_t num_tokens,
                                      int32_t block_size, int32_t* slot_mapping,
                                      unsigned int* err, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (num_tokens + threads - 1) / threads;
    const TokenSlots t{block_table, max_blocks, num_seqs, token_seq, token_pos, block_size};
    return launch_dependent(build_slot_mapping_kernel, dim3((unsigned)blocks), dim3(threads), 0,
                            stream, t, num_tokens, slot_mapping, err);
}

// ---------------------------------------------------------------------------
// write kernels
// ---------------------------------------------------------------------------
constexpr int kWriteWarps = 8;

// The slot of the warp's token: read from the slot mapping, or (POS) computed
// from the token's sequence and position by lane 0 and, when slots_out is
// given, stored there for the writes of later layers.
template <bool POS>
__device__ __forceinline__ int32_t warp_token_slot(const int32_t* slots, const TokenSlots& t,
                                                   int32_t* slots_out, int64_t n, int lane,
                                                   unsigned int* err) {
    if constexpr (!POS) {
        return __ldg(slots + n);
    } else {
        int32_t s = 0;
        if (lane == 0) {
            s = token_slot(t, n, err);
            if (slots_out) slots_out[n] = s;
        }
        return __shfl_sync(0xffffffffu, s, 0);
    }
}

// equal dtypes: 16-byte vector copy of row_bytes (a multiple of 16).  The
// first kPrefetch vectors of the K and V rows a lane copies are loaded before
// the slot is known (the source rows do not depend on it), so the slot
// lookup's latency overlaps theirs; a row that is not written (padding or a
// bad slot) wastes those loads only.
constexpr int kPrefetch = 4;

template <bool POS>
__global__ void __launch_bounds__(kWriteWarps * 32)
kv_write_copy_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                     const int32_t* __restrict__ slots, const TokenSlots t,
                     int32_t* __restrict__ slots_out, int64_t num_tokens,
                     uint4* __restrict__ kc, uint4* __restrict__ vc, int64_t vec_per_row,
                     int64_t num_slots, unsigned int* err) {
    PKV_DEPENDENT_PROLOGUE();
    const int lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
    if (n >= num_tokens) return;
    const uint4* ks = k + n * vec_per_row;
    const uint4* vs = v + n * vec_per_row;
    uint4 ka[kPrefetch], va[kPrefetch];
#pragma unroll
    for (int u = 0; u < kPrefetch; ++u) {
        const int64_t i = lane + 32 * u;
        if (i < vec_per_row) {
            ka[u] = __ldcs(ks + i);
            va[u] = __ldcs(vs + i);
        }
    }
    const int32_t s = warp_token_slot<POS>(slots, t, slots_out, n, lane, err);
    if (s < 0) return;
    if (s >= num_slots) {
        if (lane == 0) flag_error(err, PKV_FLAG_BAD_SLOT);
        return;
    }
    uint4* kd = kc + (int64_t)s * vec_per_row;
    uint4* vd = vc + (int64_t)s * vec_per_row;
#pragma unroll
    for (int u = 0; u < kPrefetch; ++u) {
        const int64_t i = lane + 32 * u;
        if (i < vec_per_row) {
            kd[i] = ka[u];
            vd[i] = va[u];
        }
    }
    for (int64_t i = lane + 32 * kPrefetch; i < vec_per_row; i += 32) {
        const uint4 a = __ldcs(ks + i);
        const uint4 b = __ldcs(vs + i);
        kd[i] = a;
        vd[i] = b;
    }
}

// fp32 source -> bf16 cache (round to nearest even); groups of 8 elements
template <bool POS>
__global__ void __launch_bounds__(kWriteWarps * 32)
kv_write_f32_to_bf16_kernel(const float4* __restrict__ k, const float4* __restrict__ v,
                            const int32_t* __restrict__ slots, const TokenSlots t,
                            int32_t* __restrict__ slots_out, int64_t num_tokens,
                            uint4* __restrict__ kc, uint4* __restrict__ vc, int64_t groups8,
                            int64_t num_slots, unsigned int* err) {
    PKV_DEPENDENT_PROLOGUE();
    const int lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
    if (n >= num_tokens) return;
    const int32_t s = warp_token_slot<POS>(slots, t, slots_out, n, lane, err);
    if (s < 0) return;
    if (s >= num_slots) {
        if (lane == 0) flag_error(err, PKV_FLAG_BAD_SLOT);
        return;
    }
    for (int64_t i = lane; i < groups8; i += 32) {
        const float4 a0 = __ldcs(k + (n * groups8 + i) * 2);
        const float4 a1 = __ldcs(k + (n * groups8 + i) * 2 + 1);
        const float4 b0 = __ldcs(v + (n * groups8 + i) * 2);
        const float4 b1 = __ldcs(v + (n * groups8 + i) * 2 + 1);
        kc[(int64_t)s * groups8 + i] = make_uint4(pack_bf16x2(a0.x, a0.y), pack_bf16x2(a0.z, a0.w),
                                                  pack_bf16x2(a1.x, a1.y), pack_bf16x2(a1.z, a1.w));
        vc[(int64_t)s * groups8 + i] = make_uint4(pack_bf16x2(b0.x, b0.y), pack_bf16x2(b0.z, b0.w),
                                                  pack_bf16x2(b1.x, b1.y), pack_bf16x2(b1.z, b1.w));
    }
}

// generic element-wise path: any kvDim, any dtype pair
template <bool POS>
__global__ void kv_write_scalar_kernel(const void* __restrict__ k, const void* __restrict__ v,
                                       int src_dtype, const int32_t* __restrict__ slots,
                                       const TokenSlots t, int32_t* __restrict__ slots_out,
                                       int64_t num_tokens, void* __restrict__ kc,
                                       void* __restrict__ vc, int cache_dtype, int64_t kv_dim,
                                       int64_t num_slots, unsigned int* err) {
    PKV_DEPENDENT_PROLOGUE();
    const int lane = threadIdx.x & 31;
    const int64_t n = (int64_t)blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
    if (n >= num_tokens) return;
    const int32_t s = warp_token_slot<POS>(slots, t, slots_out, n, lane, err);
    if (s < 0) return;
    if (s >= num_slots) {
        if (lane == 0) flag_error(err, PKV_FLAG_BAD_SLOT);
        return;
    }
    for (int64_t j = lane; j < kv_dim; j += 32) {
        const int64_t si = n * kv_dim + j, di = (int64_t)s * kv_dim + j;
        float a, b;
        if (src_dtype == PKV_F32) {
            a = static_cast<const float*>(k)[si];
            b = static_cast<const float*>(v)[si];
        } else {
            a = __uint_as_float((uint32_t) static_cast<const uint16_t*>(k)[si] << 16);
            b = __uint_as_float((uint32_t) static_cast<const uint16_t*>(v)[si] << 16);
        }
        if (cache_dtype == PKV_F32) {
            static_cast<float*>(kc)[di] = a;
            static_cast<float*>(vc)[di] = b;
        } else if (src_dtype == PKV_BF16) {  // bf16 -> bf16: bit copy
            static_cast<uint16_t*>(kc)[di] = static_cast<const uint16_t*>(k)[si];
            static_cast<uint16_t*>(vc)[di] = static_cast<const uint16_t*>(v)[si];
        } else {
            static_cast<uint16_t*>(kc)[di] = f32_to_bf16_bits(a);
            static_cast<uint16_t*>(vc)[di] = f32_to_bf16_bits(b);
        }
    }
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One write launch; with `pos` the slots come from the tokens' sequences and
// positions (and are stored in pos->slots_out when given), else from `slots`.
template <bool POS>
static cudaError_t launch_write_t(const void* k, const void* v, int src_dtype,
                                  const int32_t* slots, const TokenSlots& t, int32_t* slots_out,
                                  int64_t num_tokens, void* k_cache, void* v_cache,
                                  int cache_dtype, int64_t kv_dim, int64_t num_slots,
                                  unsigned int* err, cudaStream_t stream) {
    if (num_tokens == 0) return cudaSuccess;
    const int64_t grid = (num_tokens + kWriteWarps - 1) / kWriteWarps;
    const int threads = kWriteWarps * 32;
    const bool all_aligned = aligned16(k) && aligned16(v) && aligned16(k_cache) &&
                             aligned16(v_cache);
    const int src_elt = src_dtype == PKV_F32 ? 4 : 2;
    if (all_aligned && src_dtype == cache_dtype && (kv_dim * src_elt) % 16 == 0) {
        return launch_dependent(kv_write_copy_kernel<POS>, dim3((unsigned)grid), dim3(threads), 0,
                                stream, static_cast<const uint4*>(k),
                                static_cast<const uint4*>(v), slots, t, slots_out, num_tokens,
                                static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                                kv_dim * src_elt / 16, num_slots, err);
    } else if (all_aligned && src_dtype == PKV_F32 && cache_dtype == PKV_BF16 && kv_dim % 8 == 0) {
        return launch_dependent(kv_write_f32_to_bf16_kernel<POS>, dim3((unsigned)grid),
                                dim3(threads), 0, stream, static_cast<const float4*>(k),
                                static_cast<const float4*>(v), slots, t, slots_out, num_tokens,
                                static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache),
                                kv_dim / 8, num_slots, err);
    }
    return launch_dependent(kv_write_scalar_kernel<POS>, dim3((unsigned)grid), dim3(threads), 0,
                            stream, k, v, src_dtype, slots, t, slots_out, num_tokens, k_cache,
                            v_cache, cache_dtype, kv_dim, num_slots, err);
}

cudaError_t launch_kv_write(const void* k, const void* v, int src_dtype, const int32_t* slots,
                            int64_t num_tokens, void* k_cache, void* v_cache, int cache_dtype,
                            int64_t kv_dim, int64_t num_slots, unsigned int* err,
                            cudaStream_t stream) {
    return launch_write_t<false>(k, v, src_dtype, slots, TokenSlots{}, nullptr, num_tokens,
                                 k_cache, v_cache, cache_dtype, kv_dim, num_slots, err, stream);
}

cudaError_t launch_kv_write_positions(const void* k, const void* v, int src_dtype,
                                      const int32_t* block_table, int32_t max_blocks,
                                      int32_t num_seqs, const int32_t* token_seq,
                                      const int32_t* token_pos, int64_t num_tokens,
                                      int32_t block_size, int32_t* slots_out, void* k_cache,
                                      void* v_cache, int cache_dtype, int64_t kv_dim,
                                      int64_t num_slots, unsigned int* err, cudaStream_t stream) {
    const TokenSlots t{block_table, max_blocks, num_seqs, token_seq, token_pos, block_size};
    return launch_write_t<true>(k, v, src_dtype, nullptr, t, slots_out, num_tokens, k_cache,
                                v_cache, cache_dtype, kv_dim, num_slots, err, stream);
}

// ---------------------------------------------------------------------------
// block copies (copy-on-write, "11. Paged attention 与 online softmax" §11.3)
// ---------------------------------------------------------------------------
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;  // 16-byte vectors in flight per thread and pool

// grid (chunks of kCopyThreads * kCopyUnroll vectors, pairs): each CTA copies
// one chunk of block src[pair] to block dst[pair] in both pools
__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(uint4* __restrict__ kc, uint4* __restrict__ vc,
                   const int32_t* __restrict__ src, const int32_t* __restrict__ dst,
                   int64_t vec_per_block, int64_t num_blocks, unsigned int* err) {
    PKV_DEPENDENT_PROLOGUE();
    const int32_t s = __ldg(src + blockIdx.y), d = __ldg(dst + blockIdx.y);
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(err, PKV_FLAG_BAD_BLOCK);
        return;
    }
    const int64_t base = (int64_t)blockIdx.x * kCopyThreads * kCopyUnroll + threadIdx.x;
    const uint4* ks = kc + s * vec_per_block;
    const uint4* vs = vc + s * vec_per_block;
    uint4* kd = kc + d * vec_per_block;
    uint4* vd = vc + d * vec_per_block;
    uint4 a[kCopyUnroll], b[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + u * kCopyThreads;
        if (i < vec_per_block) {
            a[u] = __ldcs(ks + i);
            b[u] = __ldcs(vs + i);
        }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
        const int64_t i = base + u * kCopyThreads;
        if (i < vec_per_block) {
            __stcs(kd + i, a[u]);
            __stcs(vd + i, b[u]);
        }
    }
}

// element-wise fallback for pools whose blocks are not 16-byte multiples
__global__ void copy_blocks_bytes_kernel(unsigned char* __restrict__ kc,
                                         unsigned char* __restrict__ vc,
                                         const int32_t* __restrict__ src,
                                         const int32_t* __restrict__ dst, int64_t block_bytes,
                                         int64_t num_blocks, unsigned int* err) {
    PKV_DEPENDENT_PROLOGUE();
    const int32_t s = src[blockIdx.y], d = dst[blockIdx.y];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
        if (threadIdx.x == 0 && blockIdx.x == 0) flag_error(err, PKV_FLAG_BAD_BLOCK);
        return;
    }
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < block_bytes;
         i += (int64_t)gridDim.x * blockDim.x) {
        kc[d * block_bytes + i] = kc[s * block_bytes + i];
        vc[d * block_bytes + i] = vc[s * block_bytes + i];
    }
}

cudaError_t launch_copy_blocks(void* k_cache, void* v_cache, const int32_t* src,
                               const int32_t* dst, int32_t n_pairs, int64_t block_bytes,
                               int64_t num_blocks, unsigned int* err, cudaStream_t stream) {
    if (n_pairs == 0) return cudaSuccess;
    if (block_bytes % 16 == 0 && aligned16(k_cache) && aligned16(v_cache)) {
        const int64_t vec = block_bytes / 16;
        const int64_t per_cta = (int64_t)kCopyThreads * kCopyUnroll;
        const dim3 grid((unsigned)((vec + per_cta - 1) / per_cta), (unsigned)n_pairs);
        return launch_dependent(copy_blocks_kernel, grid, dim3(kCopyThreads), 0, stream,
                                static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), src,
                                dst, vec, num_blocks, err);
    } else {
        const dim3 grid((unsigned)std::min<int64_t>((block_bytes + 255) / 256, 64),
                        (unsigned)n_pairs);
        return launch_dependent(copy_blocks_bytes_kernel, grid, dim3(256), 0, stream,
                                static_cast<unsigned char*>(k_cache),
                                static_cast<unsigned char*>(v_cache), src, dst, block_bytes,
                                num_blocks, err);
    }
    return cudaGetLastError();
}

}  // namespace pkv
