// prefill.cu -- causal varlen prefill over a paged KV cache on the sm_103a
// tensor cores (tcgen05.mma, TMEM accumulators, TMA).
//
// What it computes ("从零开始写Qwen3（六）PagedAttention", "fast-attn 库的使用":
// prefix cache / chunked prefill read the cache through block_table;
// "Sayfalı dikkat" varlen path; FlashAttention tiling and online softmax of
// "结合nanovllm的FlashAttention和PagedAttention主要原理概述" 题目3 and
// "11. Paged attention 与 online softmax" §11.2):
//   request r owns query rows [cu_q[r], cu_q[r+1]) and keys 0 .. k_len-1 read
//   through block_table row r; query i (0-based in the request) sees key j iff
//   j <= i + k_len - q_len (causal, bottom-right) and j < k_len;
//   out = softmax(scale * Q K^T) V over the visible keys, 0 for a row that
//   sees none.
//
// GB300 design, one CTA per (128-query tile, query head, request):
//   warp 4   TMA producer: K and V tiles of 128 keys x 128 dims (bf16) into a
//            2-stage ring, 128-byte swizzle; a tile is assembled from one box
//            per page piece (min(B,128) rows) addressed through the block
//            table; boxes past the request's keys use an out-of-range row and
//            arrive zero-filled.
//   warp 5   owns TMEM (512 columns: S double buffer 2 x 128, O 128) and is the
//            single MMA issuer: S_j = Q K_j^T (M=N=128, K=16 per instruction,
//            both operands K-major), then O += P_j V_j (P K-major, V MN-major),
//            completion signalled with tcgen05.commit on mbarriers.
//   warps 0-3 softmax: thread t owns query row t = TMEM lane t.  Per tile it
//            reads its S row (tcgen05.ld), masks, keeps the running max m and
//            sum l, writes p = 2^(s - m) as bf16 into the swizzled P tile, and
//            rescales its O row in TMEM only when some row of the warp saw a
//            larger max.  The epilogue divides O by l and stores bf16 rows.
// Every mbarrier wait is time-limited; a timeout sets PKV_FLAG_TIMEOUT and the
// CTA drains its copies and frees TMEM before returning.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace pkv {

namespace {

constexpr int BM = 128;  // query rows per CTA
constexpr int BN = 128;  // keys per tile
constexpr int HD = 128;  // head_dim
constexpr int STAGES = 2;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr uint32_t kTileBytes = BN * HD * 2;     // 32 KiB: one K (or V) tile
constexpr uint32_t kRegionBytes = BN * 128;      // 16 KiB: 64 dims (128 B) x 128 rows
constexpr float kLog2e = 1.4426950408889634f;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_P = OFF_Q + kTileBytes;
constexpr uint32_t OFF_K = OFF_P + kTileBytes;
constexpr uint32_t OFF_V = OFF_K + STAGES * kTileBytes;
constexpr uint32_t OFF_BAR = OFF_V + STAGES * kTileBytes;
constexpr uint32_t BAR_BYTES = 256;
constexpr uint32_t GUARD_BYTES = 4096;  // unused tail after the barriers
constexpr size_t kSmemBytes = OFF_BAR + BAR_BYTES + GUARD_BYTES + 1024;

// instruction descriptors: D fp32, A/B bf16, M = N = 128
constexpr uint32_t idesc(uint32_t b_mn_major) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (0u << 15) | (b_mn_major << 16) |
           ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
constexpr uint32_t IDESC_QK = idesc(0);
constexpr uint32_t IDESC_PV = idesc(1);

// shared-memory matrix descriptor, 128-byte swizzle
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

#define PKV_R32(p) \
    "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3]), "=r"(p[4]), "=r"(p[5]), "=r"(p[6]), \
    "=r"(p[7]), "=r"(p[8]), "=r"(p[9]), "=r"(p[10]), "=r"(p[11]), "=r"(p[12]), "=r"(p[13]), \
    "=r"(p[14]), "=r"(p[15]), "=r"(p[16]), "=r"(p[17]), "=r"(p[18]), "=r"(p[19]), "=r"(p[20]), \
    "=r"(p[21]), "=r"(p[22]), "=r"(p[23]), "=r"(p[24]), "=r"(p[25]), "=r"(p[26]), "=r"(p[27]), \
    "=r"(p[28]), "=r"(p[29]), "=r"(p[30]), "=r"(p[31])
#define PKV_W32(p) \
    "r"(p[0]), "r"(p[1]), "r"(p[2]), "r"(p[3]), "r"(p[4]), "r"(p[5]), "r"(p[6]), "r"(p[7]), \
    "r"(p[8]), "r"(p[9]), "r"(p[10]), "r"(p[11]), "r"(p[12]), "r"(p[13]), "r"(p[14]), \
    "r"(p[15]), "r"(p[16]), "r"(p[17]), "r"(p[18]), "r"(p[19]), "r"(p[20]), "r"(p[21]), \
    "r"(p[22]), "r"(p[23]), "r"(p[24]), "r"(p[25]), "r"(p[26]), "r"(p[27]), "r"(p[28]), \
    "r"(p[29]), "r"(p[30]), "r"(p[31])

// 32 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : PKV_R32(r)
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        PKV_W32(r)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// byte offset of 16-byte chunk `c` (0..15) of row `r` in a 128-row x 256-byte
// tile stored as two 128-byte-swizzled regions (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B and the MMA reads as a K-major operand)
__device__ __forceinline__ uint32_t swz(int r, int c) {
    return (uint32_t)((c >> 3) * kRegionBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

struct PrefillArgs {
    const uint16_t* q;
    uint16_t* out;
    const int32_t* cu_q;
    const int32_t* cu_k;
    const int32_t* table;
    unsigned int* err;
    int64_t num_blocks;
    float scale_log2;
    int32_t max_blocks;
    int32_t hq;
    int32_t group;  // hq / hkv
    int32_t block_size;
    int32_t piece;  // rows per TMA box = min(B, 128)
    int32_t oob_row;  // a row index beyond the pools (zero-filled by TMA)
    int32_t tiles_q;
    int32_t causal;
};

__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint64_t* kv_full = bars;             // [STAGES]
    uint64_t* kv_empty = bars + 2;        // [STAGES]
    uint64_t* s_full = bars + 4;          // [2]
    uint64_t* s_free = bars + 6;          // [2]
    uint64_t* p_full = bars + 8;
    uint64_t* o_ready = bars + 9;
    uint64_t* q_ready = bars + 10;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 12);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.z, h = blockIdx.y;
    const int qt = a.tiles_q - 1 - (int)blockIdx.x;  // later (heavier) tiles first
    const int32_t cq0 = a.cu_q[r], cq1 = a.cu_q[r + 1];
    const int32_t ck0 = a.cu_k[r], ck1 = a.cu_k[r + 1];
    int32_t q_len = cq1 - cq0, k_len = ck1 - ck0;
    const int32_t cap = a.max_blocks * a.block_size;
    if (q_len < 0 || k_len < 0 || k_len > cap || q_len > a.tiles_q * BM) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            flag_error(a.err, PKV_FLAG_BAD_LENGTH);
        if (q_len < 0) q_len = 0;
        k_len = k_len < 0 ? 0 : (k_len > cap ? cap : k_len);
    }
    const int32_t q0 = qt * BM;
    if (q0 >= q_len) return;
    const int rows = min(BM, q_len - q0);
    const int32_t diag = k_len - q_len;  // query i sees key j <= i + diag
    int32_t last_key = k_len - 1;
    if (a.causal) last_key = min(last_key, q0 + rows - 1 + diag);
    const int n_tiles = last_key < 0 ? 0 : last_key / BN + 1;
    const int64_t out_row0 = (int64_t)cq0 + q0;

    if (n_tiles == 0) {  // no query row of this tile sees a key: output 0
        for (int i = threadIdx.x; i < rows * (HD / 8); i += blockDim.x) {
            const int rr = i / (HD / 8), c = i % (HD / 8);
            *reinterpret_cast<uint4*>(a.out + ((out_row0 + rr) * a.hq + h) * HD + c * 8) =
                make_uint4(0, 0, 0, 0);
        }
        return;
    }
    const int kvh = h / a.group;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&s_free[b], 4);
        }
        mbar_init(p_full, 4);
        mbar_init(o_ready, 1);
        mbar_init(q_ready, 4);
        fence_barrier_init();
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tm_s[2] = {tmem, tmem + 128};
    const uint32_t tm_o = tmem + 256;

    if (warp == 4) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            const int pieces = BN / a.piece;
            int issued = 0;
            for (int j = 0; j < n_tiles; ++j) {
                const int s = j % STAGES;
                if (!mbar_wait(&kv_empty[s], ((j / STAGES) & 1) ^ 1, a.err)) break;
                mbar_arrive_expect_tx(&kv_full[s], 2 * kTileBytes);
                unsigned char* kd = sm + OFF_K + s * kTileBytes;
                unsigned char* vd = sm + OFF_V + s * kTileBytes;
                for (int p = 0; p < pieces; ++p) {
                    const int32_t key = j * BN + p * a.piece;
                    int32_t row = a.oob_row;
                    if (key < k_len) {
                        const int32_t phys = a.table[(int64_t)r * a.max_blocks + key / a.block_size];
                        if (phys < 0 || phys >= a.num_blocks)
                            flag_error(a.err, PKV_FLAG_BAD_BLOCK);
                        else
                            row = phys * a.block_size + key % a.block_size;
                    }
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t off = hh * kRegionBytes + p * a.piece * 128;
                        tma_load_3d(kd + off, &tmap_k, hh * 64, kvh, row, &kv_full[s]);
                        tma_load_3d(vd + off, &tmap_v, hh * 64, kvh, row, &kv_full[s]);
                    }
                }
                ++issued;
            }
            // drain: every issued tile has landed before the CTA can exit
            for (int j = max(0, issued - STAGES); j < issued; ++j)
                mbar_wait(&kv_full[j % STAGES], (j / STAGES) & 1, a.err);
        }
    } else if (warp == 5) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            const uint32_t q_base = smem_u32(sm + OFF_Q), p_base = smem_u32(sm + OFF_P);
            bool ok = mbar_wait(q_ready, 0, a.err);
            auto issue_qk = [&](int j) -> bool {
                const int s = j % STAGES;
                if (!mbar_wait(&kv_full[s], (j / STAGES) & 1, a.err)) return false;
                if (j >= 2 && !mbar_wait(&s_free[j & 1], ((j - 2) >> 1) & 1, a.err)) return false;
                tc_fence_after();
                const uint32_t k_base = smem_u32(sm + OFF_K + s * kTileBytes);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k) {
                    const uint32_t off = (k >> 2) * kRegionBytes + (k & 3) * 32;
                    mma_bf16(tm_s[j & 1], sdesc(q_base + off, 16, 1024),
                             sdesc(k_base + off, 16, 1024), IDESC_QK, k > 0);
                }
                mma_commit(&s_full[j & 1]);
                return true;
            };
            if (ok) ok = issue_qk(0);
            for (int j = 0; ok && j < n_tiles; ++j) {
                if (j + 1 < n_tiles && !issue_qk(j + 1)) break;
                if (!mbar_wait(p_full, j & 1, a.err)) break;
                tc_fence_after();
                const int s = j % STAGES;
                const uint32_t v_base = smem_u32(sm + OFF_V + s * kTileBytes);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) {
                    const uint32_t poff = (k >> 2) * kRegionBytes + (k & 3) * 32;
                    mma_bf16(tm_o, sdesc(p_base + poff, 16, 1024),
                             sdesc(v_base + k * 2048, kRegionBytes, 1024), IDESC_PV,
                             (j > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(o_ready);
                mma_commit(&kv_empty[s]);
            }
        }
    } else {
        // ------------------------------ softmax warps ------------------------------
        const int t = threadIdx.x;  // query row within the tile == TMEM lane
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        {   // Q row t -> swizzled shared tile (zeros past the request)
            unsigned char* qs = sm + OFF_Q;
            const bool valid = t < rows;
            // rows past the request read row 0 of the tile (always in bounds), then zero it
            const int64_t qrow = out_row0 + (valid ? t : 0);
            const uint4* src = reinterpret_cast<const uint4*>(a.q + (qrow * a.hq + h) * HD);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                uint4 v = __ldg(src + c);
                if (!valid) v = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4*>(qs + swz(t, c)) = v;
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(q_ready);
        }
        const int32_t row_i = q0 + t;  // query index within the request
        int32_t lim = k_len - 1;
        if (a.causal) lim = min(lim, row_i + diag);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            if (!__all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, a.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld32(tm_s[j & 1] + lane_base + c * 32, sr + c * 32);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_free[j & 1]);

            const int32_t key0 = j * BN;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; ++c) {
                const float x = (key0 + c <= lim) ? __uint_as_float(sr[c]) * a.scale_log2 : -INFINITY;
                sr[c] = __float_as_uint(x);
                mx = fmaxf(mx, x);
            }
            const float m_new = fmaxf(m, mx);
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
            const float alpha = ex2(m - m_use);
            float sum = 0.f;
            uint32_t* pk = sr;  // packed bf16 pairs overwrite the scores already consumed
#pragma unroll
            for (int c = 0; c < BN; c += 2) {
                const float p0 = ex2(__uint_as_float(sr[c]) - m_use);
                const float p1 = ex2(__uint_as_float(sr[c + 1]) - m_use);
                sum += p0 + p1;
                pk[c >> 1] = pack_bf16x2(p0, p1);
            }
            l = l * alpha + sum;
            m = m_new;

            if (j > 0) {
                // PV_{j-1} done: P tile free and O stable
                if (!__all_sync(0xffffffffu, mbar_wait(o_ready, (j - 1) & 1, a.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
                    for (int c = 0; c < HD / 32; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tm_o + lane_base + c * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tmem_st32(tm_o + lane_base + c * 32, o);
                    }
                    tmem_wait_st();
                }
            }
            // keys past the request in the last tile: zero their V rows so that
            // p = 0 never meets a non-finite value left in the pool
            if (key0 + BN > k_len) {
                const int s = j % STAGES;
                if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[s], (j / STAGES) & 1, a.err))) {
                    ok = false;
                    break;
                }
                if (key0 + t >= k_len) {
                    unsigned char* vs = sm + OFF_V + s * kTileBytes;
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        *reinterpret_cast<uint4*>(vs + swz(t, c)) = make_uint4(0, 0, 0, 0);
                }
            }
            unsigned char* ps = sm + OFF_P;
#pragma unroll
            for (int c = 0; c < 16; ++c)
                *reinterpret_cast<uint4*>(ps + swz(t, c)) =
                    make_uint4(pk[c * 4], pk[c * 4 + 1], pk[c * 4 + 2], pk[c * 4 + 3]);
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_ready, (n_tiles - 1) & 1, a.err));
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint16_t* dst = a.out + ((out_row0 + t) * a.hq + h) * HD;
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tm_o + lane_base + c * 32, o);
                tmem_wait_ld();
                if (t < rows) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                        *reinterpret_cast<uint4*>(dst + c * 32 + e) = w;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// pool [num_blocks*B rows, Hkv, 128] bf16 viewed as 3-D (dim, head, row); box
// (64 dims, 1 head, piece rows), 128-byte swizzle
bool make_pool_map(CUtensorMap* map, const void* base, int hkv, int64_t rows, int piece) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)hkv, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)HD * 2, (cuuint64_t)hkv * HD * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)piece};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_workspace_bytes(int32_t, int32_t, int) { return 0; }

cudaError_t launch_prefill(const DeviceInfo& dev, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* cu_q, const int32_t* cu_k,
                           int32_t batch, int32_t max_seqlen_q, int32_t max_seqlen_k,
                           const int32_t* block_table, int32_t max_blocks, int causal,
                           float scale, void* out, void* workspace, int hq, int hkv, int d,
                           int block_size, int64_t num_blocks, unsigned int* err,
                           cudaStream_t stream) {
    (void)max_seqlen_k;
    (void)workspace;
    if (d != HD) return cudaErrorNotSupported;
    // a TMA box of min(B,128) rows must tile 128 keys on 1024-byte boundaries
    const bool b_ok = (block_size >= 128) ? (block_size % 128 == 0)
                                          : (block_size >= 8 && 128 % block_size == 0);
    if (!b_ok || batch > 65535 || hq > 65535) return cudaErrorNotSupported;
    if (dev.max_smem_optin < kSmemBytes) return cudaErrorNotSupported;
    const int64_t rows = num_blocks * block_size;
    if (rows + 128 > 0x7fffffffLL) return cudaErrorNotSupported;
    const int piece = block_size < BN ? block_size : BN;
    CUtensorMap mk, mv;
    if (!make_pool_map(&mk, k_cache, hkv, rows, piece) ||
        !make_pool_map(&mv, v_cache, hkv, rows, piece))
        return cudaErrorInvalidValue;
    PrefillArgs a;
    a.q = static_cast<const uint16_t*>(q);
    a.out = static_cast<uint16_t*>(out);
    a.cu_q = cu_q;
    a.cu_k = cu_k;
    a.table = block_table;
    a.err = err;
    a.num_blocks = num_blocks;
    a.scale_log2 = scale * kLog2e;
    a.max_blocks = max_blocks;
    a.hq = hq;
    a.group = hq / hkv;
    a.block_size = block_size;
    a.piece = piece;
    a.oob_row = (int32_t)rows;
    a.tiles_q = (max_seqlen_q + BM - 1) / BM;
    a.causal = causal ? 1 : 0;
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    dim3 grid(a.tiles_q, hq, batch);
    prefill_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(mk, mv, a);
    return cudaGetLastError();
}

}  // namespace pkv
