// prefix.cu -- the shared-prefix pass of grouped decode on the sm_103a tensor
// cores (tcgen05.mma, TMEM, TMA).
//
// What it computes ("11. Paged attention 与 online softmax" §11.3: sequences
// that share blocks; "结合nanovllm的FlashAttention和PagedAttention主要原理概述"
// 题目6: the prefix cache; §11.2: online softmax and the boxed merge rule):
// sequences group_cu[g] .. group_cu[g+1]-1 of a decode batch hold their first
// group_plen[g] keys in the same physical blocks, read through the block-table
// row of the group's first sequence.  For every sequence b of the group and
// query head h, over those keys j (or the chunk of them one work item covers):
//   s_j = scale * q[b,h] . k_j * log2(e)          (scores in log2 units)
//   out = sum_j 2^(s_j) v_j / sum_j 2^(s_j),   lse = log2(sum_j 2^(s_j)),
// the state (m = lse, l = 1, o = out) that the decode's combine merges with the
// sequence's own keys by the boxed rule.  A chunk with no keys leaves lse =
// -inf (the merge skips it).
//
// GB300 design.  One CTA per (group, KV head, key chunk, block of members):
//   - its single 128-row Q tile holds the group's queries of the KV head's G
//     query heads, row = member * G + head, loaded by one TMA box of (64 dims,
//     G heads, 128 / G sequences) per half of the head dims (rows past the
//     batch arrive zero-filled; rows of other groups are computed and not
//     stored), so one MMA serves every member and head of the KV head;
//   - K/V tiles of 128 keys stream through rings of 3 stages, one TMA box per
//     page piece (min(B, 128) rows) addressed through the block table; with
//     several pieces per tile warps 8, 10 and 11 share the copies and read the
//     table one tile ahead; pieces past the chunk's keys use an out-of-range
//     row and arrive zero-filled.  (Filling the swizzled tiles with 16-byte
//     cp.async copies from those warps instead was measured at a quarter of
//     the box copies' rate for 16-key pages.);
//   - two softmax warpgroups take alternate key tiles (A, warps 0-3: the even
//     tiles; B, warps 4-7: the odd ones), each with its own S and O in TMEM and
//     its own online state, so the tensor core runs one tile's QK^T and PV
//     while the other group's softmax runs; warp 9 issues every MMA in the
//     order QK(0), QK(1), then per tile j: PV(j), QK(j + 2);
//   - the epilogue merges the two states row by row with the boxed rule (A
//     writes the first half of the head dims and the lse, B the second half).
// The softmax keeps a lagging reference maximum (rescaled only when a row's
// maximum grows by more than 2^8, so every p <= 256) and speculates that it
// still holds, as the prefill does; the final o / l does not depend on it.
// Every mbarrier wait is time-limited (PKV_FLAG_TIMEOUT); a timed-out CTA
// drains its copies and waits for its MMAs before it frees TMEM.
#include <algorithm>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kPBN = 128;   // keys per K/V tile
constexpr int kPSK = 3;     // K ring depth
constexpr int kPSV = 3;     // V ring depth
constexpr int kPThreads = 384;
constexpr int kPRegsLow = 88;    // producer / MMA warpgroup after setmaxnreg
constexpr int kPRegsHigh = 208;  // softmax warpgroups
static_assert(8 * kPRegsHigh + 4 * kPRegsLow <= 12 * 168, "register split exceeds the launch");
constexpr float kPLog2e = 1.4426950408889634f;
constexpr float kPRescaleLog2 = 8.0f;
constexpr uint32_t kPBarBytes = 256;

template <int HD>
struct PShape {
    static_assert(HD == 64 || HD == 128, "head_dim 64 or 128");
    static constexpr uint32_t kTileBytes = kPBN * HD * 2;  // 128 rows of HD bf16
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_K = OFF_Q + kTileBytes;
    static constexpr uint32_t OFF_V = OFF_K + kPSK * kTileBytes;
    static constexpr uint32_t OFF_BAR = OFF_V + kPSV * kTileBytes;
    static constexpr size_t kSmemBytes = OFF_BAR + kPBarBytes + 1024;  // + alignment slack
    static constexpr uint32_t IDESC_QK = idesc(0, kPBN);
    static constexpr uint32_t IDESC_PV = idesc(1, HD);
};

struct PrefixArgs {
    const int32_t* group_cu;    // [n_groups + 1]
    const int32_t* group_plen;  // [n_groups]
    const int32_t* table;       // [batch, max_blocks]
    uint16_t* x_out;            // [kchunks, batch, hq, HD] bf16
    float* x_lse;               // [kchunks, batch, hq]
    unsigned int* err;
    int64_t num_blocks;
    float scale_log2;
    int32_t max_blocks;
    int32_t batch;
    int32_t hq;
    int32_t group;       // G = hq / hkv
    int32_t block_size;
    int32_t piece;       // rows per K/V box = min(B, 128)
    int32_t oob_row;     // a row beyond the pools (zero-filled by TMA)
    int32_t kchunks;
    int32_t n_groups;
};

template <int HD>
__global__ void __launch_bounds__(kPThreads, 1)
prefix_attn_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, const PrefixArgs a) {
    using Sh = PShape<HD>;
    constexpr uint32_t kTileBytes = Sh::kTileBytes;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Sh::OFF_BAR);
    uint64_t* k_full = bars;              // [kPSK]
    uint64_t* k_empty = k_full + kPSK;    // [kPSK]
    uint64_t* v_full = k_empty + kPSK;    // [kPSV]
    uint64_t* v_empty = v_full + kPSV;    // [kPSV]
    uint64_t* s_full = v_empty + kPSV;    // [2] per softmax group
    uint64_t* p_full = s_full + 2;        // [2]
    uint64_t* o_ready = p_full + 2;       // [2] after the group's last PV
    uint64_t* q_ready = o_ready + 2;
    uint64_t* mma_done = q_ready + 1;     // every MMA of the CTA complete
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

    // The inputs come from before the call: kernels launched after this one
    // (the decode split, which needs none of its results) may start at once.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.group;
    const int per_blk = 128 / G;  // members per CTA
    const int kvh = blockIdx.y;
    const int g = blockIdx.z / a.kchunks, chunk = blockIdx.z % a.kchunks;
    const int32_t gm0 = a.group_cu[g], gm1 = a.group_cu[g + 1];
    const int32_t m0 = gm0 + (int32_t)blockIdx.x * per_blk;
    if (m0 >= gm1 || m0 >= a.batch || m0 < 0) return;  // no member in this block
    const int32_t m1 = min(min(gm1, m0 + per_blk), a.batch);
    // the prefix: whole pieces only (a piece past the keys arrives zero-filled)
    const int32_t cap = a.max_blocks * a.block_size;
    int32_t plen = a.group_plen[g];
    if (plen < 0 || plen > cap || plen % a.block_size) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            flag_error(a.err, PKV_FLAG_BAD_LENGTH);
        plen = plen < 0 ? 0 : (plen > cap ? cap : plen);
    }
    plen -= plen % a.piece;
    const int32_t per = ((plen + a.kchunks - 1) / a.kchunks + kPBN - 1) / kPBN * kPBN;
    const int32_t kbase = chunk * per;
    const int32_t klen = max(0, min(per, plen - kbase));
    const int n_tiles = (klen + kPBN - 1) / kPBN;
    const int64_t xrow0 = (int64_t)chunk * a.batch;  // this chunk's output block

    if (n_tiles == 0) {  // no key in this chunk: the merge skips the state
        for (int t = threadIdx.x; t < (m1 - m0) * G; t += blockDim.x)
            a.x_lse[(xrow0 + m0 + t / G) * a.hq + kvh * G + t % G] = -INFINITY;
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPSK; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kPSV; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_full[x], 4);
            mbar_init(&o_ready[x], 1);
        }
        mbar_init(q_ready, 1);
        mbar_init(mma_done, 1);
        fence_barrier_init();
    }
    if (warp == 9) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp >= 8) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPRegsLow));
        if (warp != 9) {
            // ------------------------------ TMA producer ------------------------------
            // lane l of producer warp w (8, 10, 11) takes page piece 3l + w of
            // every tile (a box copy takes ~100 cycles to issue, and with
            // 16-key pages a tile is 16 boxes of K and 16 of V); warp 8's lane
            // 0 also loads Q and sets each stage's expected bytes (a copy that
            // lands first takes the count below zero until then).  Table
            // entries are read one tile ahead.
            const int pw = warp == 8 ? 0 : warp - 9;  // 0, 1, 2
            const int pieces = kPBN / a.piece;
            const int my_piece = lane * 3 + pw;
            const int32_t* trow = a.table + (int64_t)gm0 * a.max_blocks;
            auto entry = [&](int j) -> int32_t {  // table entry of my piece of tile j
                const int32_t key = j * kPBN + my_piece * a.piece;
                if (my_piece >= pieces || key >= klen) return 0;
                return trow[(kbase + key) / a.block_size];
            };
            auto row_of = [&](int j, int32_t phys) -> int32_t {
                const int32_t key = j * kPBN + my_piece * a.piece;
                if (key >= klen) return a.oob_row;
                if (phys < 0 || phys >= a.num_blocks) {
                    flag_error(a.err, PKV_FLAG_BAD_BLOCK);
                    return a.oob_row;
                }
                return phys * a.block_size + (kbase + key) % a.block_size;
            };
            if (pw == 0 && lane == 0) {
                mbar_arrive_expect_tx(q_ready, kTileBytes);
                tma_load_3d(sm + Sh::OFF_Q, &tmap_q, 0, kvh * G, m0, q_ready);
                if constexpr (HD > 64)
                    tma_load_3d(sm + Sh::OFF_Q + kRegionBytes, &tmap_q, 64, kvh * G, m0, q_ready);
            }
            const bool active = my_piece < pieces;
            int issued = 0, issued_v = 0;
            int32_t e_cur = entry(0);
            for (int j = 0; j < n_tiles; ++j) {
                const int sk = j % kPSK, sv = j % kPSV;
                const int32_t e_next = j + 1 < n_tiles ? entry(j + 1) : 0;
                const int32_t my_row = row_of(j, e_cur);
                e_cur = e_next;
                int ok = 1;
                if (lane == 0) {
                    ok = mbar_wait(&k_empty[sk], ((j / kPSK) & 1) ^ 1, a.err);
                    if (ok && pw == 0) mbar_arrive_expect_tx(&k_full[sk], kTileBytes);
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                if (active) {
                    unsigned char* kd = sm + Sh::OFF_K + sk * kTileBytes + my_piece * a.piece * 128;
                    tma_load_3d(kd, &tmap_k, 0, kvh, my_row, &k_full[sk]);
                    if constexpr (HD > 64)
                        tma_load_3d(kd + kRegionBytes, &tmap_k, 64, kvh, my_row, &k_full[sk]);
                }
                ++issued;
                if (lane == 0) {
                    ok = mbar_wait(&v_empty[sv], ((j / kPSV) & 1) ^ 1, a.err);
                    if (ok && pw == 0) mbar_arrive_expect_tx(&v_full[sv], kTileBytes);
                }
                if (!__shfl_sync(0xffffffffu, ok, 0)) break;
                if (active) {
                    unsigned char* vd = sm + Sh::OFF_V + sv * kTileBytes + my_piece * a.piece * 128;
                    tma_load_3d(vd, &tmap_v, 0, kvh, my_row, &v_full[sv]);
                    if constexpr (HD > 64)
                        tma_load_3d(vd + kRegionBytes, &tmap_v, 64, kvh, my_row, &v_full[sv]);
                }
                ++issued_v;
            }
            // drain: every issued copy has landed before the CTA can exit
            if (pw == 0 && lane == 0) {
                mbar_wait(q_ready, 0, a.err);
                for (int j = max(0, issued - kPSK); j < issued; ++j)
                    mbar_wait(&k_full[j % kPSK], (j / kPSK) & 1, a.err);
                for (int j = max(0, issued_v - kPSV); j < issued_v; ++j)
                    mbar_wait(&v_full[j % kPSV], (j / kPSV) & 1, a.err);
            }
        } else if (lane == 0) {
            // ------------------------------ MMA issuer ------------------------------
            // S_x at TMEM columns 128 x, O_x at 256 + 128 x
            // descriptor low words of k-step 0; k-step k adds (k>>2)*16 KiB + (k&3)*32 B
            // (K-major) or k*2 KiB (V, MN-major), in 16-byte units
            const uint32_t q_lo = desc_lo(smem_u32(sm + Sh::OFF_Q), 16);
            const uint32_t k_lo0 = desc_lo(smem_u32(sm + Sh::OFF_K), 16);
            const uint32_t v_lo0 = desc_lo(smem_u32(sm + Sh::OFF_V), kRegionBytes);
            // S_x = Q K(j)^T; the commits release the K stage and signal S
            auto qk = [&](int j) {
                const int x = j & 1, sk = j % kPSK;
                const uint32_t kb = k_lo0 + sk * (kTileBytes >> 4);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k) {
                    const uint32_t off = ((k >> 2) * kRegionBytes + (k & 3) * 32) >> 4;
                    mma_ss(tmem + x * 128, q_lo + off, kb + off, Sh::IDESC_QK, k > 0);
                }
                mma_commit(&k_empty[sk]);
                mma_commit(&s_full[x]);
            };
            // O_x += P_x V(j) with P_x (bf16) in the first 64 columns of S_x
            auto pv = [&](int j) {
                const int x = j & 1, sv = j % kPSV;
                const uint32_t vb = v_lo0 + sv * (kTileBytes >> 4);
#pragma unroll
                for (int k = 0; k < kPBN / 16; ++k)
                    mma_ts(tmem + 256 + x * 128, tmem + x * 128 + k * 8, vb + k * (2048 >> 4), Sh::IDESC_PV,
                           (j >= 2 || k > 0) ? 1u : 0u);
                mma_commit(&v_empty[sv]);
            };
            bool ok = mbar_wait(q_ready, 0, a.err);
            for (int j = 0; ok && j < min(2, n_tiles); ++j) {
                if (!(ok = mbar_wait(&k_full[j % kPSK], (j / kPSK) & 1, a.err))) break;
                tc_fence_after();
                qk(j);
            }
            // A commit tracks every earlier MMA of this thread: S(j + 2) done
            // implies PV(j) done, and the last tile's PV covers everything.
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int x = j & 1;
                if (!(ok = mbar_wait(&v_full[j % kPSV], (j / kPSV) & 1, a.err))) break;
                if (!(ok = mbar_wait(&p_full[x], (j >> 1) & 1, a.err))) break;
                tc_fence_after();
                pv(j);
                if (j + 2 < n_tiles) {
                    if (!(ok = mbar_wait(&k_full[(j + 2) % kPSK], ((j + 2) / kPSK) & 1, a.err)))
                        break;
                        tc_fence_after();
                    qk(j + 2);
                } else {
                    mma_commit(&o_ready[x]);
                }
            }
            // TMEM is freed below: first let every MMA this thread issued
            // complete (after a timed-out wait some may still be running)
            mma_commit(mma_done);
            mbar_wait(mma_done, 0, a.err);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPRegsHigh));
        // ------------------------------ softmax warps ------------------------------
        const int x = warp >> 2;          // 0: even tiles (A), 1: odd tiles (B)
        const int t = threadIdx.x & 127;  // Q row == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tm_s = tmem + x * 128 + lane_base;
        const float sl = a.scale_log2;
        float m_ref = -INFINITY;  // lagging reference max (raw score units)
        float l = 0.f;
        bool ok = true;
        int i = 0;
        for (int j = x; j < n_tiles; j += 2, ++i) {
            if (!warp_wait(&s_full[x], i & 1, a.err)) { ok = false; break; }
            tc_fence_after();
            uint32_t sr[kPBN];
#pragma unroll
            for (int c = 0; c < kPBN / 32; ++c) tmem_ld32(tm_s + c * 32, sr + c * 32);
            tmem_wait_ld();
            const int32_t lim = klen - j * kPBN;  // keys at or past lim are masked
            const bool ragged = lim < kPBN;
            auto mask = [&](uint32_t* v, int c0, int n) {
#pragma unroll
                for (int c = 0; c < n; ++c)
                    if (c0 + c >= lim) v[c] = __float_as_uint(-INFINITY);
            };
            if (ragged) mask(sr, 0, kPBN);
            // p = 2^(s*scale*log2e - m_ref*scale*log2e) in place (bf16 pairs
            // into sr[0..63]); returns the row sum of this tile
            auto exp_pass = [&]() -> float {
                const float ms = (m_ref == -INFINITY) ? 0.f : m_ref * sl;
                const float2 sl2 = make_float2(sl, sl), nms2 = make_float2(-ms, -ms);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int pr = 0; pr < kPBN / 2; ++pr) {
                    const float2 x2 = ffma2(make_float2(__uint_as_float(sr[2 * pr]),
                                                        __uint_as_float(sr[2 * pr + 1])),
                                            sl2, nms2);
                    const float2 p2 = make_float2(ex2(x2.x), ex2(x2.y));
                    acc[pr & 3] = fadd2(acc[pr & 3], p2);
                    sr[pr] = pack_bf16x2(p2.x, p2.y);
                }
                const float2 acct = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
                return acct.x + acct.y;
            };
            bool resc = false;
            float alpha = 1.f;
            auto update_ref = [&](float mx) {
                const float m_new = fmaxf(m_ref, mx);
                resc = (m_new - m_ref) * sl > kPRescaleLog2;
                if (resc) {
                    alpha = (m_ref == -INFINITY) ? 0.f : ex2((m_ref - m_new) * sl);
                    m_ref = m_new;
                }
            };
            float psum;
            if (__any_sync(0xffffffffu, m_ref == -INFINITY)) {
                float mxv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    mxv[u] = fmaxf(__uint_as_float(sr[u]), __uint_as_float(sr[8 + u]));
#pragma unroll
                for (int c = 16; c < kPBN; c += 16)
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        mxv[u] = fmax3(mxv[u], __uint_as_float(sr[c + u]),
                                       __uint_as_float(sr[c + 8 + u]));
                update_ref(fmax3(fmax3(mxv[0], mxv[1], mxv[2]), fmax3(mxv[3], mxv[4], mxv[5]),
                                 fmaxf(mxv[6], mxv[7])));
                psum = exp_pass();
            } else {
                // speculate that the reference still holds: every p <= 2^8
                // unless the tile's sum exceeds 2^8 (or overflowed)
                psum = exp_pass();
                if (__any_sync(0xffffffffu, !(psum <= 256.f))) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int c = 0; c < kPBN / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tm_s + c * 32, v);
                        tmem_wait_ld();
                        if (ragged) mask(v, c * 32, 32);
#pragma unroll
                        for (int e = 0; e < 32; e += 2)
                            mx = fmax3(mx, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
                    }
                    update_ref(mx);
                    if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
                        for (int c = 0; c < kPBN / 32; ++c) tmem_ld32(tm_s + c * 32, sr + c * 32);
                        tmem_wait_ld();
                        if (ragged) mask(sr, 0, kPBN);
                        psum = exp_pass();
                    }
                }
            }
            l = l * alpha + psum;
            tmem_st32(tm_s, sr);
            tmem_st32(tm_s + 32, sr + 32);
            if (i > 0 && __any_sync(0xffffffffu, resc)) {
                // S_x(j) complete implies PV_x(j - 2) is: O_x is stable; scale
                // it before PV_x(j) accumulates
                const uint32_t tm_o = tmem + 256 + x * 128 + lane_base;
#pragma unroll
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tm_o + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(tm_o + c * 32, o);
                }
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x]);
        }
        // Epilogue.  The last tile's PV completes after every other MMA
        // (QK^T of the last tile included), so after it the Q tile is dead:
        // it holds the per-row (m, l) the two groups exchange.
        if (ok) ok = warp_wait(&o_ready[(n_tiles - 1) & 1], 0, a.err);
        float2* xch = reinterpret_cast<float2*>(sm + Sh::OFF_Q);
        xch[x * 128 + t] = make_float2(l > 0.f ? m_ref * sl : -INFINITY, l);
        asm volatile("bar.sync 1, 256;" ::: "memory");
        const float2 sa = xch[t], sb = xch[128 + t];
        const float M = fmaxf(sa.x, sb.x);
        const float fa = sa.x == -INFINITY ? 0.f : ex2(sa.x - M);
        const float fb = sb.x == -INFINITY ? 0.f : ex2(sb.x - M);
        const float lt = sa.y * fa + sb.y * fb;
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        const int32_t member = m0 + t / G;
        const int h = kvh * G + t % G;
        const bool store = ok && member < m1;
        const int64_t orow = (xrow0 + member) * a.hq + h;
        if (store && x == 0) a.x_lse[orow] = lt > 0.f ? M + __log2f(lt) : -INFINITY;
        if (ok) {
            tc_fence_after();
            // group x writes head dims [x * HD / 2, (x + 1) * HD / 2)
            const uint32_t ta = tmem + 256 + lane_base, tb = tmem + 384 + lane_base;
            uint16_t* dst = a.x_out + orow * HD + x * (HD / 2);
#pragma unroll
            for (int c = 0; c < HD / 64; ++c) {
                const int col = x * (HD / 2) + c * 32;
                uint32_t oa[32], ob[32];
                tmem_ld32(ta + col, oa);
                tmem_ld32(tb + col, ob);
                tmem_wait_ld();
                if (store) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 w;
                        // a group with no key (B on a one-tile chunk) left its O
                        // unwritten: its factor is 0 and its columns are not read
                        auto mix = [&](int k) {
                            const float va = fa > 0.f ? __uint_as_float(oa[k]) * fa : 0.f;
                            const float vb = fb > 0.f ? __uint_as_float(ob[k]) * fb : 0.f;
                            return (va + vb) * inv;
                        };
                        w.x = pack_bf16x2(mix(e), mix(e + 1));
                        w.y = pack_bf16x2(mix(e + 2), mix(e + 3));
                        w.z = pack_bf16x2(mix(e + 4), mix(e + 5));
                        w.w = pack_bf16x2(mix(e + 6), mix(e + 7));
                        *reinterpret_cast<uint4*>(dst + c * 32 + e) = w;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512)
                     : "memory");
    }
}

}  // namespace

cudaError_t launch_prefix(const DeviceInfo& dev, const PrefixLaunch& p, cudaStream_t stream) {
    if (p.hd != 128 && p.hd != 64) return cudaErrorNotSupported;
    if (p.hkv <= 0 || p.hq % p.hkv) return cudaErrorNotSupported;
    const int G = p.hq / p.hkv;
    if (G > 128 || 128 % G) return cudaErrorNotSupported;
    const int B = p.block_size;
    const bool b_ok = (B >= 128) ? (B % 128 == 0) : (B >= 8 && 128 % B == 0);
    if (!b_ok || p.n_groups > 65535 || p.hkv > 65535) return cudaErrorNotSupported;
    const size_t smem = p.hd == 128 ? PShape<128>::kSmemBytes : PShape<64>::kSmemBytes;
    if (dev.max_smem_optin < smem) return cudaErrorNotSupported;
    const int64_t rows = p.num_blocks * B;
    if (rows + 128 > 0x7fffffffLL) return cudaErrorNotSupported;
    const int per_blk = 128 / G;
    const int mtiles = (p.max_group_size + per_blk - 1) / per_blk;
    if (mtiles <= 0 || mtiles > 65535 || (int64_t)p.n_groups * p.kchunks > 65535)
        return cudaErrorNotSupported;
    CUtensorMap mq, mk, mv;
    const int piece = B >= 128 ? 128 : B;
    if (!make_map_3d(&mq, p.q, p.hq, p.batch, G, per_blk, p.hd) ||
        !make_rows_map(&mk, p.k_cache, p.hkv, rows, piece, p.hd) ||
        !make_rows_map(&mv, p.v_cache, p.hkv, rows, piece, p.hd))
        return cudaErrorInvalidValue;
    PrefixArgs a;
    a.group_cu = p.group_cu;
    a.group_plen = p.group_plen;
    a.table = p.table;
    a.x_out = static_cast<uint16_t*>(p.x_out);
    a.x_lse = p.x_lse;
    a.err = p.err;
    a.num_blocks = p.num_blocks;
    a.scale_log2 = p.scale * kPLog2e;
    a.max_blocks = p.max_blocks;
    a.batch = p.batch;
    a.hq = p.hq;
    a.group = G;
    a.block_size = B;
    a.piece = piece;
    a.oob_row = (int32_t)rows;
    a.kchunks = p.kchunks;
    a.n_groups = p.n_groups;
    auto kern = p.hd == 128 ? prefix_attn_kernel<128> : prefix_attn_kernel<64>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid(mtiles, p.hkv, p.n_groups * p.kchunks);
    if (p.pdl) return launch_dependent(kern, grid, dim3(kPThreads), smem, stream, mq, mk, mv, a);
    kern<<<grid, kPThreads, smem, stream>>>(mq, mk, mv, a);
    return cudaGetLastError();
}

}  // namespace pkv
