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
// GB300 design, one CTA per request and two Q tiles A and B that read the
// same K/V stream: one 128-query tile of a pair of query heads of one KV head
// (even GQA group), or two consecutive 128-query tiles of one head (odd group,
// e.g. MHA); later (heavier) tiles first:
//   warp 8   TMA producer: first the two Q tiles (one box per 64 dims,
//            ending at the tile's last query row so that a ragged tile never
//            reads past its request), then K and V tiles of 128 keys x 128
//            dims (bf16) into separate rings (3 K stages, 2 V stages),
//            128-byte swizzle; a K/V tile is assembled from one box per page
//            piece (min(B,128) rows) addressed through the block table; boxes
//            past the request's keys use an out-of-range row and arrive
//            zero-filled.  With several pieces per tile (B < 128) warps 8, 10
//            and 11 share the copies and read the table one tile ahead.
//   warp 9   owns TMEM (512 columns: S_A, S_B, O_A, O_B, 128 each) and issues
//            every tcgen05.mma: S_X = Q_X K^T (both operands K-major in shared
//            memory), O_X += P_X V with P_X read from TMEM (the bf16 P tile
//            overwrites the first 64 columns of S_X) and V MN-major.  The
//            issue order PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1) keeps the
//            tensor core on one tile while the other tile's softmax runs.
//   warps 0-3 / 4-7  softmax of tile A / B: thread t owns query row t = TMEM
//            lane t.  Per K/V tile it reads its S row, masks only on diagonal
//            or ragged tiles, and computes p = 2^(s*scale*log2e - m_ref) with
//            one FMA and one MUFU op per element.  m_ref is a lagging reference
//            maximum: it (and O, l) is rescaled only when the row maximum grows
//            by more than 2^8, so p <= 256 and the final o/l is unchanged.
//            Once a reference exists, the exponentials run before any max is
//            taken: a tile whose row sum stays <= 2^8 cannot hold a p > 2^8,
//            and only otherwise is the row max read again from TMEM (S is
//            still there) to decide whether to move the reference and redo.
//   The epilogue divides O by l and stages the bf16 rows in the (now dead)
//   Q tile; a full tile leaves by two TMA boxes, a ragged one with coalesced
//   16-byte writes of its valid rows.
// Also served by the same kernel: packed K/V (no block table; flash-attn's
// varlen call without a prefix cache): request r's keys are rows cu_k[r] ..
// of [rows, Hkv, d] arrays, one 128-row box per K/V tile.  (The shared-prefix
// pass of grouped decode, a non-causal attention of many short query sets,
// has a kernel of its own: prefix.cu.)
// The prefill starts as a programmatic dependent of the kernel before it and
// waits for it; after that it lets its own dependents start (it writes
// nothing they read).
// Every mbarrier wait is time-limited; a timeout sets PKV_FLAG_TIMEOUT and the
// CTA drains its copies, waits for its issued MMAs and frees TMEM before
// returning.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "launch.h"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int BM = 128;  // query rows per Q tile
constexpr int BN = 128;  // keys per K/V tile (head_dim HD is a template parameter: 64 or 128)
constexpr int SK = 3;    // K ring depth
constexpr int SV = 2;    // V ring depth
constexpr int kThreads = 384;  // 8 softmax warps, TMA warp, MMA warp, 2 spare
// Register split (setmaxnreg): launched at 168 per thread; the producer
// warpgroup (warps 8-11) drops to 88 and the two softmax warpgroups rise to
// 208: 8*208 + 4*88 = 12*168 per thread-lane, and per SM quarter (3 warps)
// 208+208+88 <= 512 registers per lane.
constexpr int kRegsLow = 88;
constexpr int kRegsHigh = 208;
static_assert(8 * kRegsHigh + 4 * kRegsLow <= 12 * 168, "register split exceeds the launch");
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.0f;  // rescale when the row max grows by > 2^8


constexpr uint32_t BAR_BYTES = 256;

constexpr uint32_t IDESC_QK = idesc(0, BN);  // S = Q K^T: N = 128 keys

// Per head_dim: a Q, K or V tile is 128 rows of HD bf16 in HD / 64 swizzled
// 128-byte regions; the shared memory map (offsets from a 1024-byte aligned
// base) and the PV descriptor (N = HD).
template <int HD>
struct Shape {
    static_assert(HD == 64 || HD == 128, "head_dim 64 or 128");
    static constexpr uint32_t kTileBytes = BN * HD * 2;  // 16 or 32 KiB
    static constexpr uint32_t OFF_Q = 0;                 // Q_A, Q_B
    static constexpr uint32_t OFF_K = OFF_Q + 2 * kTileBytes;
    static constexpr uint32_t OFF_V = OFF_K + SK * kTileBytes;
    static constexpr uint32_t OFF_BAR = OFF_V + SV * kTileBytes;
    static constexpr size_t kSmemBytes = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t IDESC_PV = idesc(1, HD);
};

struct PrefillArgs {
    uint16_t* out;
    const int32_t* cu_q;
    const int32_t* cu_k;
    const int32_t* table;
    unsigned int* err;
    int64_t num_blocks;
    float scale_log2;
    int32_t max_blocks;
    int32_t hq;
    int32_t group;       // hq / hkv
    int32_t pair_heads;  // 1: a CTA takes query heads (2p, 2p+1); 0: head p alone
    int32_t block_size;
    int32_t piece;    // rows per TMA box = min(B, 128)
    int32_t oob_row;  // a row index beyond the pools (zero-filled by TMA)
    int32_t tiles_q;
    int32_t causal;
    int32_t pair_tiles;  // 1: a CTA takes query tiles qt and qt - 1 of one head
};

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_o,
                  const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, const PrefillArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    using Sh = Shape<HD>;
    constexpr uint32_t kTileBytes = Sh::kTileBytes;
    constexpr uint32_t OFF_Q = Sh::OFF_Q, OFF_K = Sh::OFF_K, OFF_V = Sh::OFF_V;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Sh::OFF_BAR);
    uint64_t* k_full = bars;             // [SK]
    uint64_t* k_empty = k_full + SK;     // [SK]
    uint64_t* v_full = k_empty + SK;     // [SV]
    uint64_t* v_empty = v_full + SV;     // [SV]
    uint64_t* s_full = v_empty + SV;     // [2] per Q tile
    uint64_t* p_full = s_full + 2;       // [2]
    uint64_t* o_ready = p_full + 2;      // [2] last PV of the tile done
    uint64_t* q_ready = o_ready + 2;
    uint64_t* mma_done = q_ready + 1;    // every MMA of the CTA complete
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);

    // Launched as a programmatic dependent of the kernel before it (typically
    // the write of the new rows), the prefill waits for that kernel before
    // reading anything.  Only then may a kernel launched after this one
    // start; one that does not wait (the shared-prefix pass of the mixed
    // step) thus still runs after the write.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = (int)blockIdx.z;
    const int h_a = a.pair_heads ? 2 * (int)blockIdx.y : (int)blockIdx.y;
    const int32_t cq0 = a.cu_q[r], cq1 = a.cu_q[r + 1];
    const int32_t ck0 = a.cu_k[r], ck1 = a.cu_k[r + 1];
    int32_t q_len = cq1 - cq0, k_len = ck1 - ck0;
    const int64_t trow = r;
    // keys a request may have: its block-table row, or (packed K/V) the rows
    // from its first key to the end of the arrays
    const int32_t cap = a.table ? a.max_blocks * a.block_size : max(0, a.oob_row - ck0);
    if (q_len < 0 || k_len < 0 || k_len > cap || q_len > a.tiles_q * BM ||
        (!a.table && ck0 < 0)) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0)
            flag_error(a.err, PKV_FLAG_BAD_LENGTH);
        if (q_len < 0) q_len = 0;
        k_len = k_len < 0 ? 0 : (k_len > cap ? cap : k_len);
    }
    // The CTA's two Q tiles, A (x = 0) and B (x = 1), share every K/V tile:
    //   - pair_heads: one 128-row query tile for query heads h_a and h_a + 1
    //     (the same KV head);
    //   - pair_tiles (one query head per KV head): query tiles qt and qt - 1
    //     of head h_a, A the later one (it sees the most keys; a last key
    //     tile beyond B's rows is fully masked for B); B is absent at qt = 0;
    //   - otherwise A alone.
    // Later (heavier) tiles come first in the grid.
    int qt, qt_b;
    if (a.pair_tiles) {
        qt = (q_len + BM - 1) / BM - 1 - 2 * (int)blockIdx.x;
        qt_b = qt - 1;
    } else {
        qt = a.tiles_q - 1 - (int)blockIdx.x;
        qt_b = qt;
    }
    if (qt < 0 || qt * BM >= q_len) return;
    const bool has_b = a.pair_tiles ? qt_b >= 0 : (a.pair_heads && h_a + 1 < a.hq);
    // Per Q tile: first query row, rows, head and output row.  The Q box
    // always ends at the tile's last query row, so a ragged tile (rows < 128;
    // only a request's last tile) starts `shift` rows early: smem row / TMEM
    // lane t holds query q0 + t - shift, and lanes below `shift` are not
    // stored.
    int32_t tq0[2], trows[2], tshift[2], tbox[2], thead[2];
    int64_t tout[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        const int q = x == 0 ? qt : max(qt_b, 0);
        tq0[x] = q * BM;
        trows[x] = min(BM, q_len - tq0[x]);
        tshift[x] = BM - trows[x];
        tbox[x] = cq0 + tq0[x] + trows[x] - BM;  // negative rows arrive zero-filled
        thead[x] = a.pair_tiles ? h_a : h_a + x;
        tout[x] = (int64_t)cq0 + tq0[x];
    }
    const int32_t diag = k_len - q_len;  // query i sees key j <= i + diag
    int32_t last_key = k_len - 1;
    if (a.causal) last_key = min(last_key, tq0[0] + trows[0] - 1 + diag);
    const int n_tiles = last_key < 0 ? 0 : last_key / BN + 1;

    if (n_tiles == 0) {  // no query row of these tiles sees a key: output 0
        const int nh = has_b ? 2 : 1;
        for (int x = 0; x < nh; ++x) {
            for (int i = threadIdx.x; i < pick(trows, x) * (HD / 8); i += blockDim.x) {
                const int rr = i / (HD / 8), c = i % (HD / 8);
                const int64_t row = pick(tout, x) + rr;
                *reinterpret_cast<uint4*>(a.out + (row * a.hq + pick(thead, x)) * HD + c * 8) =
                    make_uint4(0, 0, 0, 0);
            }
        }
        return;
    }
    const int kvh = h_a / a.group;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SK; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < SV; ++s) {
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
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (warp >= 8) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
      if (warp == 8 || (warp >= 10 && a.piece < BN)) {
        // ------------------------------ TMA producer ------------------------------
        if (a.piece < BN) {
            // Several page pieces per tile: 2 box copies per piece, and a copy
            // takes ~100+ cycles to issue, so warps 8, 10 and 11 share them:
            // lane l of producer warp w takes piece 3l + w.  The lane finds
            // the piece's pool row (its block-table entry read one tile
            // ahead, so that the lookups overlap the previous tile's copies)
            // and issues its two box copies once its warp's lane 0 has seen
            // the ring slot free.  Warp 8 alone sets each slot's expected
            // bytes (a copy may complete first: the count goes below zero
            // until then, and the phase cannot complete without that arrive).
            const int pw = warp == 8 ? 0 : warp - 9;  // 0, 1, 2
            const int piece_of_lane = lane * 3 + pw;
            const int pieces = BN / a.piece;
            const uint32_t all = 0xffffffffu;
            int issued = 0, issued_v = 0;
            const int32_t* trow_ptr = a.table ? a.table + trow * a.max_blocks : nullptr;
            const int32_t lane_key = piece_of_lane < pieces ? piece_of_lane * a.piece
                                                            : INT32_MAX - BN * n_tiles;
            // the table entry behind this lane's piece of tile j (0 if none is read)
            auto entry = [&](int j) -> int32_t {
                const int32_t key = j * BN + lane_key;
                if (key >= k_len || !trow_ptr) return 0;
                return trow_ptr[key / a.block_size];
            };
            auto row_of = [&](int j, int32_t phys) -> int32_t {
                const int32_t key = j * BN + lane_key;
                if (key >= k_len) return a.oob_row;  // zero-filled by TMA (and idle lanes)
                if (!trow_ptr) return ck0 + key;  // packed K/V
                if (phys < 0 || phys >= a.num_blocks) {
                    flag_error(a.err, PKV_FLAG_BAD_BLOCK);
                    return a.oob_row;
                }
                return phys * a.block_size + key % a.block_size;
            };
            if (pw == 0 && lane == 0) {
                const int nq = has_b ? 2 : 1;
                mbar_arrive_expect_tx(q_ready, nq * kTileBytes);
                for (int x = 0; x < nq; ++x) {
                    unsigned char* qd = sm + OFF_Q + x * kTileBytes;
                    const int hh = pick(thead, x), row = pick(tbox, x);
                    tma_load_3d(qd, &tmap_q, 0, hh, row, q_ready);
                    if constexpr (HD > 64)
                        tma_load_3d(qd + kRegionBytes, &tmap_q, 64, hh, row, q_ready);
                }
            }
            int32_t e_cur = entry(0);
            for (int j = 0; j < n_tiles; ++j) {
                const int sk = j % SK, sv = j % SV;
                const int32_t e_next = j + 1 < n_tiles ? entry(j + 1) : 0;
                const int32_t my_row = row_of(j, e_cur);
                e_cur = e_next;
                int ok = 1;
                if (lane == 0) {
                    ok = mbar_wait(&k_empty[sk], ((j / SK) & 1) ^ 1, a.err);
                    if (ok && pw == 0) mbar_arrive_expect_tx(&k_full[sk], kTileBytes);
                }
                if (!__shfl_sync(all, ok, 0)) break;
                if (piece_of_lane < pieces) {
                    unsigned char* kd =
                        sm + OFF_K + sk * kTileBytes + piece_of_lane * a.piece * 128;
                    tma_load_3d(kd, &tmap_k, 0, kvh, my_row, &k_full[sk]);
                    if constexpr (HD > 64)
                        tma_load_3d(kd + kRegionBytes, &tmap_k, 64, kvh, my_row, &k_full[sk]);
                }
                ++issued;
                if (lane == 0) {
                    ok = mbar_wait(&v_empty[sv], ((j / SV) & 1) ^ 1, a.err);
                    if (ok && pw == 0) mbar_arrive_expect_tx(&v_full[sv], kTileBytes);
                }
                if (!__shfl_sync(all, ok, 0)) break;
                if (piece_of_lane < pieces) {
                    unsigned char* vd =
                        sm + OFF_V + sv * kTileBytes + piece_of_lane * a.piece * 128;
                    tma_load_3d(vd, &tmap_v, 0, kvh, my_row, &v_full[sv]);
                    if constexpr (HD > 64)
                        tma_load_3d(vd + kRegionBytes, &tmap_v, 64, kvh, my_row, &v_full[sv]);
                }
                ++issued_v;
            }
            // drain: every issued tile (all three warps' copies) has landed
            // before the CTA can exit
            if (pw == 0 && lane == 0) {
                mbar_wait(q_ready, 0, a.err);
                for (int j = max(0, issued - SK); j < issued; ++j)
                    mbar_wait(&k_full[j % SK], (j / SK) & 1, a.err);
                for (int j = max(0, issued_v - SV); j < issued_v; ++j)
                    mbar_wait(&v_full[j % SV], (j / SV) & 1, a.err);
            }
        } else if (lane == 0) {
            // one page piece per tile: lane 0 alone reads the table and issues
            const int pieces = 1;
            int issued = 0, issued_v = 0;
            auto page_row = [&](int32_t key) -> int32_t {
                if (key >= k_len) return a.oob_row;  // zero-filled by TMA
                if (!a.table) return ck0 + key;       // packed K/V
                const int32_t phys = a.table[trow * a.max_blocks + key / a.block_size];
                if (phys < 0 || phys >= a.num_blocks) {
                    flag_error(a.err, PKV_FLAG_BAD_BLOCK);
                    return a.oob_row;
                }
                return phys * a.block_size + key % a.block_size;
            };
            const int nq = has_b ? 2 : 1;
            mbar_arrive_expect_tx(q_ready, nq * kTileBytes);
            for (int x = 0; x < nq; ++x) {
                unsigned char* qd = sm + OFF_Q + x * kTileBytes;
                const int hh = pick(thead, x), row = pick(tbox, x);
                tma_load_3d(qd, &tmap_q, 0, hh, row, q_ready);
                if constexpr (HD > 64)
                    tma_load_3d(qd + kRegionBytes, &tmap_q, 64, hh, row, q_ready);
            }
            for (int j = 0; j < n_tiles; ++j) {
                const int sk = j % SK, sv = j % SV;
                if (!mbar_wait(&k_empty[sk], ((j / SK) & 1) ^ 1, a.err)) break;
                mbar_arrive_expect_tx(&k_full[sk], kTileBytes);
                for (int p = 0; p < pieces; ++p) {
                    const int32_t row = page_row(j * BN + p * a.piece);
                    unsigned char* kd = sm + OFF_K + sk * kTileBytes + p * a.piece * 128;
                    tma_load_3d(kd, &tmap_k, 0, kvh, row, &k_full[sk]);
                    if constexpr (HD > 64)
                        tma_load_3d(kd + kRegionBytes, &tmap_k, 64, kvh, row, &k_full[sk]);
                }
                ++issued;
                if (!mbar_wait(&v_empty[sv], ((j / SV) & 1) ^ 1, a.err)) break;
                mbar_arrive_expect_tx(&v_full[sv], kTileBytes);
                for (int p = 0; p < pieces; ++p) {
                    const int32_t row = page_row(j * BN + p * a.piece);
                    unsigned char* vd = sm + OFF_V + sv * kTileBytes + p * a.piece * 128;
                    tma_load_3d(vd, &tmap_v, 0, kvh, row, &v_full[sv]);
                    if constexpr (HD > 64)
                        tma_load_3d(vd + kRegionBytes, &tmap_v, 64, kvh, row, &v_full[sv]);
                }
                ++issued_v;
            }
            // drain: every issued tile has landed before the CTA can exit
            mbar_wait(q_ready, 0, a.err);
            for (int j = max(0, issued - SK); j < issued; ++j)
                mbar_wait(&k_full[j % SK], (j / SK) & 1, a.err);
            for (int j = max(0, issued_v - SV); j < issued_v; ++j)
                mbar_wait(&v_full[j % SV], (j / SV) & 1, a.err);
        }
    } else if (warp == 9) {
        // ------------------------------ MMA issuer ------------------------------
        if (lane == 0) {
            const uint32_t tm_s[2] = {tmem, tmem + 128};
            const uint32_t tm_o[2] = {tmem + 256, tmem + 384};
            const int nx = has_b ? 2 : 1;
            // descriptor low words of k-step 0; k-step k adds (k>>2)*16 KiB + (k&3)*32 B
            // (K-major) or k*2 KiB (V, MN-major), in 16-byte units
            const uint32_t q_lo0 = desc_lo(smem_u32(sm + OFF_Q), 16);
            const uint32_t k_lo0 = desc_lo(smem_u32(sm + OFF_K), 16);
            const uint32_t v_lo0 = desc_lo(smem_u32(sm + OFF_V), kRegionBytes);
            auto qk = [&](int x, int sk) {
                const uint32_t qa = q_lo0 + x * (kTileBytes >> 4);
                const uint32_t kb = k_lo0 + sk * (kTileBytes >> 4);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k) {
                    const uint32_t off = ((k >> 2) * kRegionBytes + (k & 3) * 32) >> 4;
                    mma_ss(tm_s[x], qa + off, kb + off, IDESC_QK, k > 0);
                }
                mma_commit(&s_full[x]);
            };
            // A commit tracks every earlier MMA of this thread, so S(j) being
            // complete implies PV(j-1) is: O needs its own signal only after the
            // last PV (for the epilogue).
            auto pv = [&](int x, int sv, bool first, bool last) {
                const uint32_t vb = v_lo0 + sv * (kTileBytes >> 4);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k)
                    mma_ts(tm_o[x], tm_s[x] + k * 8, vb + k * (2048 >> 4), Sh::IDESC_PV,
                           (!first || k > 0) ? 1u : 0u);
                if (last) mma_commit(&o_ready[x]);
            };
            bool ok = mbar_wait(q_ready, 0, a.err) && mbar_wait(&k_full[0], 0, a.err);
            if (ok) {
                tc_fence_after();
                for (int x = 0; x < nx; ++x) qk(x, 0);
                mma_commit(&k_empty[0]);
            }
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int sv = j % SV, sk1 = (j + 1) % SK;
                const bool more = j + 1 < n_tiles;
                if (!(ok = mbar_wait(&v_full[sv], (j / SV) & 1, a.err))) break;
                for (int x = 0; x < nx; ++x) {
                    if (!(ok = mbar_wait(&p_full[x], j & 1, a.err))) break;
                    tc_fence_after();
                    pv(x, sv, j == 0, !more);
                    if (more) {
                        // K(j+1) is needed only now, not before PV(j)
                        if (x == 0 && !(ok = mbar_wait(&k_full[sk1], ((j + 1) / SK) & 1, a.err)))
                            break;
                        tc_fence_after();
                        qk(x, sk1);
                    }
                }
                if (!ok) break;
                mma_commit(&v_empty[sv]);
                if (more) mma_commit(&k_empty[sk1]);
            }
            // TMEM is freed below: first let every MMA this thread issued
            // complete (after a timed-out wait some may still be running)
            mma_commit(mma_done);
            mbar_wait(mma_done, 0, a.err);
        }
    }
    } else {
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
      if (warp < 4 || has_b) {
        // ------------------------------ softmax warps ------------------------------
        const int x = warp >> 2;        // Q tile: 0 = A, 1 = B
        const int t = threadIdx.x & 127;  // query row in the tile == TMEM lane
        const int h = pick(thead, x);
        const int shift = pick(tshift, x);
        const int64_t out_row0 = pick(tout, x);
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tm_s = tmem + x * 128 + lane_base;
        const uint32_t tm_o = tmem + 256 + x * 128 + lane_base;
        const int32_t row_i = pick(tq0, x) + t - shift;  // query index within the request
        int32_t lim = k_len - 1;
        if (a.causal) lim = min(lim, row_i + diag);
        const float sl = a.scale_log2;
        float m_ref = -INFINITY;  // lagging reference max (raw score units)
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            if (!warp_wait(&s_full[x], j & 1, a.err)) { ok = false; break; }
            tc_fence_after();
            uint32_t sr[BN];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) tmem_ld32(tm_s + c * 32, sr + c * 32);
            tmem_wait_ld();
            const int32_t key0 = j * BN;
            const bool ragged = __any_sync(0xffffffffu, key0 + BN - 1 > lim);
            auto mask = [&](uint32_t* v, int c0, int n) {
#pragma unroll
                for (int c = 0; c < n; ++c)
                    if (key0 + c0 + c > lim) v[c] = __float_as_uint(-INFINITY);
            };
            if (ragged) mask(sr, 0, BN);
            // p = 2^(s*scale*log2e - m_ref*scale*log2e) in place (bf16 pairs
            // into sr[0..63]); returns the row sum of this tile
            auto exp_pass = [&]() -> float {
                const float ms = (m_ref == -INFINITY) ? 0.f : m_ref * sl;
                const float2 sl2 = make_float2(sl, sl), nms2 = make_float2(-ms, -ms);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int pr = 0; pr < BN / 2; ++pr) {
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
            // move the reference to max(m_ref, mx) only when that grows it by
            // more than 2^kRescaleLog2 (false when both are -inf)
            bool resc = false;
            float alpha = 1.f;
            auto update_ref = [&](float mx) {
                const float m_new = fmaxf(m_ref, mx);
                resc = (m_new - m_ref) * sl > kRescaleLog2;
                if (resc) {
                    alpha = (m_ref == -INFINITY) ? 0.f : ex2((m_ref - m_new) * sl);
                    m_ref = m_new;
                }
            };
            float psum;
            if (__any_sync(0xffffffffu, m_ref == -INFINITY)) {
                // no reference yet: the row max first (8 independent chains)
                float mxv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    mxv[u] = fmaxf(__uint_as_float(sr[u]), __uint_as_float(sr[8 + u]));
#pragma unroll
                for (int c = 16; c < BN; c += 16)
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
                    // S is still in TMEM: its row max decides
                    float mx = -INFINITY;
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c) {
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
                        for (int c = 0; c < BN / 32; ++c) tmem_ld32(tm_s + c * 32, sr + c * 32);
                        tmem_wait_ld();
                        if (ragged) mask(sr, 0, BN);
                        psum = exp_pass();
                    }
                }
            }
            l = l * alpha + psum;
            uint32_t* pk = sr;
            tmem_st32(tm_s, pk);
            tmem_st32(tm_s + 32, pk + 32);
            if (j > 0 && __any_sync(0xffffffffu, resc)) {
                // S(j) is complete, hence PV(j-1) too: O is stable; scale it
                // before PV(j) accumulates
#pragma unroll
                for (int c = 0; c < HD / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(tm_o + c * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(tm_o + c * 32, o);
                }
            }
            // keys past the request in the last tile: zero their V rows so that
            // p = 0 never meets a non-finite value left in the pool
            if (x == 0 && key0 + BN > k_len) {
                const int sv = j % SV;
                if (!warp_wait(&v_full[sv], (j / SV) & 1, a.err)) { ok = false; break; }
                if (key0 + t >= k_len) {
                    unsigned char* vs = sm + OFF_V + sv * kTileBytes;
#pragma unroll
                    for (int c = 0; c < HD / 8; ++c)
                        *reinterpret_cast<uint4*>(vs + swz(t, c)) = make_uint4(0, 0, 0, 0);
                }
                fence_async_smem();
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[x]);
        }
        if (ok) ok = warp_wait(&o_ready[x], 0, a.err);  // last PV done
        // Epilogue: O / l as bf16 rows staged in this tile's Q buffer (its
        // last reader, QK of the final K tile, completed before o_ready),
        // then stored with coalesced 16-byte writes, 16 threads per row.
        unsigned char* stage = sm + OFF_Q + x * kTileBytes;
        if (ok) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
                uint32_t o[32];
                tmem_ld32(tm_o + c * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; e += 8) {
                    uint4 w;
                    w.x = pack_bf16x2(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv);
                    w.y = pack_bf16x2(__uint_as_float(o[e + 2]) * inv, __uint_as_float(o[e + 3]) * inv);
                    w.z = pack_bf16x2(__uint_as_float(o[e + 4]) * inv, __uint_as_float(o[e + 5]) * inv);
                    w.w = pack_bf16x2(__uint_as_float(o[e + 6]) * inv, __uint_as_float(o[e + 7]) * inv);
                    *reinterpret_cast<uint4*>(stage + swz(t, c * 4 + e / 8)) = w;
                }
            }
        }
        fence_async_smem();  // the staged rows are read by TMA below
        asm volatile("bar.sync %0, 128;" ::"r"(1 + x) : "memory");  // the tile's 4 warps
        if (ok && shift == 0) {
            // a full tile: two TMA boxes (64 dims x 128 rows each)
            if (t == 0) {
                tma_store_3d(&tmap_o, stage, 0, h, (int32_t)out_row0);
                if constexpr (HD > 64)
                    tma_store_3d(&tmap_o, stage + kRegionBytes, 64, h, (int32_t)out_row0);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            }
        } else if (ok) {
#pragma unroll 4
            for (int i = t; i < BM * (HD / 8); i += 128) {
                const int rr = i / (HD / 8), c = i % (HD / 8);
                if (rr >= shift)
                    *reinterpret_cast<uint4*>(a.out + ((out_row0 + rr - shift) * a.hq + h) * HD +
                                              c * 8) =
                        *reinterpret_cast<const uint4*>(stage + swz(rr, c));
            }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
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
    if (d != 128 && d != 64) return cudaErrorNotSupported;
    const size_t smem = d == 128 ? Shape<128>::kSmemBytes : Shape<64>::kSmemBytes;
    // a TMA box of min(B,128) rows must tile 128 keys on 1024-byte boundaries
    // (packed K/V: one 128-row box per tile, any block_size)
    const bool packed = block_table == nullptr;
    const bool b_ok = packed || ((block_size >= 128) ? (block_size % 128 == 0)
                                                     : (block_size >= 8 && 128 % block_size == 0));
    if (!b_ok || batch > 65535 || hq > 65535) return cudaErrorNotSupported;
    if (dev.max_smem_optin < smem) return cudaErrorNotSupported;
    const int64_t rows = num_blocks * block_size;
    if (rows + 128 > 0x7fffffffLL) return cudaErrorNotSupported;
    const int piece = (packed || block_size >= BN) ? BN : block_size;
    // q holds at most batch * max_seqlen_q rows; no box reaches past the
    // last row of its own request, so this bound never clips a valid row
    const int64_t q_rows = std::min<int64_t>((int64_t)batch * max_seqlen_q, 0x7fffffffLL);
    CUtensorMap mq, mo, mk, mv;
    const int64_t o_rows = q_rows;
    if (!make_rows_map(&mq, q, hq, q_rows, BM, d) || !make_rows_map(&mo, out, hq, o_rows, BM, d) ||
        !make_rows_map(&mk, k_cache, hkv, rows, piece, d) ||
        !make_rows_map(&mv, v_cache, hkv, rows, piece, d))
        return cudaErrorInvalidValue;
    PrefillArgs a;
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
    a.pair_heads = (a.group % 2 == 0) ? 1 : 0;
    // one query head per KV head: the CTA's second Q tile is the query tile
    // before the first (same head, same keys) instead of a second head
    a.pair_tiles = a.pair_heads ? 0 : 1;
    a.block_size = block_size;
    a.piece = piece;
    a.oob_row = (int32_t)rows;
    a.tiles_q = (max_seqlen_q + BM - 1) / BM;
    a.causal = causal ? 1 : 0;
    auto kern = d == 128 ? prefill_tc_kernel<128> : prefill_tc_kernel<64>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.pair_tiles ? (a.tiles_q + 1) / 2 : a.tiles_q, a.pair_heads ? (hq + 1) / 2 : hq,
              batch);
    // a programmatic dependent of the previous kernel: the prefill waits for
    // it in the kernel
    return launch_dependent(kern, grid, dim3(kThreads), smem, stream, mq, mo, mk, mv, a);
}

}  // namespace pkv
