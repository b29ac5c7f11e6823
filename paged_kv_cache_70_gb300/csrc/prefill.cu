// prefill.cu -- attention on the sm_103a tensor cores (tcgen05.mma, TMEM
// accumulators, TMA): causal varlen prefill over a paged KV cache, and the
// shared-prefix pass of grouped decode.
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
// Also served by the same code: packed K/V (no block table; flash-attn's
// varlen call without a prefix cache): request r's keys are rows cu_k[r] ..
// of [rows, Hkv, d] arrays, one 128-row box per K/V tile.
// The shared-prefix pass of grouped decode (a non-causal attention of many
// short query sets over one long prefix each, further below) is a second kind
// of work item of the same kernel, attention_tc_kernel: one launch can hold
// prefill items and prefix items (the mixed step), or either alone.
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

// One prefill work item: request bz, query-head pair (or head) by, query
// tile (pair) bx counted from the request's last tile.
template <int HD>
__device__ __forceinline__ void prefill_cta(const CUtensorMap& tmap_q, const CUtensorMap& tmap_o,
                                            const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                            const PrefillArgs& a, int bx, int by, int bz) {
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
    const int r = bz;
    const int h_a = a.pair_heads ? 2 * by : by;
    const int32_t cq0 = a.cu_q[r], cq1 = a.cu_q[r + 1];
    const int32_t ck0 = a.cu_k[r], ck1 = a.cu_k[r + 1];
    int32_t q_len = cq1 - cq0, k_len = ck1 - ck0;
    const int64_t trow = r;
    // keys a request may have: its block-table row, or (packed K/V) the rows
    // from its first key to the end of the arrays
    const int32_t cap = a.table ? a.max_blocks * a.block_size : max(0, a.oob_row - ck0);
    if (q_len < 0 || k_len < 0 || k_len > cap || q_len > a.tiles_q * BM ||
        (!a.table && ck0 < 0)) {
        if (threadIdx.x == 0 && bx == 0 && by == 0)
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
        qt = (q_len + BM - 1) / BM - 1 - 2 * bx;
        qt_b = qt - 1;
    } else {
        qt = a.tiles_q - 1 - bx;
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
// The shared-prefix pass of grouped decode
// ---------------------------------------------------------------------------
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
// With no group arrays every sequence is a group of one whose "prefix" is all
// of its seqlens[b] keys, in chunks of chunk_keys: bf16 decode with 4 or more
// query heads per KV head on the tensor cores.  Its last tile may end inside a
// page; those scores are masked like any ragged tile's, and the V rows past
// the keys are zeroed in shared memory before PV.
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
    const int32_t* group_cu;    // [n_groups + 1]; null: every sequence its own group
    const int32_t* group_plen;  // [n_groups]
    const int32_t* seqlens;     // groups of one: all seqlens[g] keys of sequence g
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
    int32_t chunk_keys;  // > 0: keys per chunk (a multiple of 128), else prefix / kchunks
    int32_t n_groups;
};

// One shared-prefix work item: group and key chunk bz, KV head by, block
// of members bx.
template <int HD>
__device__ __forceinline__ void prefix_cta(const CUtensorMap& tmap_q, const CUtensorMap& tmap_k,
                                           const CUtensorMap& tmap_v, const PrefixArgs& a, int bx,
                                           int by, int bz) {
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
    // (An item with nothing to do returns before any CTA-wide barrier; the
    // items of one launch are separate CTAs.)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.group;
    const int per_blk = 128 / G;  // members per CTA
    const int kvh = by;
    const int g = bz / a.kchunks, chunk = bz % a.kchunks;
    const bool own = a.group_cu == nullptr;  // groups of one sequence
    const int32_t gm0 = own ? g : a.group_cu[g], gm1 = own ? g + 1 : a.group_cu[g + 1];
    const int32_t m0 = gm0 + (int32_t)bx * per_blk;
    if (m0 >= gm1 || m0 >= a.batch || m0 < 0) return;  // no member in this block
    const int32_t m1 = min(min(gm1, m0 + per_blk), a.batch);
    // the prefix: whole pieces only (a piece past the keys arrives zero-filled)
    const int32_t cap = a.max_blocks * a.block_size;
    int32_t plen;
    if (own) {  // all of the sequence's keys; the last piece may be partial
        plen = a.seqlens[g];
        if (plen < 0 || plen > cap) {
            if (threadIdx.x == 0 && bz % a.kchunks == 0 && by == 0)
                flag_error(a.err, PKV_FLAG_BAD_LENGTH);
            plen = plen < 0 ? 0 : (plen > cap ? cap : plen);
        }
    } else {
        plen = a.group_plen[g];
        if (plen < 0 || plen > cap || plen % a.block_size) {
            if (threadIdx.x == 0 && bx == 0 && by == 0)
                flag_error(a.err, PKV_FLAG_BAD_LENGTH);
            plen = plen < 0 ? 0 : (plen > cap ? cap : plen);
        }
        plen -= plen % a.piece;
    }
    const int32_t per = a.chunk_keys > 0
                            ? a.chunk_keys
                            : ((plen + a.kchunks - 1) / a.kchunks + kPBN - 1) / kPBN * kPBN;
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
            if (own && ragged) {
                // a sequence's last tile may end inside a page: its V rows past
                // the keys hold whatever the pool holds there; zero them so that
                // p = 0 never meets a non-finite value
                const int sv = j % kPSV;
                if (!warp_wait(&v_full[sv], (j / kPSV) & 1, a.err)) { ok = false; break; }
                if (t >= lim) {
                    unsigned char* vs = sm + Sh::OFF_V + sv * kTileBytes;
#pragma unroll
                    for (int c = 0; c < HD / 8; ++c)
                        *reinterpret_cast<uint4*>(vs + swz(t, c)) = make_uint4(0, 0, 0, 0);
                }
                fence_async_smem();
            }
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


// ---------------------------------------------------------------------------
// One launch for both kinds of work item: blocks [0, n_prefix) are
// shared-prefix items, the rest prefill items.  Both use 12 warps with the same
// register split, ~225 KB of shared memory and the CTA's 512 TMEM columns, so
// the SMs take either kind as they free up; the prefill items wait for the
// kernel before them (the write of their new rows), the prefix items do not.
// ---------------------------------------------------------------------------
struct TcGrid {
    int n_prefix;  // prefix items: (px, py, pz) blocks, x fastest
    int px, py;
    int fx, fy;    // prefill items: (fx, fy, fz) blocks, x fastest
};

// Prefill items alone (the plain prefill): a kernel of its own, compiled
// without the prefix code path, which costs the prefill ~6% when present.
template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap fq, const __grid_constant__ CUtensorMap fo,
                  const __grid_constant__ CUtensorMap fk, const __grid_constant__ CUtensorMap fv,
                  const PrefillArgs pa) {
    prefill_cta<HD>(fq, fo, fk, fv, pa, blockIdx.x, blockIdx.y, blockIdx.z);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
attention_tc_kernel(const __grid_constant__ CUtensorMap fq, const __grid_constant__ CUtensorMap fo,
                    const __grid_constant__ CUtensorMap fk, const __grid_constant__ CUtensorMap fv,
                    const __grid_constant__ CUtensorMap xq, const __grid_constant__ CUtensorMap xk,
                    const __grid_constant__ CUtensorMap xv, const PrefillArgs pa,
                    const PrefixArgs xa, const TcGrid g) {
    int lin = (int)blockIdx.x;
    if (lin < g.n_prefix) {
        prefix_cta<HD>(xq, xk, xv, xa, lin % g.px, (lin / g.px) % g.py, lin / (g.px * g.py));
    } else {
        lin -= g.n_prefix;
        prefill_cta<HD>(fq, fo, fk, fv, pa, lin % g.fx, (lin / g.fx) % g.fy, lin / (g.fx * g.fy));
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
}  // namespace

size_t prefill_workspace_bytes(int32_t, int32_t, int) { return 0; }

namespace {

// Arguments, tensor maps and grid of a prefill; cudaErrorNotSupported for a
// shape the kernel does not cover.
cudaError_t prepare_prefill(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* cu_q, const int32_t* cu_k, int32_t batch,
                            int32_t max_seqlen_q, const int32_t* block_table, int32_t max_blocks,
                            int causal, float scale, void* out, int hq, int hkv, int d,
                            int block_size, int64_t num_blocks, unsigned int* err, PrefillArgs* a,
                            CUtensorMap* maps, int* gx, int* gy, int* gz) {
    if (d != 128 && d != 64) return cudaErrorNotSupported;
    // a TMA box of min(B,128) rows must tile 128 keys on 1024-byte boundaries
    // (packed K/V: one 128-row box per tile, any block_size)
    const bool packed = block_table == nullptr;
    const bool b_ok = packed || ((block_size >= 128) ? (block_size % 128 == 0)
                                                     : (block_size >= 8 && 128 % block_size == 0));
    if (!b_ok || batch > 65535 || hq > 65535) return cudaErrorNotSupported;
    const int64_t rows = num_blocks * block_size;
    if (rows + 128 > 0x7fffffffLL) return cudaErrorNotSupported;
    const int piece = (packed || block_size >= BN) ? BN : block_size;
    // q holds at most batch * max_seqlen_q rows; no box reaches past the
    // last row of its own request, so this bound never clips a valid row
    const int64_t q_rows = std::min<int64_t>((int64_t)batch * max_seqlen_q, 0x7fffffffLL);
    if (!make_rows_map(&maps[0], q, hq, q_rows, BM, d) ||
        !make_rows_map(&maps[1], out, hq, q_rows, BM, d) ||
        !make_rows_map(&maps[2], k_cache, hkv, rows, piece, d) ||
        !make_rows_map(&maps[3], v_cache, hkv, rows, piece, d))
        return cudaErrorInvalidValue;
    a->out = static_cast<uint16_t*>(out);
    a->cu_q = cu_q;
    a->cu_k = cu_k;
    a->table = block_table;
    a->err = err;
    a->num_blocks = num_blocks;
    a->scale_log2 = scale * kLog2e;
    a->max_blocks = max_blocks;
    a->hq = hq;
    a->group = hq / hkv;
    a->pair_heads = (a->group % 2 == 0) ? 1 : 0;
    // one query head per KV head: the CTA's second Q tile is the query tile
    // before the first (same head, same keys) instead of a second head
    a->pair_tiles = a->pair_heads ? 0 : 1;
    a->block_size = block_size;
    a->piece = piece;
    a->oob_row = (int32_t)rows;
    a->tiles_q = (max_seqlen_q + BM - 1) / BM;
    a->causal = causal ? 1 : 0;
    *gx = a->pair_tiles ? (a->tiles_q + 1) / 2 : a->tiles_q;
    *gy = a->pair_heads ? (hq + 1) / 2 : hq;
    *gz = batch;
    return cudaSuccess;
}

// Arguments, tensor maps and grid of a shared-prefix pass.
cudaError_t prepare_prefix(const PrefixLaunch& p, PrefixArgs* a, CUtensorMap* maps, int* gx,
                           int* gy, int* gz) {
    if (p.hd != 128 && p.hd != 64) return cudaErrorNotSupported;
    if (p.hkv <= 0 || p.hq % p.hkv) return cudaErrorNotSupported;
    const int G = p.hq / p.hkv;
    if (G > 128 || 128 % G) return cudaErrorNotSupported;
    const int B = p.block_size;
    const bool b_ok = (B >= 128) ? (B % 128 == 0) : (B >= 8 && 128 % B == 0);
    if (!b_ok) return cudaErrorNotSupported;
    const int64_t rows = p.num_blocks * B;
    if (rows + 128 > 0x7fffffffLL) return cudaErrorNotSupported;
    const int per_blk = 128 / G;
    const int mtiles = (p.max_group_size + per_blk - 1) / per_blk;
    if (mtiles <= 0) return cudaErrorNotSupported;
    const int piece = B >= 128 ? 128 : B;
    if (!make_map_3d(&maps[0], p.q, p.hq, p.batch, G, per_blk, p.hd) ||
        !make_rows_map(&maps[1], p.k_cache, p.hkv, rows, piece, p.hd) ||
        !make_rows_map(&maps[2], p.v_cache, p.hkv, rows, piece, p.hd))
        return cudaErrorInvalidValue;
    a->group_cu = p.group_cu;
    a->group_plen = p.group_plen;
    a->seqlens = p.seqlens;
    a->chunk_keys = p.chunk_keys;
    a->table = p.table;
    a->x_out = static_cast<uint16_t*>(p.x_out);
    a->x_lse = p.x_lse;
    a->err = p.err;
    a->num_blocks = p.num_blocks;
    a->scale_log2 = p.scale * kPLog2e;
    a->max_blocks = p.max_blocks;
    a->batch = p.batch;
    a->hq = p.hq;
    a->group = G;
    a->block_size = B;
    a->piece = piece;
    a->oob_row = (int32_t)rows;
    a->kchunks = p.kchunks;
    a->n_groups = p.n_groups;
    *gx = mtiles;
    *gy = p.hkv;
    *gz = p.n_groups * p.kchunks;
    return cudaSuccess;
}

// One launch of attention_tc_kernel over the given items (either count may
// be zero; the maps of an absent kind are not read).
cudaError_t launch_tc(const DeviceInfo& dev, int hd, const CUtensorMap* fm, const PrefillArgs& pa,
                      int fx, int fy, int fz, const CUtensorMap* xm, const PrefixArgs& xa,
                      int px, int py, int pz, bool pdl, cudaStream_t stream) {
    const size_t smem = hd == 128 ? std::max(Shape<128>::kSmemBytes, PShape<128>::kSmemBytes)
                                  : std::max(Shape<64>::kSmemBytes, PShape<64>::kSmemBytes);
    if (dev.max_smem_optin < smem) return cudaErrorNotSupported;
    const int64_t nf = (int64_t)fx * fy * fz, np = (int64_t)px * py * pz;
    if (nf + np == 0) return cudaSuccess;
    if (nf + np > 0x7fffffffLL) return cudaErrorNotSupported;
    TcGrid g{(int)np, px > 0 ? px : 1, py > 0 ? py : 1, fx > 0 ? fx : 1, fy > 0 ? fy : 1};
    auto kern = hd == 128 ? attention_tc_kernel<128> : attention_tc_kernel<64>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(nf + np));
    if (pdl)
        return launch_dependent(kern, grid, dim3(kThreads), smem, stream, fm[0], fm[1], fm[2],
                                fm[3], xm[0], xm[1], xm[2], pa, xa, g);
    kern<<<grid, kThreads, smem, stream>>>(fm[0], fm[1], fm[2], fm[3], xm[0], xm[1], xm[2], pa, xa,
                                           g);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const DeviceInfo& dev, const void* q, const void* k_cache,
                           const void* v_cache, const int32_t* cu_q, const int32_t* cu_k,
                           int32_t batch, int32_t max_seqlen_q, int32_t max_seqlen_k,
                           const int32_t* block_table, int32_t max_blocks, int causal,
                           float scale, void* out, void* workspace, int hq, int hkv, int d,
                           int block_size, int64_t num_blocks, unsigned int* err,
                           cudaStream_t stream) {
    (void)max_seqlen_k;
    (void)workspace;
    PrefillArgs pa{};
    CUtensorMap fm[4];
    int fx, fy, fz;
    cudaError_t e = prepare_prefill(q, k_cache, v_cache, cu_q, cu_k, batch, max_seqlen_q,
                                    block_table, max_blocks, causal, scale, out, hq, hkv, d,
                                    block_size, num_blocks, err, &pa, fm, &fx, &fy, &fz);
    if (e != cudaSuccess) return e;
    const size_t smem = d == 128 ? Shape<128>::kSmemBytes : Shape<64>::kSmemBytes;
    if (dev.max_smem_optin < smem) return cudaErrorNotSupported;
    auto kern = d == 128 ? prefill_tc_kernel<128> : prefill_tc_kernel<64>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // a programmatic dependent of the previous kernel: the prefill waits for
    // it in the kernel
    return launch_dependent(kern, dim3(fx, fy, fz), dim3(kThreads), smem, stream, fm[0], fm[1],
                            fm[2], fm[3], pa);
}

cudaError_t launch_prefix(const DeviceInfo& dev, const PrefixLaunch& p, cudaStream_t stream) {
    PrefixArgs xa{};
    CUtensorMap xm[3];
    int px, py, pz;
    cudaError_t e = prepare_prefix(p, &xa, xm, &px, &py, &pz);
    if (e != cudaSuccess) return e;
    CUtensorMap fm[4] = {xm[0], xm[0], xm[1], xm[2]};  // not read: no prefill item
    return launch_tc(dev, p.hd, fm, PrefillArgs{}, 0, 0, 0, xm, xa, px, py, pz, p.pdl, stream);
}

cudaError_t launch_prefill_with_prefix(const DeviceInfo& dev, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* cu_q,
                                       const int32_t* cu_k, int32_t batch, int32_t max_seqlen_q,
                                       const int32_t* block_table, int32_t max_blocks,
                                       float scale, void* out, int hq, int hkv, int d,
                                       int block_size, int64_t num_blocks, unsigned int* err,
                                       const PrefixLaunch& p, cudaStream_t stream) {
    if (p.hd != d) return cudaErrorNotSupported;
    PrefillArgs pa{};
    CUtensorMap fm[4];
    int fx, fy, fz;
    cudaError_t e = prepare_prefill(q, k_cache, v_cache, cu_q, cu_k, batch, max_seqlen_q,
                                    block_table, max_blocks, 1, scale, out, hq, hkv, d, block_size,
                                    num_blocks, err, &pa, fm, &fx, &fy, &fz);
    if (e != cudaSuccess) return e;
    PrefixArgs xa{};
    CUtensorMap xm[3];
    int px, py, pz;
    e = prepare_prefix(p, &xa, xm, &px, &py, &pz);
    if (e != cudaSuccess) return e;
    return launch_tc(dev, d, fm, pa, fx, fy, fz, xm, xa, px, py, pz, true, stream);
}

}  // namespace pkv
