// decode.cu -- paged decode (one query token per sequence) for sm_103a.
//
// What it computes ("Sayfalı dikkat", decode path; "11. Paged attention 与
// online softmax" §11.1-§11.2): for sequence b and query head h,
//   out[b,h] = sum_j softmax_j(scale * q[b,h] . k_j) v_j,  j < cache_seqlens[b],
// where key j is read from the paged pool through block_table row b
// (phys = table[j / B], slot = j % B) and blocks are merged with the online
// rule  m_new = max(m, m_b),  o = o e^(m - m_new) + o_b e^(m_b - m_new),
// l likewise, out = o / l.
//
// GB300 design (HBM-bound: ~1 FMA per K/V byte for GQA group 2):
//  * Work split.  The keys of every sequence are cut into tiles of R keys
//    (R divides B, so a tile never crosses a page) and the concatenated tile
//    list of all sequences is cut into contiguous shares, one per CTA (one
//    CTA per SM), equal once each sequence start is counted as one tile.  A
//    CTA therefore covers a piece of one long sequence or several short ones;
//    each piece yields a partial (m, l, o) state that a second kernel merges
//    with the same rule.  Load balance is within about one tile whatever the
//    length mix.
//  * Data movement.  A producer warp streams each tile of K and V (all KV heads
//    of the CTA; a tile is contiguous in the pool when the CTA owns every KV
//    head) into a ring of shared-memory stages with cp.async.bulk, tracked by
//    mbarriers; ~128 KiB stay in flight per SM.  The block-table entry is read
//    and range-checked once per tile, by the producer.
//  * Math.  Eight consumer warps; each warp owns one KV head and its G query
//    heads (the K/V tile is shared across the GQA group).  For G = 4 the CTA
//    has 12 warps and setmaxnreg moves registers from the producer's
//    warpgroup to the consumers, which hold 4 heads' q and o.  Groups of 8, 16
//    and 32 run the group-4 kernel with G / 4 warps per KV head, each holding
//    4 of its query heads.  (bf16 decode with G >= 4 normally attends on the
//    tensor cores instead, through the shared-prefix pass with every sequence
//    a group of one; this split then serves fp32, the block sizes that pass
//    does not take, and the suffixes of shared-prefix steps.)  Within a warp,
//    groups of D/16 lanes take key rows, every lane holding 16 of the D
//    dimensions of q (pre-scaled by scale*log2 e) and of o as fp32 pairs; a
//    group handles two key rows at a time with packed fp32x2 FMAs (four
//    independent chains), dot products are reduced with xor shuffles, and each
//    pair of keys updates the state as one block (running max of the state and
//    both scores; o rescaled only when the max grows).
//    Exponentials are base 2 on log2-scaled scores, which is the same merge.
//  * The combine kernel (one warp per sequence and head) is launched as a
//    programmatic dependent of the split kernel, so its launch overlaps the
//    split kernel's tail.  Besides the split partials it can merge
//      - shared-prefix partials: groups of consecutive sequences that hold a
//        common prefix in the same blocks get that prefix's attention from
//        the tensor-core kernel (once per group, in key chunks; normalised
//        output and log2-sum-exp), and the split kernel then starts each
//        sequence's tile list after its group's prefix;
//      - the appended token ("Sayfalı dikkat" decode path, new k/v written
//        into the cache by the kvcache call): its score is taken from k_new,
//        it joins the merge as a one-key state, and the combine writes the
//        new K/V row through the block table (the split kernel, which read
//        only the keys before it, has completed).
//  * As a programmatic dependent of an unrelated kernel (the mixed step), the
//    split kernel holds its grid open with one otherwise idle lane waiting on
//    griddepcontrol.wait, so that its completion implies that kernel's.
//  * Safety.  Block ids and lengths are range-checked before any address is
//    formed; every mbarrier wait is time-limited (PKV_FLAG_TIMEOUT).  After
//    a timeout the consumers stop waiting but still meet at every named
//    barrier, and the producer waits (time-limited) for its last copies to
//    land before the CTA exits.
#include <float.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

constexpr int kConsumerWarps = 8;
constexpr int kDecodeThreads = (kConsumerWarps + 1) * 32;
// With 9 warps an SM sub-partition holds 3 of a CTA's warps, which caps a
// thread at 168 registers: enough for GQA groups of 1 and 2.  A group of 4
// keeps 4 heads' q and o per lane, so that kernel runs 12 warps (8 consumers,
// the producer, 3 that only complete its warpgroup) and moves registers from
// the producer warpgroup to the consumers with setmaxnreg: 8 x 208 + 4 x 88 =
// 2016 <= 12 x 168 per thread-lane, and 208 + 208 + 88 <= 512 per
// sub-partition lane.
template <int G>
constexpr int decode_threads() { return G >= 4 ? 12 * 32 : kDecodeThreads; }
constexpr int kDecodeMaxWarps = 12;
constexpr int kConsumerRegs4 = 208;
constexpr int kProducerRegs4 = 88;
static_assert(8 * kConsumerRegs4 + 4 * kProducerRegs4 <= 12 * 168,
              "register split exceeds the launch");
constexpr int kMaxStages = 8;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeArgs {
    const void* q;
    const unsigned char* k_cache;
    const unsigned char* v_cache;
    const int32_t* table;
    const int32_t* seqlens;
    float* part_o;        // [ctas + batch][hq][D]
    float* part_ml;       // [ctas + batch][hq][2]
    int32_t* tstart_out;  // [batch + 1]
    // shared-prefix mode (else null): sequences group_cu[g] .. group_cu[g+1]-1
    // share their first group_plen[g] keys, which this kernel then skips
    const int32_t* group_cu;
    const int32_t* group_plen;
    unsigned int* err;
    int64_t num_blocks;
    float qscale;  // scale * log2(e)
    int32_t max_blocks;
    int32_t batch;
    int32_t hq;
    int32_t hkv;
    int32_t hc;  // KV heads per CTA
    int32_t gfull;   // query heads per KV head (Hq / Hkv)
    int32_t gsplit;  // warps (query-head subsets of G each) per KV head and row
    int32_t block_size;
    int32_t rows;  // R
    int32_t stages;
    int32_t n_groups;
    int32_t wait_prior;  // this grid completes only after the previous kernel has
    int32_t wait_inputs;  // wait for the previous kernel before reading any input
    // one-launch step (else null): each CTA adds 1 here once its partial
    // states are stored (the combine CTAs of the same grid wait for them)
    unsigned int* done;
};

// The split's shares.  Tile t of sequence b sits at position
//   u(t) = t + kSeqCost * (b + 1)
// of a cost line (starting a sequence costs a CTA about kSeqCost tiles: its
// queries, its partial state, the merge), and the line is cut into equal
// pieces, one per CTA.  u is increasing, so a piece is a contiguous run of
// tiles; the combine finds a sequence's pieces from the same formula.
constexpr int32_t kSeqCost = 1;
__device__ __forceinline__ int32_t share_cost(int32_t total, int32_t batch, int ctas) {
    const int32_t u = total + kSeqCost * batch;
    return u > 0 ? (u + ctas - 1) / ctas : 1;
}
// the first tile t with u(t) >= x (total if none)
__device__ __forceinline__ int32_t first_tile_at(const int32_t* tstart, int batch, int64_t x) {
    int lo = 0, hi = batch;  // first b whose last tile's position is >= x
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)tstart[mid + 1] - 1 + (int64_t)kSeqCost * (mid + 1) >= x) hi = mid;
        else lo = mid + 1;
    }
    if (lo >= batch) return tstart[batch];
    const int64_t t = x - (int64_t)kSeqCost * (lo + 1);
    return (int32_t)max((int64_t)tstart[lo], t);
}

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ constexpr size_t merge_bytes(int G, int D) {
    return align_up((size_t)kConsumerWarps * G * (D + 2) * sizeof(float), 128);
}
// per-sequence tables in shared memory: tile starts [batch + 1], first keys
// [batch], clamped lengths [batch]
__host__ __device__ constexpr size_t seq_table_bytes(int batch) {
    return align_up((size_t)(batch + 1) * 4, 128) + 2 * align_up((size_t)batch * 4, 128);
}
// [ring barriers 128 B][stage tags 128 B][merge barriers 128 B][sequence
// tables][merge scratch][stages]
constexpr size_t kDecodeHeaderBytes = 384;
__host__ __device__ constexpr size_t decode_fixed_smem(int G, int D, int batch) {
    return kDecodeHeaderBytes + seq_table_bytes(batch) + merge_bytes(G, D);
}

// two bf16 packed in a word -> (element 2i, element 2i+1) as fp32 (exact)
__device__ __forceinline__ float2 bf2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// 8 consecutive elements as 4 fp32 pairs
template <bool BF16>
__device__ __forceinline__ void load8_smem(const unsigned char* p, float2* x) {
    if constexpr (BF16) {
        const uint4 w = *reinterpret_cast<const uint4*>(p);
        x[0] = bf2(w.x); x[1] = bf2(w.y); x[2] = bf2(w.z); x[3] = bf2(w.w);
    } else {
        const float4 a = *reinterpret_cast<const float4*>(p);
        const float4 b = *reinterpret_cast<const float4*>(p + 16);
        x[0] = make_float2(a.x, a.y); x[1] = make_float2(a.z, a.w);
        x[2] = make_float2(b.x, b.y); x[3] = make_float2(b.z, b.w);
    }
}

template <bool BF16>
__device__ __forceinline__ void load8_global(const void* base, int64_t elem, float2* x) {
    if constexpr (BF16) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + elem));
        x[0] = bf2(w.x); x[1] = bf2(w.y); x[2] = bf2(w.z); x[3] = bf2(w.w);
    } else {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
        const float4 a = __ldg(p), b = __ldg(p + 1);
        x[0] = make_float2(a.x, a.y); x[1] = make_float2(a.z, a.w);
        x[2] = make_float2(b.x, b.y); x[3] = make_float2(b.z, b.w);
    }
}

__device__ __forceinline__ int32_t clamp_len(int32_t L, int32_t cap) {
    return L < 0 ? 0 : (L > cap ? cap : L);
}

// Per-sequence plan of the CTA, in shared memory (all threads take part):
//   slen[b]   cache_seqlens[b] clamped to [0, the table's capacity];
//   sfirst[b] first key of b's own tiles: 0, or in shared-prefix mode its
//             group's prefix length (a multiple of the block size, at most
//             L; anything else is flagged and rounded down to a whole tile);
//   tstart[b] exclusive prefix sum of the tile counts, tstart[batch] = total.
// All global loads of a step are issued together (the group bounds first,
// then every sequence's length and prefix length), so the plan costs about
// two memory round trips.
__device__ void plan_tiles(const DecodeArgs& a, int32_t* tstart, int32_t* sfirst,
                           int32_t* slen) {
    __shared__ int32_t warp_tot[kDecodeMaxWarps];
    const int tid = threadIdx.x, nthr = blockDim.x;
    const int32_t cap = a.max_blocks * a.block_size;
    if (a.group_cu) {
        // group bounds into tstart (scratch until the scan below)
        for (int g = tid; g <= a.n_groups; g += nthr) tstart[g] = __ldg(a.group_cu + g);
        __syncthreads();
    }
    for (int b = tid; b < a.batch; b += nthr) {
        const int32_t L = clamp_len(a.seqlens[b], cap);
        int32_t st = 0;
        if (a.group_cu) {
            int lo = 0, hi = a.n_groups;  // the last g with group_cu[g] <= b
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (tstart[mid] <= b) lo = mid; else hi = mid;
            }
            st = __ldg(a.group_plen + lo);
            if (st < 0 || st > L || st % a.block_size) {
                flag_error(a.err, PKV_FLAG_BAD_LENGTH);
                st = st < 0 ? 0 : (st > L ? L : st);
                st -= st % a.rows;
            }
        }
        slen[b] = L;
        sfirst[b] = st;
    }
    __syncthreads();
    // block-wide exclusive scan of the tile counts
    const int per = (a.batch + nthr - 1) / nthr;
    const int lo = tid * per, hi = min(lo + per, a.batch);
    int32_t sum = 0;
    for (int b = lo; b < hi; ++b) sum += (slen[b] - sfirst[b] + a.rows - 1) / a.rows;
    const int lane = tid & 31, warp = tid >> 5;
    int32_t inc = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += y;
    }
    if (lane == 31) warp_tot[warp] = inc;
    __syncthreads();
    int32_t base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    int32_t run = base + inc - sum;  // exclusive prefix of this thread's first sequence
    for (int b = lo; b < hi; ++b) {
        tstart[b] = run;
        run += (slen[b] - sfirst[b] + a.rows - 1) / a.rows;
    }
    if (tid == nthr - 1) tstart[a.batch] = base + inc;
}

// the sequence b with tstart[b] <= t < tstart[b+1]
__device__ __forceinline__ int seq_of_tile(const int32_t* tstart, int batch, int32_t t) {
    int lo = 0, hi = batch;  // first index in [0, batch] with tstart[idx] > t
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (tstart[mid] <= t) lo = mid + 1; else hi = mid;
    }
    return lo - 1;
}

// One CTA of the split: share bx of gx along the tile list, KV-head group by.
// Run by decode_split_kernel, and by the one-launch step kernel with
// a.done set (there the CTA has 12 warps; warps past the producer leave).
template <int D, bool BF16, int G>
__device__ __forceinline__ void split_cta(const DecodeArgs& a, const int bx, const int by,
                                          const int gx) {
    constexpr int ELT = BF16 ? 2 : 4;
    constexpr int TG = D / 16;    // lanes per key row
    constexpr int GPW = 32 / TG;  // key rows processed side by side by a warp
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    // per stage: valid block id, tile index, piece (CTA or chunk) index, and
    // whether the tile ends its piece
    int32_t* stage_ok = reinterpret_cast<int32_t*>(smem + 128);
    int32_t* stage_tile = stage_ok + kMaxStages;
    int32_t* stage_piece = stage_tile + kMaxStages;
    int32_t* stage_last = stage_piece + kMaxStages;
    uint64_t* merge_bar = reinterpret_cast<uint64_t*>(smem + 256);  // [2]
    int32_t* tstart = reinterpret_cast<int32_t*>(smem + kDecodeHeaderBytes);
    int32_t* sfirst = tstart + align_up((size_t)(a.batch + 1) * 4, 128) / 4;
    int32_t* slen = sfirst + align_up((size_t)a.batch * 4, 128) / 4;
    float* mscratch = reinterpret_cast<float*>(smem + kDecodeHeaderBytes + seq_table_bytes(a.batch));
    unsigned char* stage_base = smem + decode_fixed_smem(G, D, a.batch);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = a.stages, R = a.rows, HC = a.hc;
    const size_t row_bytes = (size_t)HC * D * ELT;    // one key row of the CTA's heads
    const size_t half_bytes = (size_t)R * row_bytes;  // K (or V) part of a stage
    const int32_t cap = a.max_blocks * a.block_size;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(&merge_bar[0], kConsumerWarps);
        mbar_init(&merge_bar[1], kConsumerWarps);
        fence_barrier_init();
    }
    // launched as a programmatic dependent: the lengths, table and K/V may come
    // from the kernel before (the new token's write)
    if (a.wait_inputs) asm volatile("griddepcontrol.wait;" ::: "memory");
    // Kernels launched after this one may be scheduled now (the combine waits
    // for this grid's results).  After the wait above, so that one that does
    // not wait would still start only after everything before this grid.
    // Block (0, 0) lets them start only once it has stored the tile starts
    // (below), which the combine reads before its wait.
    const bool first_cta = bx == 0 && by == 0;
    if (!first_cta) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    plan_tiles(a, tstart, sfirst, slen);
    __syncthreads();

    // Holding the grid open (see DecodeArgs::wait_prior): block (0, 0) does
    // not exit before the kernel launched before this one has completed.
    // Its producer waits after issuing its copies; with no work it waits here.
    const bool holder = a.wait_prior && bx == 0 && by == 0;
    const int32_t total = tstart[a.batch];
    if (first_cta) {
        for (int b = threadIdx.x; b <= a.batch; b += blockDim.x) a.tstart_out[b] = tstart[b];
        for (int b = threadIdx.x; b < a.batch; b += blockDim.x) {
            const int32_t L = a.seqlens[b];
            if (L < 0 || L > cap) flag_error(a.err, PKV_FLAG_BAD_LENGTH);
        }
        __threadfence();
        __syncthreads();
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    // this CTA's share [t0, t1) of the tile list
    const int32_t chunk = share_cost(total, a.batch, gx);
    const int32_t t0 = first_tile_at(tstart, a.batch, (int64_t)bx * chunk);
    const int32_t t1 = first_tile_at(tstart, a.batch, (int64_t)(bx + 1) * chunk);
    if (t0 >= t1) {
        if (holder && threadIdx.x == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
        if (a.done && threadIdx.x == 0) {  // nothing to store
            __threadfence();
            atomicAdd(a.done, 1u);
        }
        return;
    }
    const int head0 = by * HC;  // first KV head of this CTA

    if (warp >= kConsumerWarps) {
        if constexpr (G >= 4) {
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs4));
        }
        if (warp > kConsumerWarps) return;  // only complete the warpgroup or the CTA
        // ------------------------------ producer ------------------------------
        // The 32 lanes prepare 32 tiles at a time (sequence, first key, rows,
        // block-table entry: the entries of a batch are read together); lane 0
        // waits for ring slots and issues the copies.
        const uint64_t pol = l2_evict_first_policy();
        const unsigned all = 0xffffffffu;
#ifdef PKV_TEST_SPLIT_PRODUCER_IDLE
        // test-only build: issue nothing, so the consumers' first wait runs out
        if (holder && lane == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
#endif
        int32_t k = 0;  // stages filled so far (lane 0)
        bool stop = false;
        {
            // the CTA's piece: its share [t0, t1) of the tile list
            const int32_t piece = bx, pt0 = t0, pt1 = t1;
            for (int32_t tb = pt0; tb < pt1 && !stop; tb += 32) {
                // lane i: tile tb + i's block-table entry and (first key's slot
                // in the block) * 64 + rows (rows <= 32); the batch's table
                // reads are covered by the stages still queued in the ring
                int32_t my_phys = 0, my_slot_rows = 0;
                if (tb + lane < pt1) {
                    const int32_t t = tb + lane;
                    const int bb = seq_of_tile(tstart, a.batch, t);
                    const int32_t pos0 = sfirst[bb] + (t - tstart[bb]) * R;
                    my_slot_rows = (pos0 % a.block_size) * 64 + min(R, slen[bb] - pos0);
                    my_phys = a.table[(int64_t)bb * a.max_blocks + pos0 / a.block_size];
                }
                const int n = min(32, pt1 - tb);
                for (int i = 0; i < n; ++i) {
                    const int32_t phys = __shfl_sync(all, my_phys, i);
                    const int32_t slot_rows = __shfl_sync(all, my_slot_rows, i);
                    if (lane != 0 || stop) continue;
                    const int32_t rows = slot_rows & 63, off = slot_rows >> 6;
                    const int s = k % S;
                    if (!mbar_wait(&empty[s], ((k / S) & 1) ^ 1, a.err)) {
                        stop = true;
                        continue;
                    }
                    ++k;
                    stage_tile[s] = tb + i;
                    stage_piece[s] = piece;
                    stage_last[s] = (tb + i + 1 == pt1) ? 1 : 0;
                    if (phys < 0 || phys >= a.num_blocks) {
                        flag_error(a.err, PKV_FLAG_BAD_BLOCK);
                        stage_ok[s] = 0;
                        mbar_arrive(&full[s]);
                        continue;
                    }
                    stage_ok[s] = 1;
                    const int64_t row0 = (int64_t)phys * a.block_size + off;
                    unsigned char* kd = stage_base + (size_t)s * 2 * half_bytes;
                    unsigned char* vd = kd + half_bytes;
                    const uint32_t bytes = (uint32_t)(rows * row_bytes);
                    mbar_arrive_expect_tx(&full[s], 2 * bytes);
                    if (HC == a.hkv) {
                        const size_t o = (size_t)row0 * row_bytes;
                        bulk_g2s(kd, a.k_cache + o, bytes, &full[s], pol);
                        bulk_g2s(vd, a.v_cache + o, bytes, &full[s], pol);
                    } else {
                        const size_t pool_row = (size_t)a.hkv * D * ELT;
                        for (int r = 0; r < rows; ++r) {
                            const size_t o = (size_t)(row0 + r) * pool_row + (size_t)head0 * D * ELT;
                            bulk_g2s(kd + r * row_bytes, a.k_cache + o, (uint32_t)row_bytes, &full[s], pol);
                            bulk_g2s(vd + r * row_bytes, a.v_cache + o, (uint32_t)row_bytes, &full[s], pol);
                        }
                    }
                }
                stop = __shfl_sync(all, stop ? 1 : 0, 0) != 0;
            }
        }
        // the end of the CTA's tiles: a stage with tile -1 (no copy)
        if (!stop && lane == 0) {
            const int s = k % S;
            if (mbar_wait(&empty[s], ((k / S) & 1) ^ 1, a.err)) {
                stage_tile[s] = -1;
                stage_ok[s] = 0;
                mbar_arrive(&full[s]);
                ++k;
            }
        }
        if (lane != 0) return;
        // The CTA must not exit while a copy into its shared memory is in
        // flight: wait (time-limited) for the last fill of every stage.  In a
        // normal run the consumers wait for the same phases, so this costs
        // nothing; after a timeout the consumers may have stopped waiting.
        for (int32_t j = k > S ? k - S : 0; j < k; ++j)
            if (!mbar_wait(&full[j % S], (j / S) & 1, a.err)) break;
        if (holder) asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }

    // ------------------------------- consumers --------------------------------
    if constexpr (G >= 4) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs4));
    // warp -> (local KV head, subset of G query heads, rank among the warps
    // that share both and split the tile's rows)
    const int GS = a.gsplit;
    const int hc = warp % HC;
    const int gs = (warp / HC) % GS;
    const int wrank = warp / (HC * GS);
    const int WH = kConsumerWarps / (HC * GS);
    const int qh0 = (head0 + hc) * a.gfull + gs * G;  // the warp's first query head
    const int grp = lane / TG, tl = lane % TG;
    const int warp_row0 = wrank * GPW;  // first row of the warp in a tile
    const int row_step = WH * GPW;      // rows between a group's consecutive rows
    // this lane's dimensions: [tl*8, +8) and [TG*8 + tl*8, +8)
    const int dim0 = tl * 8, dim1 = TG * 8 + tl * 8;

    float2 q2[G][8], o2[G][8];
    float m[G], l[G];
    int b = 0;
    int loaded = -1;     // the sequence whose queries are in registers
    bool fresh = false;  // the state holds no key of the current piece yet
    int32_t L = 0, st = 0;

    // The consumers follow the stages' tags (tile, piece, piece end) until the
    // closing stage.  A timed-out wait ends the warp's loop; the other
    // warps then time out at the next merge barrier or ring stage, so every
    // wait of the CTA still ends.
    int merges = 0;       // merge-barrier rounds so far (phase parity)
    int32_t prev_t = -2;  // previous tile (consecutive tiles keep the sequence cursor)
    for (int32_t k = 0;; ++k) {
        const int s = k % S;
        if (!__all_sync(0xffffffffu, mbar_wait(&full[s], (k / S) & 1, a.err))) break;
        const int32_t t = stage_tile[s];
        if (t < 0) break;  // the closing stage
        const int32_t piece = stage_piece[s];
        const bool piece_end = stage_last[s] != 0;
        const bool stage_valid = stage_ok[s] != 0;
        if (t != prev_t + 1) {
            b = seq_of_tile(tstart, a.batch, t);
        } else {
            while (t >= tstart[b + 1]) ++b;
        }
        prev_t = t;
        if (b != loaded) {
            loaded = b;
            fresh = false;
            // the queries first: their loads overlap the length lookups
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int64_t qb = ((int64_t)b * a.hq + qh0 + g) * D;
                load8_global<BF16>(a.q, qb + dim0, &q2[g][0]);
                load8_global<BF16>(a.q, qb + dim1, &q2[g][4]);
            }
            L = slen[b];
            st = sfirst[b];
            const float2 sc2 = make_float2(a.qscale, a.qscale);
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < 8; ++e) q2[g][e] = fmul2(q2[g][e], sc2);
        }
        if (!fresh) {  // a new piece: empty state (the queries stay)
            fresh = true;
#pragma unroll
            for (int g = 0; g < G; ++g) {
#pragma unroll
                for (int e = 0; e < 8; ++e) o2[g][e] = make_float2(0.f, 0.f);
                m[g] = -INFINITY;
                l[g] = 0.f;
            }
        }
        const int32_t rows = min(R, L - st - (t - tstart[b]) * R);
        if (stage_valid) {
            const unsigned char* ks = stage_base + (size_t)s * 2 * half_bytes;
            const unsigned char* vs = ks + half_bytes;
            // warp-uniform loop over pairs of rows (ra, rb = ra + row_step)
            for (int base = warp_row0; base < rows; base += 2 * row_step) {
                const int ra = base + grp, rb = ra + row_step;
                const bool va = ra < rows, vb = rb < rows;
                const int ia = va ? ra : 0, ib = vb ? rb : 0;
                const unsigned char* kra = ks + ((size_t)ia * HC + hc) * D * ELT;
                const unsigned char* krb = ks + ((size_t)ib * HC + hc) * D * ELT;
                float2 ka[8], kb[8];
                load8_smem<BF16>(kra + dim0 * ELT, &ka[0]);
                load8_smem<BF16>(kra + dim1 * ELT, &ka[4]);
                load8_smem<BF16>(krb + dim0 * ELT, &kb[0]);
                load8_smem<BF16>(krb + dim1 * ELT, &kb[4]);
                float sa[G], sb[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float2 acca = make_float2(0.f, 0.f), accb = make_float2(0.f, 0.f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        acca = ffma2(q2[g][e], ka[e], acca);
                        accb = ffma2(q2[g][e], kb[e], accb);
                    }
                    sa[g] = acca.x + acca.y;
                    sb[g] = accb.x + accb.y;
                }
#pragma unroll
                for (int off = 1; off < TG; off <<= 1) {
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        sa[g] += __shfl_xor_sync(0xffffffffu, sa[g], off);
                        sb[g] += __shfl_xor_sync(0xffffffffu, sb[g], off);
                    }
                }
                // both rows in one update (a block of two keys): one max test
                // and one rescale per pair, the two exponentials independent
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    if (!va) sa[g] = -INFINITY;
                    if (!vb) sb[g] = -INFINITY;
                    const float mn = fmax3(m[g], sa[g], sb[g]);
                    if (mn > m[g]) {  // running max grows: rescale the state
                        const float c = ex2(m[g] - mn);
                        l[g] *= c;
                        const float2 c2 = make_float2(c, c);
#pragma unroll
                        for (int e = 0; e < 8; ++e) o2[g][e] = fmul2(o2[g][e], c2);
                        m[g] = mn;
                    }
                    // (a pair of rows past the tile's end on a fresh state: m = -inf)
                    const float mr = (m[g] == -INFINITY) ? 0.f : m[g];
                    const float pa = ex2(sa[g] - mr), pb = ex2(sb[g] - mr);
                    l[g] += pa + pb;
                    sa[g] = pa;
                    sb[g] = pb;
                }
                {  // row a (p = 0 when past the end: row 0's values, finite, times 0)
                    const unsigned char* vr = vs + ((size_t)ia * HC + hc) * D * ELT;
                    float2 vx[8];
                    load8_smem<BF16>(vr + dim0 * ELT, &vx[0]);
                    load8_smem<BF16>(vr + dim1 * ELT, &vx[4]);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float2 p2 = make_float2(sa[g], sa[g]);
#pragma unroll
                        for (int e = 0; e < 8; ++e) o2[g][e] = ffma2(p2, vx[e], o2[g][e]);
                    }
                }
                if (vb) {
                    const unsigned char* vr = vs + ((size_t)ib * HC + hc) * D * ELT;
                    float2 vx[8];
                    load8_smem<BF16>(vr + dim0 * ELT, &vx[0]);
                    load8_smem<BF16>(vr + dim1 * ELT, &vx[4]);
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float2 p2 = make_float2(sb[g], sb[g]);
#pragma unroll
                        for (int e = 0; e < 8; ++e) o2[g][e] = ffma2(p2, vx[e], o2[g][e]);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);

        // end of this piece of sequence b: merge and store the partial state
        const bool seg_end = piece_end || (t + 1 >= tstart[b + 1]);
        if (!seg_end) continue;
        // merge the groups of the warp (lanes with equal tl hold the same dims)
#pragma unroll
        for (int off = TG; off < 32; off <<= 1) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float mo = __shfl_xor_sync(0xffffffffu, m[g], off);
                const float lo = __shfl_xor_sync(0xffffffffu, l[g], off);
                const float M = fmaxf(m[g], mo);
                const float ca = (m[g] == -INFINITY) ? 0.f : ex2(m[g] - M);
                const float cb = (mo == -INFINITY) ? 0.f : ex2(mo - M);
                l[g] = l[g] * ca + lo * cb;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float ox = __shfl_xor_sync(0xffffffffu, o2[g][e].x, off);
                    const float oy = __shfl_xor_sync(0xffffffffu, o2[g][e].y, off);
                    o2[g][e] = make_float2(o2[g][e].x * ca + ox * cb, o2[g][e].y * ca + oy * cb);
                }
                m[g] = M;
            }
        }
        if (WH > 1) {  // several warps share this KV head: merge through shared memory
            float* my = mscratch + (size_t)warp * G * (D + 2);
            if (grp == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        my[g * (D + 2) + dim0 + 2 * e] = o2[g][e].x;
                        my[g * (D + 2) + dim0 + 2 * e + 1] = o2[g][e].y;
                        my[g * (D + 2) + dim1 + 2 * e] = o2[g][4 + e].x;
                        my[g * (D + 2) + dim1 + 2 * e + 1] = o2[g][4 + e].y;
                    }
                    if (tl == 0) {
                        my[g * (D + 2) + D] = m[g];
                        my[g * (D + 2) + D + 1] = l[g];
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&merge_bar[0]);
            if (!__all_sync(0xffffffffu, mbar_wait(&merge_bar[0], merges & 1, a.err))) break;
            if (wrank == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float M = -INFINITY;
                    for (int w = 0; w < WH; ++w)
                        M = fmaxf(M, mscratch[(size_t)((w * GS + gs) * HC + hc) * G * (D + 2) +
                                              g * (D + 2) + D]);
                    float lt = 0.f;
                    float2 ot[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) ot[e] = make_float2(0.f, 0.f);
                    for (int w = 0; w < WH; ++w) {
                        const float* src = mscratch + (size_t)((w * GS + gs) * HC + hc) * G * (D + 2) +
                                           g * (D + 2);
                        const float mw = src[D];
                        const float c = (mw == -INFINITY) ? 0.f : ex2(mw - M);
                        lt += src[D + 1] * c;
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            ot[e].x += src[dim0 + 2 * e] * c;
                            ot[e].y += src[dim0 + 2 * e + 1] * c;
                            ot[4 + e].x += src[dim1 + 2 * e] * c;
                            ot[4 + e].y += src[dim1 + 2 * e + 1] * c;
                        }
                    }
                    m[g] = M;
                    l[g] = lt;
#pragma unroll
                    for (int e = 0; e < 8; ++e) o2[g][e] = ot[e];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&merge_bar[1]);
            if (!__all_sync(0xffffffffu, mbar_wait(&merge_bar[1], merges & 1, a.err))) break;
            ++merges;
        }
        if (wrank == 0 && grp == 0) {
            const int64_t slot = (int64_t)piece + b;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int64_t qh = qh0 + g;
                float* dst = a.part_o + (slot * a.hq + qh) * D;
                *reinterpret_cast<float4*>(dst + dim0) =
                    make_float4(o2[g][0].x, o2[g][0].y, o2[g][1].x, o2[g][1].y);
                *reinterpret_cast<float4*>(dst + dim0 + 4) =
                    make_float4(o2[g][2].x, o2[g][2].y, o2[g][3].x, o2[g][3].y);
                *reinterpret_cast<float4*>(dst + dim1) =
                    make_float4(o2[g][4].x, o2[g][4].y, o2[g][5].x, o2[g][5].y);
                *reinterpret_cast<float4*>(dst + dim1 + 4) =
                    make_float4(o2[g][6].x, o2[g][6].y, o2[g][7].x, o2[g][7].y);
                if (tl == 0) {
                    a.part_ml[(slot * a.hq + qh) * 2 + 0] = m[g];
                    a.part_ml[(slot * a.hq + qh) * 2 + 1] = l[g];
                }
            }
        }
        fresh = false;  // the next tile starts a new piece
    }
    if (a.done) {  // every consumer warp has stored its partial states
        asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(a.done, 1u);
        }
    }
}

template <int D, bool BF16, int G>
__global__ void __launch_bounds__(decode_threads<G>(), 1) decode_split_kernel(const DecodeArgs a) {
    split_cta<D, BF16, G>(a, blockIdx.x, blockIdx.y, gridDim.x);
}


// Inputs of the combine kernel.
struct CombineArgs {
    const float* part_o;
    const float* part_ml;
    const int32_t* tstart;  // null: no split pieces (the prefix chunks hold every key)
    int32_t batch;
    int ctas;
    int hq;
    void* out;
    // shared-prefix mode (else null): x_chunks prefix partials per (sequence,
    // head), normalised output (bf16) and log2-sum-exp
    const uint16_t* x_out;
    const float* x_lse;
    int x_chunks;
    // in-place append (else null): sequence b's new token (k_new, v_new
    // [batch, hkv, D]) joins the attention as one more key and is written to
    // the cache at position seqlens[b] through the block table
    const void* q;
    const void* k_new;
    const void* v_new;
    unsigned char* k_cache;
    unsigned char* v_cache;
    const int32_t* table;
    const int32_t* seqlens;
    int64_t num_blocks;
    int32_t max_blocks;
    int32_t block_size;
    int32_t hkv;
    float qscale;
    unsigned int* err;
};

constexpr int kCombineWarps = 4;  // (sequence, head) pairs per CTA of the combine

// DPL consecutive elements of a bf16 or fp32 row as fp32
template <bool BF16, int DPL>
__device__ __forceinline__ void load_row(const void* base, int64_t elem, float* x) {
    if constexpr (BF16) {
        const uint16_t* p = static_cast<const uint16_t*>(base) + elem;
        if constexpr (DPL == 4) {
            const uint2 w = *reinterpret_cast<const uint2*>(p);
            x[0] = bf16lo(w.x); x[1] = bf16hi(w.x); x[2] = bf16lo(w.y); x[3] = bf16hi(w.y);
        } else {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
            x[0] = bf16lo(w); x[1] = bf16hi(w);
        }
    } else {
        const float* p = static_cast<const float*>(base) + elem;
        if constexpr (DPL == 4) {
            const float4 w = *reinterpret_cast<const float4*>(p);
            x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
        } else {
            const float2 w = *reinterpret_cast<const float2*>(p);
            x[0] = w.x; x[1] = w.y;
        }
    }
}

// The boxed merge rule applied to a running state (M, L, acc) and one more
// state (m, l, o): M' = max(M, m), both sides rescaled by 2^(. - M').  A state
// with m = -inf holds nothing and is skipped.
template <int DPL>
__device__ __forceinline__ void merge_state(float& M, float& L, float* acc, float m, float l,
                                            const float* o) {
    if (m == -INFINITY) return;
    const float Mn = fmaxf(M, m);
    const float a = (M == -INFINITY) ? 0.f : ex2(M - Mn);
    const float w = ex2(m - Mn);
    L = L * a + l * w;
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = acc[e] * a + o[e] * w;
    M = Mn;
}

// Merge the partial states of every (sequence, head) and normalise.  One warp
// per (sequence, head); lane i owns dims [i*D/32, (i+1)*D/32).  Each state
// joins a running (M, L, acc) by the boxed rule as it arrives, so the loads of
// U split pieces (and, first, of the prefix chunks and the new key) are in
// flight together: a sequence with up to U pieces costs one memory round trip
// after the split (the tile starts are read before the wait).  U is
// 16 for batches of few sequences (long contexts, many pieces each) and 4 for
// large batches, whose warps must all fit on the GPU at once.  Shared-prefix
// mode adds the prefix chunks, each as the state (m = lse, l = 1, o = out);
// append mode adds the new key (m = its score, l = 1, o = its V row) and the
// first warp of each KV head writes the new K/V row into the cache (the split
// kernel, which read only the keys before it, has completed).
// The combine of (sequence, head) pair w by one warp.  With pdl_wait the warp
// waits for the split grid (griddepcontrol.wait) after its own loads; without
// it the caller has already waited for the split's states.
// With H = 2, two warps share pair w: warp `half` merges its half of the
// split's pieces, and half 1 hands its state to half 0 through xch (shared
// memory, 32 * (D / 32 + 2) floats) at named barrier bar_id (64 threads);
// half 0 alone takes the prefix chunks and the appended key, and stores.
template <int D, bool BF16, int U, int H = 1>
__device__ __forceinline__ void combine_warp(const CombineArgs& c, const int64_t w,
                                             const bool pdl_wait, const int half = 0,
                                             float* xch = nullptr, const int bar_id = 0) {
    constexpr int DPL = D / 32;
    const int lane = threadIdx.x & 31;
    const int hq = c.hq, batch = c.batch;
    const bool live = w < (int64_t)batch * hq;
    const int b = live ? (int)(w / hq) : 0, h = live ? (int)(w % hq) : 0;
    const int64_t bh = (int64_t)b * hq + h;
    const int G = hq / (c.hkv > 0 ? c.hkv : 1);
    const int kvh = h / G;
    // Before the wait: what the split kernel does not write (the appended
    // key's score and V row, and where its K/V row goes), so that these loads
    // overlap the split kernel's tail.
    float M = -INFINITY, L = 0.f, acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
    int64_t new_slot = -1;  // the appended row's slot, when this warp writes it
    if (c.k_new && live && (H == 1 || half == 0)) {  // the appended key: q . k_new, log2 units
        const int64_t row = ((int64_t)b * c.hkv + kvh) * D + lane * DPL;
        float qv[DPL], kv[DPL], vv[DPL];
        load_row<BF16, DPL>(c.q, bh * D + lane * DPL, qv);
        load_row<BF16, DPL>(c.k_new, row, kv);
        load_row<BF16, DPL>(c.v_new, row, vv);
        if (h % G == 0) {  // the first warp of each KV head writes the row
            const int32_t Lb = c.seqlens[b];
            const int32_t B = c.block_size;
            if (Lb < 0 || Lb >= c.max_blocks * B) {
                if (lane == 0) flag_error(c.err, PKV_FLAG_BAD_LENGTH);
            } else {
                const int32_t phys = c.table[(int64_t)b * c.max_blocks + Lb / B];
                if (phys < 0 || phys >= c.num_blocks) {
                    if (lane == 0) flag_error(c.err, PKV_FLAG_BAD_BLOCK);
                } else {
                    new_slot = (int64_t)phys * B + Lb % B;
                }
            }
        }
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) dot = fmaf(qv[e], kv[e], dot);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
        merge_state<DPL>(M, L, acc, dot * c.qscale, 1.f, vv);
    }
    // The split's tile starts: stored (and fenced) by its first block before
    // any of its blocks let this kernel start, so they are read before the
    // wait, from L2.
    int32_t total = 0, tb0 = 0, tb1 = 0;
    if (c.tstart && live) {
        total = __ldcg(c.tstart + batch);
        tb0 = __ldcg(c.tstart + b);
        tb1 = __ldcg(c.tstart + b + 1);
    }
    // wait until the split kernel's partials are complete and visible
    if (pdl_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!live) return;
    const int32_t chunk = share_cost(total, batch, c.ctas);
    const int32_t ub = kSeqCost * (b + 1);  // u(t) - t for this sequence's tiles
    int c0 = (tb0 + ub) / chunk, c1 = tb1 > tb0 ? (tb1 - 1 + ub) / chunk : c0 - 1;
    if constexpr (H == 2) {  // this warp's half of the pieces
        const int mid = c0 + (c1 - c0 + 2) / 2;
        if (half == 0) c1 = mid - 1;
        else c0 = mid;
    }
    // the prefix chunks' states (rounds of UX), then the split's pieces c0 ..
    // c1 (rounds of U), every load of a round in flight
    constexpr int UX = U < 8 ? U : 8;
    const int64_t xstride = (int64_t)batch * hq;  // one prefix chunk's (sequence, head) count
    for (int base = 0; (H == 1 || half == 0) && base < c.x_chunks; base += UX) {
        float mx[UX];
        float xo[UX][DPL];
#pragma unroll
        for (int i = 0; i < UX; ++i) {
            mx[i] = -INFINITY;
            if (base + i < c.x_chunks) {
                const int64_t xi = (int64_t)(base + i) * xstride + bh;
                mx[i] = c.x_lse[xi];
                load_row<true, DPL>(c.x_out, xi * D + lane * DPL, xo[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < UX; ++i) merge_state<DPL>(M, L, acc, mx[i], 1.f, xo[i]);
    }
    for (int base = c0; base <= c1; base += U) {
        float2 ml[U];
        float o[U][DPL];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            ml[i] = make_float2(-INFINITY, 0.f);
            if (base + i <= c1) {
                const int64_t slot = (int64_t)(base + i) + b;
                ml[i] = *reinterpret_cast<const float2*>(c.part_ml + (slot * hq + h) * 2);
                load_row<false, DPL>(c.part_o, (slot * hq + h) * D + lane * DPL, o[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < U; ++i) merge_state<DPL>(M, L, acc, ml[i].x, ml[i].y, o[i]);
    }
    if constexpr (H == 2) {  // half 1's state joins half 0's
        float* x = xch + lane * (DPL + 2);
        if (half == 1) {
            x[0] = M;
            x[1] = L;
#pragma unroll
            for (int e = 0; e < DPL; ++e) x[2 + e] = acc[e];
        }
        asm volatile("bar.sync %0, 64;" ::"r"(bar_id) : "memory");
        if (half == 1) return;
        float o1[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) o1[e] = x[2 + e];
        merge_state<DPL>(M, L, acc, x[0], x[1], o1);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int64_t oi = bh * D + lane * DPL;
    if constexpr (BF16) {
        uint16_t* o = static_cast<uint16_t*>(c.out) + oi;
        if constexpr (DPL == 4) {
            *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                      pack_bf16x2(acc[2] * inv, acc[3] * inv));
        } else {
            *reinterpret_cast<uint32_t*>(o) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        }
    } else {
        float* o = static_cast<float*>(c.out) + oi;
#pragma unroll
        for (int e = 0; e < DPL; ++e) o[e] = acc[e] * inv;
    }
    // the new K/V row into the cache (after the wait: the split kernel has
    // read every cached key)
    if (new_slot >= 0) {
        constexpr int ELT = BF16 ? 2 : 4;
        const int64_t src = ((int64_t)b * c.hkv + kvh) * D + lane * DPL;
        const int64_t dst = (new_slot * c.hkv + kvh) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL * ELT; e += 4) {
            *reinterpret_cast<uint32_t*>(c.k_cache + dst * ELT + e) =
                *reinterpret_cast<const uint32_t*>(static_cast<const unsigned char*>(c.k_new) +
                                                   src * ELT + e);
            *reinterpret_cast<uint32_t*>(c.v_cache + dst * ELT + e) =
                *reinterpret_cast<const uint32_t*>(static_cast<const unsigned char*>(c.v_new) +
                                                   src * ELT + e);
        }
    }
}

template <int D, bool BF16, int U>
__global__ void __launch_bounds__(kCombineWarps * 32, U > 8 ? 4 : (U > 4 ? 7 : 8))
decode_combine_kernel(const CombineArgs c) {
    combine_warp<D, BF16, U>(c, (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5), true);
}

// Two warps per (sequence, head): for few sequences with more pieces each
// than one round holds, so that every piece is loaded in one round.
template <int D, bool BF16, int U>
__global__ void __launch_bounds__(kCombineWarps * 32, 4) decode_combine2_kernel(const CombineArgs c) {
    __shared__ float xch[kCombineWarps / 2][32 * (D / 32 + 2)];
    const int warp = threadIdx.x >> 5, p = warp >> 1;
    combine_warp<D, BF16, U, 2>(c, (int64_t)blockIdx.x * (kCombineWarps / 2) + p, true, warp & 1,
                                xch[p], 1 + p);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static int largest_pow2_divisor(int x, int cap) {
    int r = 1;
    while (r * 2 <= cap && x % (r * 2) == 0) r *= 2;
    return r;
}

bool plan_decode(const DeviceInfo& dev, int32_t batch, int hq, int hkv, int d, int block_size,
                 int elt, DecodePlan* p) {
    if (d != 64 && d != 128) return false;
    if (hkv <= 0 || hq % hkv) return false;
    const int G = hq / hkv;
    // groups of 1, 2 and 4, and of 8, 16 and 32: G / 4 warps per KV head, each
    // with 4 of its query heads, share the K/V tile (G / 4 divides the 8
    // consumer warps, so every warp has a KV head and a subset)
    int gsplit = 1;
    if (G == 1 || G == 2 || G == 4) gsplit = 1;
    else if (G == 8 || G == 16 || G == 32) gsplit = G / 4;
    else return false;
    const int G_warp = G / gsplit;  // query heads a consumer warp holds
    if (batch < 0 || batch > kDecodeMaxBatch) return false;
    if (block_size > (1 << 24)) return false;  // the producer packs slot * 64 + rows
    int HC;  // KV heads per CTA: gsplit warps each, 8 consumer warps
    const int head_slots = kConsumerWarps / gsplit;
    if (hkv <= head_slots) {
        if (head_slots % hkv) return false;
        HC = hkv;
    } else {
        if (hkv % head_slots) return false;
        HC = head_slots;
    }
    const size_t row_bytes = (size_t)HC * d * elt;
    // ~64 KiB of K+V per stage, at most 32 keys
    int cap_rows = (int)(65536 / (2 * row_bytes));
    if (cap_rows < 1) cap_rows = 1;
    if (cap_rows > 32) cap_rows = 32;
    const int R = largest_pow2_divisor(block_size, cap_rows);
    const size_t stage = 2 * (size_t)R * row_bytes;
    const size_t fixed = decode_fixed_smem(G_warp, d, batch);
    if (dev.max_smem_optin < fixed + 2 * stage) return false;
    int stages = (int)((dev.max_smem_optin - fixed) / stage);
    if (stages > kMaxStages) stages = kMaxStages;
    p->heads_per_cta = HC;
    p->gsplit = gsplit;
    p->head_groups = hkv / HC;
    p->ctas = dev.num_sms / p->head_groups > 0 ? dev.num_sms / p->head_groups : 1;
    p->rows_per_tile = R;
    p->stages = stages;
    p->smem_bytes = fixed + (size_t)stages * stage;
    const size_t slots = (size_t)p->ctas + batch;
    p->ws_bytes = align_up((size_t)(batch + 1) * 4, 256) + align_up(slots * hq * 2 * 4, 256) +
                  align_up(slots * hq * d * 4, 256);
    return true;
}

template <int D, bool BF16, int G>
static cudaError_t launch_decode_t(const DecodePlan& plan, const DecodeArgs& a,
                                   const CombineArgs& c, bool split, cudaStream_t stream) {
    if (split) {
        auto kern = decode_split_kernel<D, BF16, G>;
        cudaError_t e = cudaFuncSetAttribute(
            kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)plan.smem_bytes);
        if (e != cudaSuccess) return e;
        e = launch_dependent(kern, dim3(plan.ctas, plan.head_groups),
                             dim3(decode_threads<G>()), plan.smem_bytes, stream, a);
        if (e != cudaSuccess) return e;
    }
    // combine: programmatic dependent of the split kernel, one warp per
    // (sequence, head), or two when a sequence has more pieces than a round
    // of 16 and the warps fit beside the split's CTAs (one round each, up to
    // 32 pieces).  Pieces in flight per round:
    //  - 8 when a sequence has few pieces (about ctas / batch + 2 <= 8) and
    //    every warp fits beside the split's CTAs while they run (72 registers:
    //    two 4-warp CTAs per SM next to a split CTA), so all start early;
    //  - 16 while every warp of the batch fits on the GPU at once (4 warps a
    //    CTA, 4 CTAs an SM);
    //  - else 4.
    cudaLaunchConfig_t cfg = {};
    const int64_t warps = (int64_t)a.batch * a.hq;
    cfg.gridDim = dim3((unsigned)((warps + kCombineWarps - 1) / kCombineWarps));
    cfg.blockDim = dim3(kCombineWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int64_t per_seq = (int64_t)plan.ctas / (a.batch > 0 ? a.batch : 1) + 2;
    if (c.tstart && per_seq > 16 && per_seq <= 32 &&
        2 * warps <= (int64_t)plan.ctas * plan.head_groups * kCombineWarps) {
        cfg.gridDim = dim3((unsigned)((warps + kCombineWarps / 2 - 1) / (kCombineWarps / 2)));
        return cudaLaunchKernelEx(&cfg, decode_combine2_kernel<D, BF16, 16>, c);
    }
    if (per_seq <= 8 && warps <= (int64_t)plan.ctas * plan.head_groups * 2 * kCombineWarps)
        return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D, BF16, 8>, c);
    if (warps <= (int64_t)plan.ctas * plan.head_groups * 4 * kCombineWarps)
        return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D, BF16, 16>, c);
    return cudaLaunchKernelEx(&cfg, decode_combine_kernel<D, BF16, 4>, c);
}

// The split's and the combine's arguments (workspace carved as the plan sized it).
static void fill_decode_args(const DecodePlan& plan, const void* q, const void* k_cache,
                             const void* v_cache, const int32_t* block_table, int32_t max_blocks,
                             const int32_t* cache_seqlens, int32_t batch, float scale, void* out,
                             void* workspace, int hq, int hkv, int block_size, int64_t num_blocks,
                             unsigned int* err, const SharedPrefix* sp, const DecodeAppend* ap,
                             const DecodeChain* chain, DecodeArgs* pa, CombineArgs* pc) {
    DecodeArgs& a = *pa;
    a = DecodeArgs{};
    a.wait_prior = (chain && chain->pdl_split) ? 1 : 0;
    a.wait_inputs = a.wait_prior ? 0 : 1;
    a.group_cu = sp ? sp->group_cu : nullptr;
    a.group_plen = sp ? sp->group_plen : nullptr;
    a.n_groups = sp ? sp->n_groups : 0;

    a.q = q;
    a.k_cache = static_cast<const unsigned char*>(k_cache);
    a.v_cache = static_cast<const unsigned char*>(v_cache);
    a.table = block_table;
    a.seqlens = cache_seqlens;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    const size_t slots = (size_t)plan.ctas + batch;
    a.tstart_out = reinterpret_cast<int32_t*>(ws);
    ws += align_up((size_t)(batch + 1) * 4, 256);
    a.part_ml = reinterpret_cast<float*>(ws);
    ws += align_up(slots * hq * 2 * 4, 256);
    a.part_o = reinterpret_cast<float*>(ws);
    a.err = err;
    a.num_blocks = num_blocks;
    a.qscale = scale * kLog2e;
    a.max_blocks = max_blocks;
    a.batch = batch;
    a.hq = hq;
    a.hkv = hkv;
    a.hc = plan.heads_per_cta;
    a.gfull = hq / hkv;
    a.gsplit = plan.gsplit;
    a.block_size = block_size;
    a.rows = plan.rows_per_tile;
    a.stages = plan.stages;
    CombineArgs& c = *pc;
    c = CombineArgs{};
    c.part_o = a.part_o;
    c.part_ml = a.part_ml;
    const bool split = !(chain && chain->no_split);
    c.tstart = split ? a.tstart_out : nullptr;
    c.batch = batch;
    c.ctas = plan.ctas;
    c.hq = hq;
    c.out = out;
    if (sp) {
        c.x_out = static_cast<const uint16_t*>(sp->x_out);
        c.x_lse = sp->x_lse;
        c.x_chunks = sp->x_chunks;
    }
    if (ap) {
        c.q = q;
        c.k_new = ap->k_new;
        c.v_new = ap->v_new;
        c.k_cache = static_cast<unsigned char*>(ap->k_cache);
        c.v_cache = static_cast<unsigned char*>(ap->v_cache);
        c.table = block_table;
        c.seqlens = cache_seqlens;
        c.num_blocks = num_blocks;
        c.max_blocks = max_blocks;
        c.block_size = block_size;
    }
    c.hkv = hkv;
    c.qscale = a.qscale;
    c.err = err;
}

cudaError_t launch_decode(const DecodePlan& plan, const void* q, const void* k_cache,
                          const void* v_cache, const int32_t* block_table, int32_t max_blocks,
                          const int32_t* cache_seqlens, int32_t batch, float scale, void* out,
                          void* workspace, int hq, int hkv, int d, int block_size,
                          int64_t num_blocks, int dtype, unsigned int* err, cudaStream_t stream,
                          const SharedPrefix* sp, const DecodeAppend* ap,
                          const DecodeChain* chain) {
    if (batch == 0) return cudaSuccess;
    DecodeArgs a;
    CombineArgs c;
    fill_decode_args(plan, q, k_cache, v_cache, block_table, max_blocks, cache_seqlens, batch,
                     scale, out, workspace, hq, hkv, block_size, num_blocks, err, sp, ap, chain,
                     &a, &c);
    const bool split = !(chain && chain->no_split);
    const int G = hq / hkv / plan.gsplit;  // query heads per consumer warp
    const bool bf = dtype == PKV_BF16;
#define PKV_DECODE_CASE(DD, BB, GG) \
    if (d == DD && bf == BB && G == GG) \
        return launch_decode_t<DD, BB, GG>(plan, a, c, split, stream);
    PKV_DECODE_CASE(128, true, 1) PKV_DECODE_CASE(128, true, 2) PKV_DECODE_CASE(128, true, 4)
    PKV_DECODE_CASE(128, false, 1) PKV_DECODE_CASE(128, false, 2) PKV_DECODE_CASE(128, false, 4)
    PKV_DECODE_CASE(64, true, 1) PKV_DECODE_CASE(64, true, 2) PKV_DECODE_CASE(64, true, 4)
    PKV_DECODE_CASE(64, false, 1) PKV_DECODE_CASE(64, false, 2) PKV_DECODE_CASE(64, false, 4)
#undef PKV_DECODE_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pkv
