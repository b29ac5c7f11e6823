// step.cu -- the translation unit of the decode, write and tensor-core kernels,
// and the continuous-batching step as ONE launch.
//
// decode.cu, write.cu and prefill.cu are compiled here as one unit, so that a
// single kernel can run their CTA functions: split_cta and combine_warp
// (decode.cu), prefix_cta and prefill_cta (prefill.cu).
//
// What the one-launch step computes is paged_mixed_step's result
// ("从零开始写Qwen3（六）PagedAttention", fast-attn 库的使用: one step mixes the
// varlen prefill call and the kvcache decode call; "Sayfalı dikkat", decode
// path: the kvcache call writes the new k and v in place; "11. Paged attention
// 与 online softmax" §11.3: blocks shared by several sequences):
//   1. the prefill requests' new K/V rows written at their slots;
//   2. the causal varlen prefill over the cache, and the attention of every
//      decode group's queries over its shared prefix, on the tensor cores;
//   3. each decode sequence's own keys by the split;
//   4. the combine: prefix chunks, split pieces and the appended token merged
//      by the boxed rule, the new K/V row of every decode sequence written.
//
// GB300 design.  One grid of 384-thread CTAs in this block order: [prefix
// items][prefill items][split CTAs][combine CTAs].  The SMs take blocks in that order as they
// free up, as with the chained launches.  In-grid dependencies replace the
// launch boundaries: a CTA that feeds later ones adds 1 to a counter once its
// results are stored, and a CTA that needs them waits, time-limited, until the
// count is complete.  The first wave (the first n_write = min(SMs, items)
// tensor-core items, all dispatched at once) first writes the prefill rows, a
// warp per row, and counts its shares; the prefill items wait for all of them.
// The combine CTAs (at most one per split CTA)
// wait until every prefix item and split CTA has counted, and their 12 warps
// then take the (sequence, head) pairs in turn.  Every CTA of one launch has
// the largest item's resources (one CTA per SM), so the combine is cut into
// as many CTAs as there are split CTAs, not one per 12 pairs, which would run
// in waves.  A CTA waits only for blocks placed before it, which in-order
// dispatch has made resident or finished.  The counters live in the workspace
// and are zeroed on the stream before the launch.
#include "decode.cu"
#include "write.cu"
#include "prefill.cu"

namespace pkv {
namespace {

struct StepOne {
    // the prefill requests' new rows: bf16, kvDim * 2 bytes per row
    const uint4* k_new;
    const uint4* v_new;
    const int32_t* slots;  // < 0: padding row, nothing written
    uint4* k_cache;
    uint4* v_cache;
    int64_t rows;
    int64_t vec_per_row;  // 16-byte vectors per row
    int64_t num_slots;
    int32_t n_tc;       // tensor-core items: g.n_prefix prefix items, then prefill items
    int32_t n_write;    // the first n_write items write the prefill rows
    int32_t n_split;    // split CTAs
    int32_t n_combine;  // combine CTAs
    unsigned int* counters;  // [0] row shares written, [1] prefix items, [2] split CTAs done
    unsigned int* err;
};

constexpr int kStepWarps = kThreads / 32;

// One thread waits until *ctr >= target (acquire), at most kWaitLimitNs; a
// wait that runs out flags PKV_FLAG_TIMEOUT and returns false.
__device__ bool wait_count(const unsigned int* ctr, unsigned int target, unsigned int* err) {
    const uint64_t t0 = global_ns();
    for (;;) {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if (global_ns() - t0 > kWaitLimitNs) {
            flag_error(err, PKV_FLAG_TIMEOUT);
            return false;
        }
        __nanosleep(256);
    }
}

// The CTA's results are stored: count it (one thread, after a CTA barrier).
__device__ __forceinline__ void publish(unsigned int* ctr) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
    }
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
step_one_kernel(const __grid_constant__ CUtensorMap fq, const __grid_constant__ CUtensorMap fo,
                const __grid_constant__ CUtensorMap fk, const __grid_constant__ CUtensorMap fv,
                const __grid_constant__ CUtensorMap xq, const __grid_constant__ CUtensorMap xk,
                const __grid_constant__ CUtensorMap xv, const PrefillArgs pa, const PrefixArgs xa,
                const TcGrid g, const DecodeArgs da, const CombineArgs ca, const StepOne s) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int item = (int)blockIdx.x;
    if (item < s.n_tc) {
        if (item < s.n_write) {
            // this item's share of the prefill rows: a warp per row, 16-byte
            // vectors of K and V to the row's slot
            for (int64_t r = (int64_t)item * kStepWarps + warp; r < s.rows;
                 r += (int64_t)s.n_write * kStepWarps) {
                const int32_t slot = __ldg(s.slots + r);
                if (slot < 0) continue;
                if (slot >= s.num_slots) {
                    if (lane == 0) flag_error(s.err, PKV_FLAG_BAD_SLOT);
                    continue;
                }
                const uint4* ks = s.k_new + r * s.vec_per_row;
                const uint4* vs = s.v_new + r * s.vec_per_row;
                uint4* kd = s.k_cache + (int64_t)slot * s.vec_per_row;
                uint4* vd = s.v_cache + (int64_t)slot * s.vec_per_row;
                for (int64_t i = lane; i < s.vec_per_row; i += 32) {
                    const uint4 a = __ldcs(ks + i), b = __ldcs(vs + i);
                    kd[i] = a;
                    vd[i] = b;
                }
            }
            // the prefill items read these rows with TMA (the async proxy)
            asm volatile("fence.proxy.async.global;" ::: "memory");
            publish(s.counters + 0);
        }
        if (item < g.n_prefix) {
            prefix_cta<HD>(xq, xk, xv, xa, item % g.px, (item / g.px) % g.py,
                           item / (g.px * g.py));
            publish(s.counters + 1);
        } else {
            if (threadIdx.x == 0 && wait_count(s.counters + 0, (unsigned)s.n_write, s.err))
                asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncthreads();
            item -= g.n_prefix;
            prefill_cta<HD>(fq, fo, fk, fv, pa, item % g.fx, (item / g.fx) % g.fy,
                            item / (g.fx * g.fy));
        }
        return;
    }
    item -= s.n_tc;
    if (item < s.n_split) {
        split_cta<HD, true, 2>(da, item, 0, s.n_split);  // counts itself in da.done
        return;
    }
    item -= s.n_split;
    if (threadIdx.x == 0) {
        wait_count(s.counters + 1, (unsigned)g.n_prefix, s.err);
        wait_count(s.counters + 2, (unsigned)s.n_split, s.err);
    }
    __syncthreads();
    const int64_t pairs = (int64_t)ca.batch * ca.hq;
    for (int64_t w = (int64_t)item * kStepWarps + warp; w < pairs;
         w += (int64_t)s.n_combine * kStepWarps)
        combine_warp<HD, true, 4>(ca, w, false);
}

}  // namespace

cudaError_t launch_step_one(const DeviceInfo& dev, const StepOneLaunch& st,
                            cudaStream_t stream) {
    const PrefixLaunch& pp = st.prefix;
    const int d = pp.hd;
    if (st.dtype != PKV_BF16 || d != 128) return cudaErrorNotSupported;
    if (st.hq / st.hkv != 2 || st.plan.gsplit != 1 || st.plan.head_groups != 1)
        return cudaErrorNotSupported;
    if (st.pf_new_tokens < 0 || ((uintptr_t)st.pf_k_new & 15) || ((uintptr_t)st.pf_v_new & 15))
        return cudaErrorNotSupported;
    // tensor-core items
    PrefillArgs pa{};
    CUtensorMap fm[4];
    int fx, fy, fz;
    cudaError_t e = prepare_prefill(st.pf_q, st.k_cache, st.v_cache, st.cu_q, st.cu_k,
                                    st.pf_batch, st.max_seqlen_q, st.pf_table, st.pf_max_blocks,
                                    1, st.scale, st.pf_out, st.hq, st.hkv, d, st.block_size,
                                    st.num_blocks, dev.err, &pa, fm, &fx, &fy, &fz);
    if (e != cudaSuccess) return e;
    PrefixArgs xa{};
    CUtensorMap xm[3];
    int px, py, pz;
    e = prepare_prefix(pp, &xa, xm, &px, &py, &pz);
    if (e != cudaSuccess) return e;
    const int64_t nf = (int64_t)fx * fy * fz, np = (int64_t)px * py * pz;
    TcGrid g{(int)np, px > 0 ? px : 1, py > 0 ? py : 1, fx > 0 ? fx : 1, fy > 0 ? fy : 1};
    // decode: split + combine, counted in the grid
    DecodeArgs da;
    CombineArgs ca;
    SharedPrefix sp{pp.group_cu, pp.group_plen, pp.n_groups, pp.x_out, pp.x_lse, pp.kchunks};
    DecodeAppend ap{st.dec_k_new, st.dec_v_new, st.k_cache, st.v_cache};
    DecodeChain ch{false, false};
    fill_decode_args(st.plan, pp.q, st.k_cache, st.v_cache, pp.table, pp.max_blocks,
                     st.dec_seqlens, pp.batch, st.scale, st.dec_out, st.workspace, st.hq, st.hkv,
                     st.block_size, st.num_blocks, dev.err, &sp, &ap, &ch, &da, &ca);
    da.wait_prior = 0;
    da.wait_inputs = 0;
    da.done = st.counters + 2;
    const int64_t warps = (int64_t)pp.batch * st.hq;
    StepOne s{};
    s.k_new = static_cast<const uint4*>(st.pf_k_new);
    s.v_new = static_cast<const uint4*>(st.pf_v_new);
    s.slots = st.pf_slots;
    s.k_cache = static_cast<uint4*>(st.k_cache);
    s.v_cache = static_cast<uint4*>(st.v_cache);
    s.rows = st.pf_new_tokens;
    s.vec_per_row = (int64_t)st.hkv * d * 2 / 16;
    s.num_slots = st.num_blocks * st.block_size;
    s.n_tc = (int32_t)(nf + np);
    s.n_split = st.plan.ctas;
    s.counters = st.counters;
    s.err = dev.err;
    s.n_write = (int32_t)std::min<int64_t>(dev.num_sms, nf + np);
    s.n_combine = (int32_t)std::max<int64_t>(
        1, std::min<int64_t>(s.n_split, (warps + kStepWarps - 1) / kStepWarps));
    const int64_t blocks = (int64_t)s.n_tc + s.n_split + s.n_combine;
    if (blocks > 0x7fffffffLL) return cudaErrorNotSupported;
    const size_t smem =
        std::max({Shape<128>::kSmemBytes, PShape<128>::kSmemBytes, st.plan.smem_bytes});
    if (dev.max_smem_optin < smem) return cudaErrorNotSupported;
    auto kern = step_one_kernel<128>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(st.counters, 0, 4 * sizeof(unsigned int), stream);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)blocks, kThreads, smem, stream>>>(fm[0], fm[1], fm[2], fm[3], xm[0], xm[1],
                                                       xm[2], pa, xa, g, da, ca, s);
    return cudaGetLastError();
}

}  // namespace pkv
