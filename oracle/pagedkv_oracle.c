/*
 * pagedkv_oracle.c -- plain, slow, obviously-correct CPU oracle for the paged
 * KV-cache hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file; only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Every floating-point result is computed in IEEE double precision from inputs
 * widened exactly (fp32 -> fp64 and bf16 -> fp64 are both exact).  There is no
 * blocking, fusion or reordering beyond what each cited definition states.
 *
 * Sources (web pages on paged attention):
 *   [P1] "11. Paged attention 与 online softmax" (dilfish.github.io):
 *        §11.1 block-table equations, §11.2 boxed merge equation, §11.3.
 *   [P2] "结合nanovllm的FlashAttention和PagedAttention主要原理概述"
 *        (meredith2328.github.io): 题目2 online softmax, 题目3 FlashAttention
 *        worked example, 题目5 block table.
 *   [P3] "从零开始写Qwen3（六）PagedAttention" (mlqm.cn): sections
 *        "分页自注意力的改进" (address formula), "fast-attn 库的使用"
 *        (call shapes, causal prefill over a prefix cache), "自己来实现一个"
 *        (slot_mapping cache-write kernel).
 *   [P4] "Sayfalı dikkat" (Hugging Face transformers docs): varlen path
 *        example (cu_seq_lens) and decode path example (cache_seqlens).
 *
 * Readings taken where the pages are silent or garbled (each is listed in the
 * design notes of the repository):
 *   - cache layout [num_blocks, B, Hkv, d], row stride kvDim = Hkv*d ([P1]
 *     offset equation; [P3] address arithmetic of its loader);
 *   - a negative slot is skipped by the write ([P3] write kernel, comparison
 *     sign lost in extraction);
 *   - causal masking is bottom-right aligned: query i of a request with q_len
 *     queries and k_len keys sees key j iff j <= i + k_len - q_len;
 *   - a query row that sees no key outputs 0;
 *   - query head h reads kv head h / (Hq/Hkv).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORA_F32 = 0, ORA_BF16 = 1 };

/* ------------------------------------------------------------------------ */
/* Element access.  bf16 is the upper half of an IEEE binary32, so widening  */
/* is a shift; both widenings to double are exact.                           */
/* ------------------------------------------------------------------------ */
static double widen_bf16(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void* base, int dtype, int64_t idx) {
    if (dtype == ORA_F32) return (double)((const float*)base)[idx];
    return widen_bf16(((const uint16_t*)base)[idx]);
}

/* Round an fp32 value to bf16, round-to-nearest, ties-to-even, on the bit
 * pattern (NaN stays a quiet NaN).  This is the cast the [P3] write kernel
 * applies when the source and cache dtypes differ. */
static uint16_t bf16_round_nearest_even(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

uint16_t ora_f32_to_bf16(float f) { return bf16_round_nearest_even(f); }

int ora_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* a0 -- block-table address translation.                                    */
/* [P1] §11.1: logical block lb = floor(p / B), slot = p mod B,              */
/* phys = table[lb]; element offset = phys*B*kvDim + slot*kvDim.             */
/* [P2] 题目5 and [P3] "分页自注意力的改进" state the same mapping.          */
/* The "slot id" used by slot_mapping is phys*B + slot, so the element       */
/* offset is slot_id * kvDim.                                                */
/* ------------------------------------------------------------------------ */
int64_t ora_slot_id(const int32_t* table_row, int32_t block_size, int64_t pos) {
    int64_t logical_block = pos / block_size;
    int64_t slot = pos % block_size;
    int64_t phys = table_row[logical_block];
    return phys * block_size + slot;
}

int64_t ora_element_offset(const int32_t* table_row, int32_t block_size, int64_t kv_dim,
                           int64_t pos) {
    int64_t logical_block = pos / block_size;
    int64_t slot = pos % block_size;
    int64_t phys = table_row[logical_block];
    return phys * block_size * kv_dim + slot * kv_dim;
}

/* slot_mapping for the new tokens of a step ([P3] "自己来实现一个": the
 * per-token internal index is computed once up front and reused by every
 * layer).  Token row n belongs to sequence token_seq[n] at logical position
 * token_pos[n]; a row with token_seq[n] < 0 is padding and maps to slot -1,
 * which the write skips. */
void ora_build_slot_mapping(const int32_t* block_table, int32_t max_blocks,
                            const int32_t* token_seq, const int32_t* token_pos,
                            int64_t num_tokens, int32_t block_size, int32_t* slot_out) {
    for (int64_t n = 0; n < num_tokens; ++n) {
        if (token_seq[n] < 0) {
            slot_out[n] = -1;
            continue;
        }
        const int32_t* row = block_table + (int64_t)token_seq[n] * max_blocks;
        slot_out[n] = (int32_t)ora_slot_id(row, block_size, token_pos[n]);
    }
}

/* ------------------------------------------------------------------------ */
/* a1 -- slot_mapping cache write ([P3] "自己来实现一个",                     */
/* _update_paged_kv_cache_kernel): token n with slot s >= 0 copies its K and */
/* V rows (kvDim elements) to cache[s*kvDim ...], cast to the cache dtype;   */
/* a negative slot writes nothing.                                           */
/* ------------------------------------------------------------------------ */
static void store_elem(void* base, int dtype, int64_t idx, const void* src, int src_dtype,
                       int64_t sidx) {
    if (dtype == src_dtype) {
        if (dtype == ORA_F32) ((float*)base)[idx] = ((const float*)src)[sidx];
        else ((uint16_t*)base)[idx] = ((const uint16_t*)src)[sidx];
    } else if (dtype == ORA_BF16) { /* fp32 source -> bf16 cache */
        ((uint16_t*)base)[idx] = bf16_round_nearest_even(((const float*)src)[sidx]);
    } else { /* bf16 source -> fp32 cache: exact widening */
        ((float*)base)[idx] = (float)widen_bf16(((const uint16_t*)src)[sidx]);
    }
}

void ora_kv_write(const void* k, const void* v, int src_dtype, const int32_t* slot_mapping,
                  int64_t num_tokens, int64_t kv_dim, void* k_cache, void* v_cache,
                  int cache_dtype) {
    for (int64_t n = 0; n < num_tokens; ++n) {
        int64_t s = slot_mapping[n];
        if (s < 0) continue;
        for (int64_t j = 0; j < kv_dim; ++j) {
            store_elem(k_cache, cache_dtype, s * kv_dim + j, k, src_dtype, n * kv_dim + j);
            store_elem(v_cache, cache_dtype, s * kv_dim + j, v, src_dtype, n * kv_dim + j);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* One-shot softmax attention of one query vector over n gathered key rows.  */
/* The plain definition ([P1] §11.2 states that the paged/online result      */
/* equals this up to rounding): s_j = scale * <q, k_j>, m = max_j s_j,       */
/* p_j = exp(s_j - m), out = sum_j p_j v_j / sum_j p_j.  n == 0 gives 0.     */
/* key_off[j] is the element offset of key row j's head slice in the cache.  */
/* ------------------------------------------------------------------------ */
static void attend_one_shot(const double* q, const void* kc, const void* vc, int dtype,
                            const int64_t* key_off, int64_t n, int32_t d, double scale,
                            double* out) {
    for (int32_t i = 0; i < d; ++i) out[i] = 0.0;
    if (n == 0) return;
    double* s = (double*)malloc((size_t)n * sizeof(double));
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int32_t i = 0; i < d; ++i) dot += q[i] * load_elem(kc, dtype, key_off[j] + i);
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double p = exp(s[j] - m);
        l += p;
        for (int32_t i = 0; i < d; ++i) out[i] += p * load_elem(vc, dtype, key_off[j] + i);
    }
    for (int32_t i = 0; i < d; ++i) out[i] /= l;
    free(s);
}

/* ------------------------------------------------------------------------ */
/* a2+a3+a4 -- paged decode, one query token per sequence.                   */
/* [P4] decode path: sequence b attends over its cache_seqlens[b] keys, read */
/* through block_table row b ([P1] §11.1 addressing).  Query head h uses kv  */
/* head h / (Hq/Hkv).  q is [batch, Hq, d]; the caches are                   */
/* [num_blocks, B, Hkv, d].  Sequences listed in seq_subset (all when NULL)  */
/* are computed; out is [n_out, Hq, d] in fp64.                              */
/* ------------------------------------------------------------------------ */
void ora_decode(const void* q, const void* k_cache, const void* v_cache, int dtype,
                const int32_t* block_table, int32_t max_blocks, const int32_t* cache_seqlens,
                int32_t batch, int32_t hq, int32_t hkv, int32_t d, int32_t block_size,
                double scale, const int32_t* seq_subset, int32_t n_subset, double* out) {
    int32_t n_out = seq_subset ? n_subset : batch;
    int32_t group = hq / hkv;
    int64_t kv_dim = (int64_t)hkv * d;
    int64_t work = (int64_t)n_out * hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t w = 0; w < work; ++w) {
        int32_t o = (int32_t)(w / hq), h = (int32_t)(w % hq);
        int32_t b = seq_subset ? seq_subset[o] : o;
        int32_t kvh = h / group;
        int64_t len = cache_seqlens[b];
        const int32_t* row = block_table + (int64_t)b * max_blocks;
        int64_t* off = (int64_t*)malloc((size_t)(len > 0 ? len : 1) * sizeof(int64_t));
        for (int64_t p = 0; p < len; ++p)
            off[p] = ora_element_offset(row, block_size, kv_dim, p) + (int64_t)kvh * d;
        double* qv = (double*)malloc((size_t)d * sizeof(double));
        for (int32_t i = 0; i < d; ++i)
            qv[i] = load_elem(q, dtype, ((int64_t)b * hq + h) * d + i);
        attend_one_shot(qv, k_cache, v_cache, dtype, off, len, d, scale,
                        out + ((int64_t)o * hq + h) * d);
        free(qv);
        free(off);
    }
}

/* ------------------------------------------------------------------------ */
/* a5 -- varlen prefill over cu_seqlens ([P3] "fast-attn 库的使用", [P4]     */
/* varlen path).  Request r owns query rows [cu_q[r], cu_q[r+1]) and keys    */
/* 0 .. k_len-1 with k_len = cu_k[r+1] - cu_k[r].  With a block table the    */
/* keys are read from the paged cache through table row r (prefix cache /    */
/* chunked prefill); without one (block_table == NULL) k_src/v_src are the   */
/* packed [total_k, Hkv, d] tensors and key j of request r is packed row     */
/* cu_k[r] + j ([P3] "一个小细节").  Causal: query i sees key j iff          */
/* j <= i + k_len - q_len.  Rows listed in row_subset (all rows when NULL)   */
/* are computed; out is [n_rows, Hq, d] in fp64.                             */
/* ------------------------------------------------------------------------ */
/* The request r with cu_q[r] <= row < cu_q[r+1] (requests with no queries are
 * passed over because their interval is empty). */
static int32_t request_of_row(const int32_t* cu_q, int32_t batch, int64_t row) {
    int32_t r = 0;
    while (r < batch - 1 && cu_q[r + 1] <= row) ++r;
    return r;
}

void ora_prefill(const void* q, const void* k_src, const void* v_src, int dtype,
                 const int32_t* cu_q, const int32_t* cu_k, int32_t batch,
                 const int32_t* block_table, int32_t max_blocks, int32_t block_size,
                 int causal, int32_t hq, int32_t hkv, int32_t d, double scale,
                 const int32_t* row_subset, int64_t n_rows_subset, double* out) {
    int64_t total_q = cu_q[batch];
    int64_t n_rows = row_subset ? n_rows_subset : total_q;
    int32_t group = hq / hkv;
    int64_t kv_dim = (int64_t)hkv * d;
    int64_t work = n_rows * hq;
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t w = 0; w < work; ++w) {
        int64_t o = w / hq;
        int32_t h = (int32_t)(w % hq);
        int64_t row = row_subset ? row_subset[o] : o;
        int32_t r = request_of_row(cu_q, batch, row);
        int64_t q_len = cu_q[r + 1] - cu_q[r];
        int64_t k_len = cu_k[r + 1] - cu_k[r];
        int64_t i = row - cu_q[r];
        int64_t visible = k_len;
        if (causal) {
            int64_t last = i + k_len - q_len; /* largest visible key index */
            visible = last + 1 < 0 ? 0 : (last + 1 > k_len ? k_len : last + 1);
        }
        int32_t kvh = h / group;
        int64_t* off = (int64_t*)malloc((size_t)(visible > 0 ? visible : 1) * sizeof(int64_t));
        for (int64_t j = 0; j < visible; ++j) {
            if (block_table) {
                const int32_t* trow = block_table + (int64_t)r * max_blocks;
                off[j] = ora_element_offset(trow, block_size, kv_dim, j) + (int64_t)kvh * d;
            } else {
                off[j] = ((int64_t)cu_k[r] + j) * kv_dim + (int64_t)kvh * d;
            }
        }
        double* qv = (double*)malloc((size_t)d * sizeof(double));
        for (int32_t t = 0; t < d; ++t) qv[t] = load_elem(q, dtype, (row * hq + h) * d + t);
        attend_one_shot(qv, k_src, v_src, dtype, off, visible, d, scale,
                        out + (o * hq + h) * d);
        free(qv);
        free(off);
    }
}

/* Request index of every packed token ([P4] varlen example: "Q request
 * index" / "K request index" rows). */
void ora_request_index(const int32_t* cu, int32_t batch, int32_t* out) {
    for (int32_t r = 0; r < batch; ++r)
        for (int32_t t = cu[r]; t < cu[r + 1]; ++t) out[t] = r;
}

/* ------------------------------------------------------------------------ */
/* Online softmax, element by element ([P2] 题目2): start at [m, l] =        */
/* [-inf, 0]; for each x: m_new = max(m, x), l = l*e^(m - m_new) +           */
/* e^(x - m_new).  The state after every element is recorded.                */
/* ------------------------------------------------------------------------ */
void ora_online_softmax_trace(const double* x, int64_t n, double* m_trace, double* l_trace) {
    double m = -INFINITY, l = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double m_new = x[j] > m ? x[j] : m;
        double corr_old = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        l = l * corr_old + exp(x[j] - m_new);
        m = m_new;
        m_trace[j] = m;
        l_trace[j] = l;
    }
}

/* ------------------------------------------------------------------------ */
/* Block-wise online attention of one query ([P1] §11.2): split the n keys   */
/* into consecutive chunks of the given lengths; per chunk b compute         */
/* m_b = max s_j, l_b = sum e^(s_j - m_b), o_b = sum e^(s_j - m_b) v_j;      */
/* merge with the boxed equation m_new = max(m, m_b),                        */
/* o_new = o e^(m - m_new) + o_b e^(m_b - m_new), l likewise; start at       */
/* m = -inf, l = 0, o = 0 (e^-inf = 0); output o / l.  K and V are dense     */
/* fp64 [n, d].  Zero-length chunks contribute nothing.                      */
/* ------------------------------------------------------------------------ */
void ora_online_attention(const double* q, const double* K, const double* V, int64_t n,
                          int32_t d, double scale, const int64_t* chunk_len, int64_t n_chunks,
                          double* out, double* m_out, double* l_out) {
    double m = -INFINITY, l = 0.0;
    double* o = (double*)calloc((size_t)d, sizeof(double));
    double* ob = (double*)calloc((size_t)d, sizeof(double));
    int64_t start = 0;
    for (int64_t c = 0; c < n_chunks; ++c) {
        int64_t len = chunk_len[c];
        if (len <= 0) continue;
        double mb = -INFINITY;
        for (int64_t j = start; j < start + len; ++j) {
            double dot = 0.0;
            for (int32_t i = 0; i < d; ++i) dot += q[i] * K[j * d + i];
            double s = scale * dot;
            if (s > mb) mb = s;
        }
        double lb = 0.0;
        for (int32_t i = 0; i < d; ++i) ob[i] = 0.0;
        for (int64_t j = start; j < start + len; ++j) {
            double dot = 0.0;
            for (int32_t i = 0; i < d; ++i) dot += q[i] * K[j * d + i];
            double p = exp(scale * dot - mb);
            lb += p;
            for (int32_t i = 0; i < d; ++i) ob[i] += p * V[j * d + i];
        }
        double m_new = mb > m ? mb : m;
        double corr_old = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        double corr_b = exp(mb - m_new);
        for (int32_t i = 0; i < d; ++i) o[i] = o[i] * corr_old + ob[i] * corr_b;
        l = l * corr_old + lb * corr_b;
        m = m_new;
        start += len;
    }
    for (int32_t i = 0; i < d; ++i) out[i] = (l > 0.0) ? o[i] / l : 0.0;
    if (m_out) *m_out = m;
    if (l_out) *l_out = l;
    free(o);
    free(ob);
}

/* ------------------------------------------------------------------------ */
/* FlashAttention tiling as taught in [P2] 题目3: Q split into row blocks of */
/* Br (outer loop), K/V into blocks of Bc (inner loop).  Per Q block keep    */
/* O (Br x d), m (Br), l (Br); for each K/V block: S = Q_i K_j^T * scale,    */
/* m_new = max(m, rowmax S), correction = e^(m - m_new), l = l*corr +        */
/* rowsum e^(S - m_new), O = O*corr + e^(S - m_new) V_j; normalise O by l    */
/* once after the inner loop.  The (m, l, correction) after every inner step */
/* is recorded into hist arrays of shape [ceil(N/Br)][ceil(N/Bc)][Br].       */
/* Non-causal; N, d small.                                                   */
/* ------------------------------------------------------------------------ */
void ora_flash_tiles(const double* Q, const double* K, const double* V, int64_t N, int32_t d,
                     int64_t Br, int64_t Bc, double scale, double* O_out, double* m_hist,
                     double* l_hist, double* corr_hist) {
    int64_t nq = (N + Br - 1) / Br, nk = (N + Bc - 1) / Bc;
    for (int64_t qi = 0; qi < nq; ++qi) {
        int64_t r0 = qi * Br, r1 = r0 + Br < N ? r0 + Br : N;
        int64_t rows = r1 - r0;
        double* O = (double*)calloc((size_t)(rows * d), sizeof(double));
        double* m = (double*)malloc((size_t)rows * sizeof(double));
        double* l = (double*)calloc((size_t)rows, sizeof(double));
        for (int64_t r = 0; r < rows; ++r) m[r] = -INFINITY;
        for (int64_t kj = 0; kj < nk; ++kj) {
            int64_t c0 = kj * Bc, c1 = c0 + Bc < N ? c0 + Bc : N;
            for (int64_t r = 0; r < rows; ++r) {
                double rowmax = -INFINITY;
                for (int64_t c = c0; c < c1; ++c) {
                    double dot = 0.0;
                    for (int32_t t = 0; t < d; ++t) dot += Q[(r0 + r) * d + t] * K[c * d + t];
                    if (scale * dot > rowmax) rowmax = scale * dot;
                }
                double m_new = rowmax > m[r] ? rowmax : m[r];
                double corr = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - m_new);
                l[r] *= corr;
                for (int32_t t = 0; t < d; ++t) O[r * d + t] *= corr;
                for (int64_t c = c0; c < c1; ++c) {
                    double dot = 0.0;
                    for (int32_t t = 0; t < d; ++t) dot += Q[(r0 + r) * d + t] * K[c * d + t];
                    double p = exp(scale * dot - m_new);
                    l[r] += p;
                    for (int32_t t = 0; t < d; ++t) O[r * d + t] += p * V[c * d + t];
                }
                m[r] = m_new;
                int64_t h = (qi * nk + kj) * Br + r;
                if (m_hist) m_hist[h] = m[r];
                if (l_hist) l_hist[h] = l[r];
                if (corr_hist) corr_hist[h] = corr;
            }
        }
        for (int64_t r = 0; r < rows; ++r)
            for (int32_t t = 0; t < d; ++t) O_out[(r0 + r) * d + t] = O[r * d + t] / l[r];
        free(O);
        free(m);
        free(l);
    }
}
