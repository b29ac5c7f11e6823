// block_manager.cu -- host-side block manager of the paged KV cache: reference
// counts, the free stack, prefix sharing of full blocks and copy-on-write.
//
// "11. Paged attention 与 online softmax" §11.3: sequences with a common
// prefix point at the same physical blocks, which are then read-only; a write
// into a shared block first takes a new block and copies the old contents.
// refs[p] counts the holders of block p (allocation 1, sharing +1, release -1);
// a block returns to the free stack only when its count reaches 0.
// "结合nanovllm的FlashAttention和PagedAttention主要原理概述" 题目6: a full
// block's content hash is chained from the previous block's; a hit shares the
// cached block (count +1), a miss allocates; a finished sequence is released
// in reverse block order and a block whose count reaches 0 leaves the cache.
//
// The chained hash is kept exact: a cache key is (physical block of the
// previous block or -1, the block's B token ids), compared in full, so two
// blocks are shared only when their whole prefixes are equal.  Only full
// blocks are cached.  Free blocks form a stack whose top is block 0 at start.
// Host code only: no CUDA call is made here (the block copies a
// copy-on-write needs are paged_copy_blocks).
#include <algorithm>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pagedkv.h"

namespace {

struct Key {
    int32_t parent;
    std::vector<int64_t> tokens;
    bool operator==(const Key& o) const { return parent == o.parent && tokens == o.tokens; }
};

struct KeyHash {
    size_t operator()(const Key& k) const {
        // 64-bit mix of the parent and every token (any hash serves: keys are
        // compared in full)
        uint64_t h = 0x9E3779B97F4A7C15ull ^ (uint64_t)(uint32_t)k.parent;
        for (int64_t t : k.tokens) {
            h ^= (uint64_t)t + 0x9E3779B97F4A7C15ull + (h << 6) + (h >> 2);
            h *= 0xBF58476D1CE4E5B9ull;
        }
        return (size_t)(h ^ (h >> 31));
    }
};

struct Seq {
    std::vector<int32_t> table;
    std::vector<int64_t> tokens;
};

}  // namespace

struct pkv_block_manager {
    int32_t B = 1;
    std::vector<int32_t> ref;
    std::vector<int32_t> free_stack;  // back() is the top
    std::unordered_map<Key, int32_t, KeyHash> cache;
    std::vector<Key> key_of;     // cache key of a cached block
    std::vector<char> keyed;     // block is in the cache
    std::unordered_map<int64_t, Seq> seqs;
    int64_t next_seq = 0;

    int32_t take() {
        const int32_t b = free_stack.back();
        free_stack.pop_back();
        ref[b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--ref[b] == 0) {
            if (keyed[b]) {
                cache.erase(key_of[b]);
                keyed[b] = 0;
                key_of[b].tokens.clear();
            }
            free_stack.push_back(b);
        }
    }
    void enter(int32_t b, Key&& k) {
        Key copy = k;
        if (cache.emplace(std::move(k), b).second) {
            key_of[b] = std::move(copy);
            keyed[b] = 1;
        }
    }
};

extern "C" {

int paged_bm_create(int64_t num_blocks, int32_t block_size, pkv_block_manager** out) {
    if (!out || num_blocks < 0 || num_blocks > 0x7fffffffLL || block_size < 1)
        return PKV_ERR_INVALID;
    pkv_block_manager* bm = new (std::nothrow) pkv_block_manager;
    if (!bm) return PKV_ERR_NO_SPACE;
    bm->B = block_size;
    bm->ref.assign((size_t)num_blocks, 0);
    bm->key_of.resize((size_t)num_blocks);
    bm->keyed.assign((size_t)num_blocks, 0);
    bm->free_stack.resize((size_t)num_blocks);
    for (int64_t i = 0; i < num_blocks; ++i)
        bm->free_stack[(size_t)i] = (int32_t)(num_blocks - 1 - i);
    *out = bm;
    return PKV_OK;
}

int paged_bm_destroy(pkv_block_manager* bm) {
    delete bm;
    return PKV_OK;
}

int paged_bm_allocate(pkv_block_manager* bm, const int64_t* tokens, int64_t n_tokens,
                      int64_t* seq_out, int64_t* cached_tokens_out) {
    if (!bm || !seq_out || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PKV_ERR_INVALID;
    const int64_t B = bm->B;
    const int64_t nblk = (n_tokens + B - 1) / B;
    // count the misses first so that a shortage changes nothing
    Key key;
    key.parent = -1;
    int64_t misses = 0;
    for (int64_t i = 0; i < nblk; ++i) {
        const int64_t lo = i * B, hi = std::min(n_tokens, lo + B);
        if (hi - lo < B) { misses = nblk - i; break; }
        key.tokens.assign(tokens + lo, tokens + hi);
        auto it = bm->cache.find(key);
        if (it == bm->cache.end()) { misses = nblk - i; break; }
        key.parent = it->second;
    }
    if (misses > (int64_t)bm->free_stack.size()) return PKV_ERR_NO_SPACE;
    Seq s;
    s.tokens.assign(tokens, tokens + n_tokens);
    s.table.reserve((size_t)nblk);
    int64_t cached = 0;
    int32_t parent = -1;
    for (int64_t i = 0; i < nblk; ++i) {
        const int64_t lo = i * B, hi = std::min(n_tokens, lo + B);
        int32_t b = -1;
        Key k;
        const bool full = hi - lo == B;
        if (full) {
            k.parent = parent;
            k.tokens.assign(tokens + lo, tokens + hi);
            auto it = bm->cache.find(k);
            if (it != bm->cache.end()) b = it->second;
        }
        if (b >= 0) {
            ++bm->ref[b];  // shared: one more reference
            cached += B;
        } else {
            b = bm->take();
            if (full) bm->enter(b, std::move(k));
        }
        s.table.push_back(b);
        parent = b;
    }
    const int64_t id = bm->next_seq++;
    bm->seqs.emplace(id, std::move(s));
    *seq_out = id;
    if (cached_tokens_out) *cached_tokens_out = cached;
    return PKV_OK;
}

int paged_bm_fork(pkv_block_manager* bm, int64_t seq, int64_t* child_out) {
    if (!bm || !child_out) return PKV_ERR_INVALID;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID;
    Seq c = it->second;
    for (int32_t b : c.table) ++bm->ref[b];
    const int64_t id = bm->next_seq++;
    bm->seqs.emplace(id, std::move(c));
    *child_out = id;
    return PKV_OK;
}

int paged_bm_append(pkv_block_manager* bm, int64_t seq, int64_t token, int32_t* cow_src_out,
                    int32_t* cow_dst_out) {
    if (!bm || !cow_src_out || !cow_dst_out) return PKV_ERR_INVALID;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID;
    Seq& s = it->second;
    const int64_t B = bm->B, L = (int64_t)s.tokens.size();
    int32_t src = -1, dst = -1;
    if (L % B == 0) {
        if (bm->free_stack.empty()) return PKV_ERR_NO_SPACE;
        s.table.push_back(bm->take());
    } else {
        const int32_t last = s.table.back();
        if (bm->ref[last] > 1) {  // shared partial block: copy on write
            if (bm->free_stack.empty()) return PKV_ERR_NO_SPACE;
            const int32_t nb = bm->take();
            bm->release(last);
            s.table.back() = nb;
            src = last;
            dst = nb;
        }
    }
    s.tokens.push_back(token);
    if ((L + 1) % B == 0) {  // the last block just filled: cache it
        Key k;
        k.parent = s.table.size() >= 2 ? s.table[s.table.size() - 2] : -1;
        k.tokens.assign(s.tokens.end() - B, s.tokens.end());
        const int32_t b = s.table.back();
        if (!bm->keyed[b] && bm->cache.find(k) == bm->cache.end()) bm->enter(b, std::move(k));
    }
    *cow_src_out = src;
    *cow_dst_out = dst;
    return PKV_OK;
}

int paged_bm_free(pkv_block_manager* bm, int64_t seq) {
    if (!bm) return PKV_ERR_INVALID;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID;
    const std::vector<int32_t>& t = it->second.table;
    for (size_t i = t.size(); i-- > 0;) bm->release(t[i]);
    bm->seqs.erase(it);
    return PKV_OK;
}

int paged_bm_block_table(const pkv_block_manager* bm, int64_t seq, int32_t* table_out,
                         int32_t capacity, int32_t* n_blocks_out) {
    if (!bm || !n_blocks_out || capacity < 0) return PKV_ERR_INVALID;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID;
    const std::vector<int32_t>& t = it->second.table;
    *n_blocks_out = (int32_t)t.size();
    if ((int64_t)t.size() > capacity || (!t.empty() && !table_out)) return PKV_ERR_INVALID;
    if (!t.empty()) std::memcpy(table_out, t.data(), t.size() * sizeof(int32_t));
    return PKV_OK;
}

int paged_bm_seq_len(const pkv_block_manager* bm, int64_t seq, int64_t* len_out) {
    if (!bm || !len_out) return PKV_ERR_INVALID;
    auto it = bm->seqs.find(seq);
    if (it == bm->seqs.end()) return PKV_ERR_INVALID;
    *len_out = (int64_t)it->second.tokens.size();
    return PKV_OK;
}

int paged_bm_ref_count(const pkv_block_manager* bm, int32_t block, int32_t* ref_out) {
    if (!bm || !ref_out || block < 0 || (size_t)block >= bm->ref.size()) return PKV_ERR_INVALID;
    *ref_out = bm->ref[(size_t)block];
    return PKV_OK;
}

int paged_bm_free_blocks(const pkv_block_manager* bm, int32_t* stack_out, int64_t capacity,
                         int64_t* n_out) {
    if (!bm || !n_out || capacity < 0) return PKV_ERR_INVALID;
    const std::vector<int32_t>& f = bm->free_stack;
    *n_out = (int64_t)f.size();
    if (!stack_out) return PKV_OK;  // count only
    if ((int64_t)f.size() > capacity) return PKV_ERR_INVALID;
    if (!f.empty()) std::memcpy(stack_out, f.data(), f.size() * sizeof(int32_t));
    return PKV_OK;
}

}  // extern "C"
