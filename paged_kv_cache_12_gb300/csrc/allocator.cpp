// Host block allocator of the paged KV cache (no GPU involved).
//
// Fixed-size blocks, a block table per sequence, a new block only when the
// token to write starts one ("PagedAttention de vLLM : comment la gestion de
// la VRAM soutient l'inference des grands modeles", deepsonar.com.cn, section
// 2.2 and section VII steps 1-2); reference counts and copy-on-write (same page,
// section 2.3); a free queue that hands out from its head and takes released
// blocks back at its tail (same page, section 2.4).  The deeplearn.tn page
// ("PagedAttention : comment optimiser la memoire GPU lors de l'inference des
// LLM", section "Un exemple concret d'allocation") walks the same rules
// through a block-size-4 example.
//
// Every entry point validates first and mutates only once the whole request
// is known to succeed, so an error leaves the allocator unchanged.

#include <cstdint>
#include <cstring>
#include <deque>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pa.h"

namespace {

struct Sequence {
    int64_t len = 0;
    std::vector<int32_t> blocks;   // logical block -> physical block
};

}  // namespace

struct pa_allocator {
    int64_t num_blocks = 0;
    int block_size = 0;
    std::deque<int32_t> free_queue;
    std::vector<int32_t> refcount;
    std::unordered_map<int64_t, Sequence> seqs;

    // Blocks a sequence needs for n more tokens: one per block boundary
    // crossed, plus one if its partial tail block is shared (copy first).
    int64_t blocks_needed(const Sequence &s, int64_t n) const {
        const int64_t bs = block_size;
        int64_t have = (s.len + bs - 1) / bs;
        int64_t want = (s.len + n + bs - 1) / bs;
        int64_t cow = (n > 0 && s.len % bs != 0 && refcount[s.blocks.back()] > 1) ? 1 : 0;
        return want - have + cow;
    }

    int32_t pop_free() {
        int32_t b = free_queue.front();
        free_queue.pop_front();
        return b;
    }
};

extern "C" {

int pa_alloc_create(int64_t num_blocks, int block_size, const int32_t *free_order,
                    pa_allocator **out) {
    if (!out || num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0)
        return PA_ERR_INVALID_ARG;
    *out = nullptr;
    pa_allocator *a = new (std::nothrow) pa_allocator();
    if (!a) return PA_ERR_STATE;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->refcount.assign((size_t)num_blocks, 0);
    if (free_order) {
        std::vector<char> seen((size_t)num_blocks, 0);
        for (int64_t i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[(size_t)b]) {
                delete a;
                return PA_ERR_INVALID_ARG;
            }
            seen[(size_t)b] = 1;
            a->free_queue.push_back(b);
        }
    } else {
        for (int64_t i = 0; i < num_blocks; ++i) a->free_queue.push_back((int32_t)i);
    }
    *out = a;
    return PA_OK;
}

int pa_alloc_destroy(pa_allocator *a) {
    if (!a) return PA_ERR_INVALID_ARG;
    delete a;
    return PA_OK;
}

int pa_alloc_add_seq(pa_allocator *a, int64_t seq_id) {
    if (!a || a->seqs.count(seq_id)) return PA_ERR_INVALID_ARG;
    a->seqs.emplace(seq_id, Sequence());
    return PA_OK;
}

int pa_alloc_append(pa_allocator *a, int num_seqs, const int64_t *seq_ids, const int32_t *counts,
                    int64_t *slots_out, int64_t *pairs_out, int pairs_capacity,
                    int *num_pairs_out) {
    if (!a || num_seqs < 0 || (num_seqs > 0 && (!seq_ids || !counts))) return PA_ERR_INVALID_ARG;
    if (num_pairs_out) *num_pairs_out = 0;
    // validate everything first
    std::vector<Sequence *> targets((size_t)num_seqs);
    std::unordered_set<int64_t> ids;
    int64_t total_tokens = 0, need = 0;
    int pairs_needed = 0;
    for (int k = 0; k < num_seqs; ++k) {
        auto it = a->seqs.find(seq_ids[k]);
        if (it == a->seqs.end() || counts[k] < 0 || !ids.insert(seq_ids[k]).second)
            return PA_ERR_INVALID_ARG;
        targets[(size_t)k] = &it->second;
        const Sequence &s = it->second;
        total_tokens += counts[k];
        need += a->blocks_needed(s, counts[k]);
        if (counts[k] > 0 && s.len % a->block_size != 0 && a->refcount[s.blocks.back()] > 1)
            ++pairs_needed;
    }
    if (total_tokens > 0 && !slots_out) return PA_ERR_INVALID_ARG;
    if (pairs_needed > 0 && (!pairs_out || pairs_capacity < pairs_needed || !num_pairs_out))
        return PA_ERR_INVALID_ARG;
    if (need > (int64_t)a->free_queue.size()) return PA_ERR_OUT_OF_BLOCKS;

    // commit
    const int64_t bs = a->block_size;
    int64_t w = 0;
    int np = 0;
    for (int k = 0; k < num_seqs; ++k) {
        Sequence &s = *targets[(size_t)k];
        for (int32_t j = 0; j < counts[k]; ++j) {
            const int64_t t = s.len;
            const int64_t off = t % bs;
            if (off == 0) {
                int32_t b = a->pop_free();
                a->refcount[(size_t)b] = 1;
                s.blocks.push_back(b);
            } else {
                int32_t tail = s.blocks.back();
                if (a->refcount[(size_t)tail] > 1) {
                    int32_t fresh = a->pop_free();
                    a->refcount[(size_t)fresh] = 1;
                    a->refcount[(size_t)tail] -= 1;
                    s.blocks.back() = fresh;
                    pairs_out[2 * np] = tail;
                    pairs_out[2 * np + 1] = fresh;
                    ++np;
                }
            }
            slots_out[w++] = (int64_t)s.blocks[(size_t)(t / bs)] * bs + off;
            s.len = t + 1;
        }
    }
    if (num_pairs_out) *num_pairs_out = np;
    return PA_OK;
}

int pa_alloc_fork(pa_allocator *a, int64_t parent_id, int64_t child_id) {
    if (!a) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(parent_id);
    if (it == a->seqs.end() || a->seqs.count(child_id)) return PA_ERR_INVALID_ARG;
    Sequence child = it->second;
    for (int32_t b : child.blocks) a->refcount[(size_t)b] += 1;
    a->seqs.emplace(child_id, std::move(child));
    return PA_OK;
}

int pa_alloc_free_seq(pa_allocator *a, int64_t seq_id) {
    if (!a) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_INVALID_ARG;
    for (int32_t b : it->second.blocks)
        if (a->refcount[(size_t)b] <= 0) return PA_ERR_STATE;
    // a block listed twice in one table would be released twice
    {
        std::unordered_map<int32_t, int> uses;
        for (int32_t b : it->second.blocks)
            if (++uses[b] > a->refcount[(size_t)b]) return PA_ERR_STATE;
    }
    for (int32_t b : it->second.blocks) {
        if (--a->refcount[(size_t)b] == 0) a->free_queue.push_back(b);
    }
    a->seqs.erase(it);
    return PA_OK;
}

int pa_alloc_seq_len(const pa_allocator *a, int64_t seq_id, int64_t *len_out) {
    if (!a || !len_out) return PA_ERR_INVALID_ARG;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_INVALID_ARG;
    *len_out = it->second.len;
    return PA_OK;
}

int pa_alloc_block_tables(const pa_allocator *a, int num_seqs, const int64_t *seq_ids,
                          int32_t *tables_out, int max_blocks, int32_t *lens_out) {
    if (!a || num_seqs < 0 || max_blocks < 0 || (num_seqs > 0 && (!seq_ids || !tables_out || !lens_out)))
        return PA_ERR_INVALID_ARG;
    for (int k = 0; k < num_seqs; ++k) {
        auto it = a->seqs.find(seq_ids[k]);
        if (it == a->seqs.end() || (int64_t)it->second.blocks.size() > max_blocks ||
            it->second.len > INT32_MAX)
            return PA_ERR_INVALID_ARG;
    }
    for (int k = 0; k < num_seqs; ++k) {
        const Sequence &s = a->seqs.find(seq_ids[k])->second;
        int32_t *row = tables_out + (int64_t)k * max_blocks;
        size_t n = s.blocks.size();
        if (n) std::memcpy(row, s.blocks.data(), n * sizeof(int32_t));
        for (int64_t j = (int64_t)n; j < max_blocks; ++j) row[j] = -1;
        lens_out[k] = (int32_t)s.len;
    }
    return PA_OK;
}

int pa_alloc_refcount(const pa_allocator *a, int64_t block, int32_t *count_out) {
    if (!a || !count_out || block < 0 || block >= a->num_blocks) return PA_ERR_INVALID_ARG;
    *count_out = a->refcount[(size_t)block];
    return PA_OK;
}

int pa_alloc_stats(const pa_allocator *a, pa_alloc_stats_t *out) {
    if (!a || !out) return PA_ERR_INVALID_ARG;
    pa_alloc_stats_t s;
    s.num_blocks = a->num_blocks;
    s.free_blocks = (int64_t)a->free_queue.size();
    s.used_blocks = 0;
    s.shared_blocks = 0;
    for (int32_t r : a->refcount) {
        if (r > 0) ++s.used_blocks;
        if (r > 1) ++s.shared_blocks;
    }
    s.num_seqs = (int64_t)a->seqs.size();
    s.logical_tokens = 0;
    for (const auto &kv : a->seqs) s.logical_tokens += kv.second.len;
    *out = s;
    return PA_OK;
}

}  // extern "C"
