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
// Optional prefix caching (same deepsonar page, section 2.4 and section VII
// step 5): every full block of a sequence whose token ids are known gets a
// chained hash SHA-256(parent block's hash, the block's token ids, an extra
// key), registered in a hash -> block map.  A released block keeps its content
// and its map entry while it waits in the free queue; the queue order is the
// eviction order: when a block leaves the head to be reused, its entry is
// dropped first.  A new sequence is matched block by block against the map;
// each hit is taken (out of the free queue if it was free) with its count
// raised, and the match stops at the first miss.  At least the last prompt
// token is always left to compute, so its logits exist.
//
// The free queue is an intrusive doubly linked list over block ids, so that a
// cached block can leave the middle of the queue in O(1).
//
// Every entry point validates first and mutates only once the whole request
// is known to succeed, so an error leaves the allocator unchanged.

#include <array>
#include <cstdint>
#include <cstring>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pa.h"
#include "sha256.h"

namespace {

using Hash = std::array<uint8_t, 32>;

struct HashKey {
    size_t operator()(const Hash &h) const {
        uint64_t v;
        std::memcpy(&v, h.data(), sizeof(v));
        return (size_t)v;
    }
};

struct Sequence {
    int64_t len = 0;
    std::vector<int32_t> blocks;   // logical block -> physical block
    // prefix caching: token ids while every token's id is known, the chained
    // hash of each full block, and the extra key mixed into every hash
    bool ids_known = true;
    std::vector<int32_t> ids;
    std::vector<Hash> chain;
    uint64_t extra_key = 0;
};

// Serialised hash input: parent hash (32 bytes), the block's token ids as
// little-endian int32, the extra key as little-endian uint64.
Hash block_hash(const Hash *parent, const int32_t *tokens, int n, uint64_t extra) {
    std::vector<uint8_t> buf(32 + 4 * (size_t)n + 8, 0);
    if (parent) std::memcpy(buf.data(), parent->data(), 32);
    for (int i = 0; i < n; ++i) {
        const uint32_t t = (uint32_t)tokens[i];
        for (int k = 0; k < 4; ++k) buf[32 + 4 * (size_t)i + k] = (uint8_t)(t >> (8 * k));
    }
    for (int k = 0; k < 8; ++k) buf[32 + 4 * (size_t)n + k] = (uint8_t)(extra >> (8 * k));
    Hash h;
    pa::sha256(buf.data(), buf.size(), h.data());
    return h;
}

}  // namespace

struct pa_allocator {
    int64_t num_blocks = 0;
    int block_size = 0;
    // free queue: doubly linked list over block ids
    std::vector<int32_t> prev, next;
    std::vector<char> is_free;
    int32_t head = -1, tail = -1;
    int64_t free_count = 0;
    std::vector<int32_t> refcount;
    std::unordered_map<int64_t, Sequence> seqs;
    // prefix cache
    bool prefix = false;
    std::vector<char> has_hash;
    std::vector<Hash> hash_of;
    std::unordered_map<Hash, int32_t, HashKey> cached;
    int64_t queries = 0, hits = 0;

    void push_tail(int32_t b) {
        prev[(size_t)b] = tail;
        next[(size_t)b] = -1;
        if (tail >= 0) next[(size_t)tail] = b; else head = b;
        tail = b;
        is_free[(size_t)b] = 1;
        ++free_count;
    }

    void unlink(int32_t b) {
        const int32_t p = prev[(size_t)b], n = next[(size_t)b];
        if (p >= 0) next[(size_t)p] = n; else head = n;
        if (n >= 0) prev[(size_t)n] = p; else tail = p;
        prev[(size_t)b] = next[(size_t)b] = -1;
        is_free[(size_t)b] = 0;
        --free_count;
    }

    // Take the block at the head of the free queue; a cached block's content
    // is evicted from the map first.
    int32_t pop_free() {
        const int32_t b = head;
        unlink(b);
        if (has_hash[(size_t)b]) {
            auto it = cached.find(hash_of[(size_t)b]);
            if (it != cached.end() && it->second == b) cached.erase(it);
            has_hash[(size_t)b] = 0;
        }
        return b;
    }

    // Blocks a sequence needs for n more tokens: one per block boundary
    // crossed, plus one if its partial tail block is shared (copy first).
    int64_t blocks_needed(const Sequence &s, int64_t n) const {
        const int64_t bs = block_size;
        int64_t have = (s.len + bs - 1) / bs;
        int64_t want = (s.len + n + bs - 1) / bs;
        int64_t cow = (n > 0 && s.len % bs != 0 && refcount[(size_t)s.blocks.back()] > 1) ? 1 : 0;
        return want - have + cow;
    }

    // After token t of s was written: if it completed a block and the
    // sequence's ids are known, hash the block and register it.
    void maybe_hash(Sequence &s, int64_t t) {
        const int64_t bs = block_size;
        if (!prefix || !s.ids_known || (t + 1) % bs != 0) return;
        const int64_t j = t / bs;
        if ((int64_t)s.chain.size() != j) return;   // chain broken earlier
        const Hash h = block_hash(j ? &s.chain[(size_t)j - 1] : nullptr, s.ids.data() + j * bs, (int)bs,
                                  s.extra_key);
        s.chain.push_back(h);
        const int32_t b = s.blocks[(size_t)j];
        if (!has_hash[(size_t)b]) {
            has_hash[(size_t)b] = 1;
            hash_of[(size_t)b] = h;
            cached.emplace(h, b);   // keeps an existing entry for the same content
        }
    }
};

extern "C" {

int pa_alloc_create(int64_t num_blocks, int block_size, const int32_t *free_order, pa_allocator **out) {
    if (!out || num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return PA_ERR_INVALID_ARG;
    *out = nullptr;
    pa_allocator *a = new (std::nothrow) pa_allocator();
    if (!a) return PA_ERR_STATE;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    const size_t n = (size_t)num_blocks;
    a->refcount.assign(n, 0);
    a->prev.assign(n, -1);
    a->next.assign(n, -1);
    a->is_free.assign(n, 0);
    a->has_hash.assign(n, 0);
    a->hash_of.resize(n);
    if (free_order) {
        std::vector<char> seen(n, 0);
        for (int64_t i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[(size_t)b]) {
                delete a;
                return PA_ERR_INVALID_ARG;
            }
            seen[(size_t)b] = 1;
        }
        for (int64_t i = 0; i < num_blocks; ++i) a->push_tail(free_order[i]);
    } else {
        for (int64_t i = 0; i < num_blocks; ++i) a->push_tail((int32_t)i);
    }
    *out = a;
    return PA_OK;
}

int pa_alloc_destroy(pa_allocator *a) {
    if (!a) return PA_ERR_INVALID_ARG;
    delete a;
    return PA_OK;
}

int pa_alloc_enable_prefix_cache(pa_allocator *a) {
    if (!a || !a->seqs.empty()) return PA_ERR_INVALID_ARG;
    a->prefix = true;
    return PA_OK;
}

int pa_alloc_add_seq(pa_allocator *a, int64_t seq_id) {
    if (!a || a->seqs.count(seq_id)) return PA_ERR_INVALID_ARG;
    a->seqs.emplace(seq_id, Sequence());
    return PA_OK;
}

int pa_alloc_match_prefix(pa_allocator *a, int64_t seq_id, const int32_t *tokens, int num_tokens, uint64_t extra_key,
                          int *cached_tokens_out) {
    if (!a || !a->prefix || num_tokens < 0 || (num_tokens > 0 && !tokens) || !cached_tokens_out ||
        a->seqs.count(seq_id))
        return PA_ERR_INVALID_ARG;
    const int64_t bs = a->block_size;
    // full blocks inside the first num_tokens - 1 tokens may hit: the last
    // prompt token is always computed
    const int64_t candidates = num_tokens > 0 ? (num_tokens - 1) / bs : 0;
    Sequence s;
    s.extra_key = extra_key;
    for (int64_t j = 0; j < candidates; ++j) {
        const Hash h = block_hash(j ? &s.chain[(size_t)j - 1] : nullptr, tokens + j * bs, (int)bs, extra_key);
        ++a->queries;
        auto it = a->cached.find(h);
        if (it == a->cached.end()) break;
        ++a->hits;
        const int32_t b = it->second;
        if (a->is_free[(size_t)b]) a->unlink(b);
        a->refcount[(size_t)b] += 1;
        s.blocks.push_back(b);
        s.chain.push_back(h);
        s.ids.insert(s.ids.end(), tokens + j * bs, tokens + (j + 1) * bs);
        s.len += bs;
    }
    *cached_tokens_out = (int)s.len;
    a->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
}

// Shared body of pa_alloc_append and pa_alloc_append_ids.
static int append_impl(pa_allocator *a, int num_seqs, const int64_t *seq_ids, const int32_t *counts,
                       bool with_ids, const int32_t *token_ids, int64_t *slots_out, int64_t *pairs_out,
                       int pairs_capacity, int *num_pairs_out) {
    if (!a || num_seqs < 0 || (num_seqs > 0 && (!seq_ids || !counts))) return PA_ERR_INVALID_ARG;
    if (num_pairs_out) *num_pairs_out = 0;
    std::vector<Sequence *> targets((size_t)num_seqs);
    std::unordered_set<int64_t> ids;
    int64_t total_tokens = 0, need = 0;
    int pairs_needed = 0;
    for (int k = 0; k < num_seqs; ++k) {
        auto it = a->seqs.find(seq_ids[k]);
        if (it == a->seqs.end() || counts[k] < 0 || !ids.insert(seq_ids[k]).second) return PA_ERR_INVALID_ARG;
        targets[(size_t)k] = &it->second;
        const Sequence &s = it->second;
        total_tokens += counts[k];
        need += a->blocks_needed(s, counts[k]);
        if (counts[k] > 0 && s.len % a->block_size != 0 && a->refcount[(size_t)s.blocks.back()] > 1)
            ++pairs_needed;
    }
    if (total_tokens > 0 && (!slots_out || (with_ids && !token_ids))) return PA_ERR_INVALID_ARG;
    if (pairs_needed > 0 && (!pairs_out || pairs_capacity < pairs_needed || !num_pairs_out))
        return PA_ERR_INVALID_ARG;
    if (need > a->free_count) return PA_ERR_OUT_OF_BLOCKS;

    const int64_t bs = a->block_size;
    int64_t w = 0;
    int np = 0;
    for (int k = 0; k < num_seqs; ++k) {
        Sequence &s = *targets[(size_t)k];
        if (!with_ids) {
            s.ids_known = false;
            s.ids.clear();
        }
        for (int32_t j = 0; j < counts[k]; ++j) {
            const int64_t t = s.len;
            const int64_t off = t % bs;
            if (off == 0) {
                int32_t b = a->pop_free();
                a->refcount[(size_t)b] = 1;
                s.blocks.push_back(b);
            } else {
                int32_t tl = s.blocks.back();
                if (a->refcount[(size_t)tl] > 1) {
                    int32_t fresh = a->pop_free();
                    a->refcount[(size_t)fresh] = 1;
                    a->refcount[(size_t)tl] -= 1;
                    s.blocks.back() = fresh;
                    pairs_out[2 * np] = tl;
                    pairs_out[2 * np + 1] = fresh;
                    ++np;
                }
            }
            slots_out[w] = (int64_t)s.blocks[(size_t)(t / bs)] * bs + off;
            if (with_ids && s.ids_known) s.ids.push_back(token_ids[w]);
            ++w;
            s.len = t + 1;
            a->maybe_hash(s, t);
        }
    }
    if (num_pairs_out) *num_pairs_out = np;
    return PA_OK;
}

int pa_alloc_append(pa_allocator *a, int num_seqs, const int64_t *seq_ids, const int32_t *counts,
                    int64_t *slots_out, int64_t *pairs_out, int pairs_capacity, int *num_pairs_out) {
    return append_impl(a, num_seqs, seq_ids, counts, false, nullptr, slots_out, pairs_out, pairs_capacity,
                       num_pairs_out);
}

int pa_alloc_append_ids(pa_allocator *a, int num_seqs, const int64_t *seq_ids, const int32_t *counts,
                        const int32_t *token_ids, int64_t *slots_out, int64_t *pairs_out, int pairs_capacity,
                        int *num_pairs_out) {
    return append_impl(a, num_seqs, seq_ids, counts, true, token_ids, slots_out, pairs_out, pairs_capacity,
                       num_pairs_out);
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
    {
        std::unordered_map<int32_t, int> uses;
        for (int32_t b : it->second.blocks)
            if (++uses[b] > a->refcount[(size_t)b]) return PA_ERR_STATE;
    }
    for (int32_t b : it->second.blocks) {
        if (--a->refcount[(size_t)b] == 0) a->push_tail(b);
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

int pa_alloc_block_tables(const pa_allocator *a, int num_seqs, const int64_t *seq_ids, int32_t *tables_out,
                          int max_blocks, int32_t *lens_out) {
    if (!a || num_seqs < 0 || max_blocks < 0 || (num_seqs > 0 && (!seq_ids || !tables_out || !lens_out)))
        return PA_ERR_INVALID_ARG;
    for (int k = 0; k < num_seqs; ++k) {
        auto it = a->seqs.find(seq_ids[k]);
        if (it == a->seqs.end() || (int64_t)it->second.blocks.size() > max_blocks || it->second.len > INT32_MAX)
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

int pa_alloc_free_queue(const pa_allocator *a, int32_t *blocks_out, int64_t capacity, int64_t *count_out) {
    if (!a || !count_out || (capacity > 0 && !blocks_out)) return PA_ERR_INVALID_ARG;
    *count_out = a->free_count;
    if (capacity < a->free_count) return PA_ERR_INVALID_ARG;
    int64_t i = 0;
    for (int32_t b = a->head; b >= 0; b = a->next[(size_t)b]) blocks_out[i++] = b;
    return PA_OK;
}

int pa_alloc_block_hash(const pa_allocator *a, int64_t block, uint8_t *hash_out, int *cached_out) {
    if (!a || !hash_out || !cached_out || block < 0 || block >= a->num_blocks) return PA_ERR_INVALID_ARG;
    *cached_out = 0;
    std::memset(hash_out, 0, 32);
    if (a->has_hash[(size_t)block]) {
        std::memcpy(hash_out, a->hash_of[(size_t)block].data(), 32);
        auto it = a->cached.find(a->hash_of[(size_t)block]);
        *cached_out = (it != a->cached.end() && it->second == block) ? 1 : 0;
    }
    return PA_OK;
}

int pa_alloc_prefix_stats(const pa_allocator *a, int64_t *cached_blocks, int64_t *queries, int64_t *hits) {
    if (!a || !cached_blocks || !queries || !hits) return PA_ERR_INVALID_ARG;
    *cached_blocks = (int64_t)a->cached.size();
    *queries = a->queries;
    *hits = a->hits;
    return PA_OK;
}

int pa_alloc_stats(const pa_allocator *a, pa_alloc_stats_t *out) {
    if (!a || !out) return PA_ERR_INVALID_ARG;
    pa_alloc_stats_t s;
    s.num_blocks = a->num_blocks;
    s.free_blocks = a->free_count;
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
