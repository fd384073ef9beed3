// Host-side KV block allocator behind the pa_alloc* / pa_append* / pa_fork /
// pa_free / pa_export entry points of pa.h.
//
// Rules, from the pages:
//   "LLM推理优化：vLLM PagedAttention深度解析与工程实践", section 3.2 (BlockManager):
//     the free list begins in block order, allocation takes from its front,
//     freeing appends to its back in the sequence's table order, and
//     allocate(seq, num_tokens) checks the free list before taking blocks.
//   "vLLM 深度拆解：当大模型推理学会「分页注意力」", section 3.3 (BlockSpaceManager):
//     append_slot fills the current block and takes a new one when it is full;
//     free returns all blocks; identical prefixes share physical blocks and a
//     shared block is copied only when a sharer writes into it.
// Reference counts decide when a shared block is free again; a sharer writing
// into a shared, partially filled last block takes a fresh block (front of the
// free list) and reports the (old, new) copy; the last remaining sharer writes
// in place.
//
// Automatic prefix caching (the untitled Qwen2.5-7B deployment page,
// mhpq.cn/news/468822, section 3.2; "LLM推理优化：vLLM PagedAttention深度解析与
// 工程实践", section 4.2): a full block is cached under the key (entry id of the
// previous block's content, or 0, the block's token ids), so a key names its
// whole prefix and a hit needs a token-exact, block-aligned prefix.  A prompt reuses cached blocks up to its first miss; a
// freed block keeps its entry while it waits on the free list (a hit takes it
// back off the list) and loses it when the free list hands it out again.
//
// Swap ("LLM推理优化：vLLM PagedAttention深度解析与工程实践", section 3.2: too few
// free blocks calls for swap or preemption; "vLLM推理加速深度解析：从PagedAttention
// 原理到生产部署实战", section 4: with swap space the KV cache moves to CPU
// memory): a swapped-out sequence's blocks, in table order, take host blocks
// from the front of a host free list and drop their device counts; swap-in
// takes fresh device blocks from the front of the device free list and returns
// the host blocks to the back of the host list.
#include <algorithm>
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
    std::vector<int32_t> table;  // logical block -> physical block
    int32_t length = 0;          // tokens written or reserved
    // prefix caching: token ids are known for every token (created by
    // pa_alloc_prompt and grown only by token appends)
    bool tracked = false;
    std::vector<int32_t> pending;  // token ids of the partial last block
    uint64_t chain = 0;            // entry id of the last full block's content
    bool swapped = false;          // blocks live in the host pool (`host`)
    std::vector<int32_t> host;
};

struct Key {
    uint64_t parent;
    std::vector<int32_t> tokens;
    bool operator==(const Key& o) const { return parent == o.parent && tokens == o.tokens; }
};

struct KeyHash {
    size_t operator()(const Key& k) const {
        // splitmix64 finaliser folded over the parent id and the token ids
        auto mix = [](uint64_t x) {
            x += 0x9E3779B97F4A7C15ull;
            x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
            x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
            return x ^ (x >> 31);
        };
        uint64_t h = mix(k.parent);
        for (int32_t t : k.tokens) h = mix(h ^ (uint64_t)(uint32_t)t);
        return (size_t)h;
    }
};

struct Entry {
    uint64_t id;
    int32_t block;
};

}  // namespace

struct pa_allocator {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    // free list: a doubly linked list over block ids (front = head), so that a
    // cache hit can take a freed block from anywhere in it
    std::vector<int32_t> fprev, fnext;
    std::vector<char> in_free;
    int32_t fhead = -1, ftail = -1, nfree = 0;
    std::vector<int32_t> ref;
    std::unordered_map<int64_t, Sequence> seqs;
    std::unordered_map<Key, Entry, KeyHash> cache;
    std::vector<const Key*> block_key;  // key of the entry a block holds, or null
    uint64_t next_entry = 1;
    pa_prefix_stats pstats{};
    std::deque<int32_t> host_free;  // swap space
    int32_t host_blocks = 0;
    int32_t swapped_seqs = 0;

    int64_t capacity(const Sequence& s) const { return (int64_t)s.table.size() * block_size; }

    void free_push_back(int32_t b) {
        fprev[b] = ftail;
        fnext[b] = -1;
        if (ftail >= 0) fnext[ftail] = b; else fhead = b;
        ftail = b;
        in_free[b] = 1;
        ++nfree;
    }

    void free_remove(int32_t b) {
        if (fprev[b] >= 0) fnext[fprev[b]] = fnext[b]; else fhead = fnext[b];
        if (fnext[b] >= 0) fprev[fnext[b]] = fprev[b]; else ftail = fprev[b];
        in_free[b] = 0;
        --nfree;
    }

    void evict(int32_t b) {
        if (!block_key[b]) return;
        cache.erase(cache.find(*block_key[b]));
        block_key[b] = nullptr;
        pstats.evicted += 1;
    }

    int32_t take_front() {
        const int32_t b = fhead;
        free_remove(b);
        evict(b);
        ref[b] = 1;
        return b;
    }

    // Registers `block` under (chain, tokens) unless that key is cached;
    // returns the entry id now naming this content.
    uint64_t register_block(uint64_t chain, const int32_t* tokens, int32_t block) {
        Key k{chain, std::vector<int32_t>(tokens, tokens + block_size)};
        auto it = cache.find(k);
        if (it != cache.end()) return it->second.id;
        const uint64_t id = next_entry++;
        auto ins = cache.emplace(std::move(k), Entry{id, block});
        block_key[block] = &ins.first->first;
        pstats.registered += 1;
        return id;
    }

    static void untrack(Sequence& s) {
        s.tracked = false;
        s.pending.clear();
    }

    // Records the token appended at the end of `s` (a tracked sequence) and
    // registers its block once full.
    void note_token(Sequence& s, int32_t token) {
        if (!s.tracked) return;
        s.pending.push_back(token);
        if ((int32_t)s.pending.size() == block_size) {
            const int32_t block = s.table[(s.length - 1) / block_size];
            s.chain = register_block(s.chain, s.pending.data(), block);
            s.pending.clear();
        }
    }

    // Blocks one append of `s` takes, given `ref_of(block)` as the current count.
    template <class RefOf>
    int32_t append_need(const Sequence& s, RefOf ref_of) const {
        if (s.length == capacity(s)) return 1;
        return ref_of(s.table[s.length / block_size]) > 1 ? 1 : 0;
    }

    // Performs one append whose blocks were checked; returns the slot.
    int64_t append_checked(Sequence& s, int32_t* cow_src, int32_t* cow_dst) {
        *cow_src = -1;
        *cow_dst = -1;
        const int32_t pos = s.length;
        if (pos == capacity(s)) {
            s.table.push_back(take_front());
        } else {
            int32_t& last = s.table[pos / block_size];
            if (ref[last] > 1) {
                int32_t fresh = take_front();
                ref[last] -= 1;
                *cow_src = last;
                *cow_dst = fresh;
                last = fresh;
            }
        }
        s.length = pos + 1;
        return (int64_t)s.table[pos / block_size] * block_size + pos % block_size;
    }
};

extern "C" {

PA_API pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size,
                                 const int32_t* init_free_order, pa_allocator** out) {
    if (!out || num_blocks < 0 || block_size <= 0) return PA_ERR_INVALID;
    *out = nullptr;
    pa_allocator* a = new (std::nothrow) pa_allocator();
    if (!a) return PA_ERR_OOM;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->ref.assign((size_t)num_blocks, 0);
    a->fprev.assign((size_t)num_blocks, -1);
    a->fnext.assign((size_t)num_blocks, -1);
    a->in_free.assign((size_t)num_blocks, 0);
    a->block_key.assign((size_t)num_blocks, nullptr);
    if (init_free_order) {
        std::vector<char> seen((size_t)num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            int32_t b = init_free_order[i];
            if (b < 0 || b >= num_blocks || seen[(size_t)b]) {
                delete a;
                return PA_ERR_INVALID;
            }
            seen[(size_t)b] = 1;
            a->free_push_back(b);
        }
    } else {
        for (int32_t b = 0; b < num_blocks; ++b) a->free_push_back(b);
    }
    *out = a;
    return PA_OK;
}

PA_API void pa_alloc_destroy(pa_allocator* a) { delete a; }

PA_API pa_status pa_alloc(pa_allocator* a, int64_t seq_id, int32_t num_tokens) {
    if (!a || num_tokens < 0) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    const bool fresh = (it == a->seqs.end());
    if (!fresh && it->second.swapped) return PA_ERR_INVALID;
    Sequence empty;
    const Sequence& cur = fresh ? empty : it->second;
    const int64_t held = a->capacity(cur);
    if (!fresh && num_tokens > cur.length && cur.length % a->block_size != 0 &&
        !cur.table.empty() && a->ref[cur.table.back()] > 1)
        return PA_ERR_INVALID;  // would write into a shared partial block
    int64_t need = 0;
    if (held < num_tokens) need = (num_tokens - held + a->block_size - 1) / a->block_size;
    if (need > (int64_t)a->nfree) return PA_ERR_OOM;
    Sequence& s = a->seqs[seq_id];
    for (int64_t k = 0; k < need; ++k) s.table.push_back(a->take_front());
    if (fresh || num_tokens > s.length) pa_allocator::untrack(s);  // token ids unknown
    s.length = std::max(s.length, num_tokens);
    return PA_OK;
}

PA_API pa_status pa_append_slot(pa_allocator* a, int64_t seq_id, int64_t* slot_out,
                                int32_t* cow_src, int32_t* cow_dst) {
    if (!a || !slot_out) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    if (it->second.length == INT32_MAX || it->second.swapped) return PA_ERR_INVALID;
    if (a->append_need(it->second, [&](int32_t b) { return a->ref[b]; }) > a->nfree)
        return PA_ERR_OOM;
    pa_allocator::untrack(it->second);  // token id unknown
    int32_t src, dst;
    *slot_out = a->append_checked(it->second, &src, &dst);
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
    return PA_OK;
}

namespace {

// pa_append_batch and pa_append_batch_tokens (tokens may be null).
pa_status append_batch(pa_allocator* a, const int64_t* seq_ids, const int32_t* tokens,
                       int32_t B, int64_t* slot_mapping, int32_t* cow_pairs, int32_t* num_cow) {
    if (!a || B < 0 || (B > 0 && (!seq_ids || !slot_mapping || !cow_pairs)) || !num_cow)
        return PA_ERR_INVALID;
    *num_cow = 0;
    std::vector<Sequence*> batch((size_t)B);
    std::unordered_set<int64_t> seen;
    seen.reserve((size_t)B * 2);
    for (int32_t i = 0; i < B; ++i) {
        if (!seen.insert(seq_ids[i]).second) return PA_ERR_INVALID;
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
        if (it->second.length == INT32_MAX || it->second.swapped) return PA_ERR_INVALID;
        batch[(size_t)i] = &it->second;
    }
    // Count the blocks the batch takes, following the counts it lowers as
    // earlier sharers in the batch copy away from a shared block.
    std::unordered_map<int32_t, int32_t> lowered;
    int64_t need = 0;
    for (Sequence* s : batch) {
        auto ref_of = [&](int32_t b) {
            auto f = lowered.find(b);
            return a->ref[b] - (f == lowered.end() ? 0 : f->second);
        };
        int32_t n = a->append_need(*s, ref_of);
        if (n && s->length != a->capacity(*s)) lowered[s->table[s->length / a->block_size]] += 1;
        need += n;
    }
    if (need > (int64_t)a->nfree) return PA_ERR_OOM;
    int32_t ncow = 0;
    for (int32_t i = 0; i < B; ++i) {
        int32_t src, dst;
        Sequence& s = *batch[(size_t)i];
        if (!tokens) pa_allocator::untrack(s);
        slot_mapping[i] = a->append_checked(s, &src, &dst);
        if (tokens) a->note_token(s, tokens[i]);
        if (src >= 0) {
            cow_pairs[2 * ncow] = src;
            cow_pairs[2 * ncow + 1] = dst;
            ++ncow;
        }
    }
    *num_cow = ncow;
    return PA_OK;
}

}  // namespace

PA_API pa_status pa_append_batch(pa_allocator* a, const int64_t* seq_ids, int32_t B,
                                 int64_t* slot_mapping, int32_t* cow_pairs, int32_t* num_cow) {
    return append_batch(a, seq_ids, nullptr, B, slot_mapping, cow_pairs, num_cow);
}

PA_API pa_status pa_append_batch_tokens(pa_allocator* a, const int64_t* seq_ids,
                                        const int32_t* tokens, int32_t B, int64_t* slot_mapping,
                                        int32_t* cow_pairs, int32_t* num_cow) {
    if (B > 0 && !tokens) return PA_ERR_INVALID;
    return append_batch(a, seq_ids, tokens, B, slot_mapping, cow_pairs, num_cow);
}

PA_API pa_status pa_alloc_prompt(pa_allocator* a, int64_t seq_id, const int32_t* tokens,
                                 int32_t num_tokens, int32_t* cached_tokens) {
    if (!a || num_tokens < 0 || (num_tokens > 0 && !tokens)) return PA_ERR_INVALID;
    if (a->seqs.count(seq_id)) return PA_ERR_INVALID;
    const int32_t bs = a->block_size;
    const int32_t full = num_tokens / bs;
    const int32_t blocks = (int32_t)(((int64_t)num_tokens + bs - 1) / bs);
    // walk the cached prefix, stopping at the first miss
    std::vector<int32_t> hits;
    uint64_t chain = 0;
    int32_t looked = 0;
    Key probe{0, std::vector<int32_t>((size_t)bs)};
    for (int32_t i = 0; i < full; ++i) {
        ++looked;
        probe.parent = chain;
        std::memcpy(probe.tokens.data(), tokens + (int64_t)i * bs, sizeof(int32_t) * (size_t)bs);
        auto it = a->cache.find(probe);
        if (it == a->cache.end()) break;
        chain = it->second.id;
        hits.push_back(it->second.block);
    }
    int32_t revive = 0;
    for (int32_t b : hits) revive += a->ref[b] == 0;
    if (blocks - (int32_t)hits.size() > a->nfree - revive) return PA_ERR_OOM;
    a->pstats.lookups += looked;
    a->pstats.hits += (int64_t)hits.size();
    Sequence s;
    for (int32_t b : hits) {
        if (a->ref[b] == 0) a->free_remove(b);
        a->ref[b] += 1;
        s.table.push_back(b);
    }
    for (int32_t i = (int32_t)hits.size(); i < blocks; ++i) {
        const int32_t b = a->take_front();
        s.table.push_back(b);
        if (i < full) chain = a->register_block(chain, tokens + (int64_t)i * bs, b);
    }
    s.length = num_tokens;
    s.tracked = true;
    s.pending.assign(tokens + (int64_t)full * bs, tokens + num_tokens);
    s.chain = chain;
    a->seqs.emplace(seq_id, std::move(s));
    if (cached_tokens) *cached_tokens = (int32_t)hits.size() * bs;
    return PA_OK;
}

PA_API pa_status pa_append_token(pa_allocator* a, int64_t seq_id, int32_t token,
                                 int64_t* slot_out, int32_t* cow_src, int32_t* cow_dst) {
    if (!a || !slot_out) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    if (it->second.length == INT32_MAX || it->second.swapped) return PA_ERR_INVALID;
    if (a->append_need(it->second, [&](int32_t b) { return a->ref[b]; }) > a->nfree)
        return PA_ERR_OOM;
    int32_t src, dst;
    *slot_out = a->append_checked(it->second, &src, &dst);
    a->note_token(it->second, token);
    if (cow_src) *cow_src = src;
    if (cow_dst) *cow_dst = dst;
    return PA_OK;
}

PA_API pa_status pa_prefix_stats_get(const pa_allocator* a, pa_prefix_stats* out) {
    if (!a || !out) return PA_ERR_INVALID;
    *out = a->pstats;
    out->entries = (int64_t)a->cache.size();
    int64_t cached_free = 0;
    for (int32_t b = a->fhead; b >= 0; b = a->fnext[b]) cached_free += a->block_key[b] != nullptr;
    out->cached_free = cached_free;
    return PA_OK;
}

PA_API pa_status pa_fork(pa_allocator* a, int64_t parent, int64_t child) {
    if (!a) return PA_ERR_INVALID;
    auto p = a->seqs.find(parent);
    if (p == a->seqs.end()) return PA_ERR_NOT_FOUND;
    if (a->seqs.count(child) || p->second.swapped) return PA_ERR_INVALID;
    Sequence copy = p->second;
    for (int32_t b : copy.table) a->ref[b] += 1;
    a->seqs.emplace(child, std::move(copy));
    return PA_OK;
}

PA_API pa_status pa_free(pa_allocator* a, int64_t seq_id) {
    if (!a) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    for (int32_t h : it->second.host) a->host_free.push_back(h);
    if (it->second.swapped) a->swapped_seqs -= 1;
    for (int32_t b : it->second.table)
        if (--a->ref[b] == 0) a->free_push_back(b);
    a->seqs.erase(it);
    return PA_OK;
}

PA_API pa_status pa_export(const pa_allocator* a, const int64_t* seq_ids, int32_t B,
                           int32_t max_blocks, int32_t* block_tables, int32_t* context_lens) {
    if (!a || B < 0 || max_blocks < 0 ||
        (B > 0 && (!seq_ids || !context_lens || (max_blocks > 0 && !block_tables))))
        return PA_ERR_INVALID;
    for (int32_t i = 0; i < B; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
        if ((int64_t)it->second.table.size() > max_blocks || it->second.swapped)
            return PA_ERR_INVALID;
    }
    for (int32_t i = 0; i < B; ++i) {
        const Sequence& s = a->seqs.find(seq_ids[i])->second;
        int32_t* row = block_tables + (int64_t)i * max_blocks;
        const int32_t n = (int32_t)s.table.size();
        if (n) std::memcpy(row, s.table.data(), sizeof(int32_t) * (size_t)n);
        for (int32_t j = n; j < max_blocks; ++j) row[j] = -1;
        context_lens[i] = s.length;
    }
    return PA_OK;
}

PA_API pa_status pa_seq_slots(const pa_allocator* a, int64_t seq_id, int32_t start,
                              int32_t count, int64_t* slots) {
    if (!a || start < 0 || count < 0 || (count > 0 && !slots)) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    const Sequence& s = it->second;
    if ((int64_t)start + count > a->capacity(s) || s.swapped) return PA_ERR_INVALID;
    for (int32_t t = 0; t < count; ++t) {
        const int32_t pos = start + t;
        slots[t] = (int64_t)s.table[pos / a->block_size] * a->block_size + pos % a->block_size;
    }
    return PA_OK;
}

PA_API pa_status pa_seq_info(const pa_allocator* a, int64_t seq_id, int32_t* length,
                             int32_t* num_table_blocks) {
    if (!a) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    if (length) *length = it->second.length;
    if (num_table_blocks) *num_table_blocks = (int32_t)it->second.table.size();
    return PA_OK;
}

PA_API pa_status pa_block_ref(const pa_allocator* a, int32_t block, int32_t* ref) {
    if (!a || !ref || block < 0 || block >= a->num_blocks) return PA_ERR_INVALID;
    *ref = a->ref[(size_t)block];
    return PA_OK;
}

PA_API pa_status pa_free_list(const pa_allocator* a, int32_t* out, int32_t cap, int32_t* n) {
    if (!a || !n || cap < 0) return PA_ERR_INVALID;
    *n = a->nfree;
    if (cap < *n) return PA_ERR_INVALID;
    int32_t i = 0;
    for (int32_t b = a->fhead; b >= 0; b = a->fnext[b]) out[i++] = b;
    return PA_OK;
}

PA_API pa_status pa_alloc_set_swap_pool(pa_allocator* a, int32_t num_host_blocks) {
    if (!a || a->host_blocks || num_host_blocks < 0) return PA_ERR_INVALID;
    a->host_blocks = num_host_blocks;
    a->host_free.clear();
    for (int32_t h = 0; h < num_host_blocks; ++h) a->host_free.push_back(h);
    return PA_OK;
}

PA_API pa_status pa_swap_out(pa_allocator* a, int64_t seq_id, int32_t* pairs, int32_t cap,
                             int32_t* n) {
    if (!a || !n || cap < 0) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    Sequence& s = it->second;
    const int32_t nb = (int32_t)s.table.size();
    if (s.swapped || cap < nb || (nb > 0 && !pairs)) return PA_ERR_INVALID;
    if (nb > (int32_t)a->host_free.size()) return PA_ERR_OOM;
    for (int32_t j = 0; j < nb; ++j) {
        const int32_t h = a->host_free.front();
        a->host_free.pop_front();
        pairs[2 * j] = s.table[(size_t)j];
        pairs[2 * j + 1] = h;
        s.host.push_back(h);
    }
    for (int32_t b : s.table)
        if (--a->ref[b] == 0) a->free_push_back(b);
    s.table.clear();
    s.swapped = true;
    a->swapped_seqs += 1;
    *n = nb;
    return PA_OK;
}

PA_API pa_status pa_swap_in(pa_allocator* a, int64_t seq_id, int32_t* pairs, int32_t cap,
                            int32_t* n) {
    if (!a || !n || cap < 0) return PA_ERR_INVALID;
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NOT_FOUND;
    Sequence& s = it->second;
    const int32_t nb = (int32_t)s.host.size();
    if (!s.swapped || cap < nb || (nb > 0 && !pairs)) return PA_ERR_INVALID;
    if (nb > a->nfree) return PA_ERR_OOM;
    for (int32_t j = 0; j < nb; ++j) {
        const int32_t b = a->take_front();
        pairs[2 * j] = s.host[(size_t)j];
        pairs[2 * j + 1] = b;
        s.table.push_back(b);
    }
    for (int32_t h : s.host) a->host_free.push_back(h);
    s.host.clear();
    s.swapped = false;
    a->swapped_seqs -= 1;
    *n = nb;
    return PA_OK;
}

PA_API pa_status pa_swap_stats_get(const pa_allocator* a, pa_swap_stats* out) {
    if (!a || !out) return PA_ERR_INVALID;
    out->host_blocks = a->host_blocks;
    out->host_free = (int32_t)a->host_free.size();
    out->swapped_seqs = a->swapped_seqs;
    return PA_OK;
}

PA_API pa_status pa_host_free_list(const pa_allocator* a, int32_t* out, int32_t cap,
                                   int32_t* n) {
    if (!a || !n || cap < 0) return PA_ERR_INVALID;
    *n = (int32_t)a->host_free.size();
    if (cap < *n) return PA_ERR_INVALID;
    int32_t i = 0;
    for (int32_t h : a->host_free) out[i++] = h;
    return PA_OK;
}

PA_API pa_status pa_alloc_stats_get(const pa_allocator* a, pa_alloc_stats* out) {
    if (!a || !out) return PA_ERR_INVALID;
    out->num_blocks = a->num_blocks;
    out->block_size = a->block_size;
    out->free_blocks = a->nfree;
    int32_t used = 0, shared = 0;
    for (int32_t r : a->ref) {
        used += r > 0;
        shared += r > 1;
    }
    out->used_blocks = used;
    out->shared_blocks = shared;
    out->num_seqs = (int32_t)a->seqs.size();
    int64_t tokens = 0;
    for (const auto& kv : a->seqs) tokens += kv.second.length;
    out->num_tokens = tokens;
    return PA_OK;
}

}  // extern "C"
