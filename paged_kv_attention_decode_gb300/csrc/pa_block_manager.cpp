// Host block manager of the paged KV cache: free list, allocate_slots,
// chained prefix keys with reference counts, copy-on-write, truncation.
// The semantics are stated in include/pa_block_manager.h.
#include "pa_block_manager.h"

#include <algorithm>
#include <cstring>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

namespace {

// FNV-1a, 64-bit (Fowler, Noll, Vo): the bucket index of a prefix key.  Keys
// are compared in full, so the hash only needs to spread them.
struct Fnv1a {
    size_t operator()(const std::string& s) const {
        uint64_t h = 1469598103934665603ull;
        for (unsigned char c : s) {
            h ^= c;
            h *= 1099511628211ull;
        }
        return static_cast<size_t>(h);
    }
};

struct BlockInfo {
    int32_t ref = 0;
    uint64_t reg = 0;      // registration id of the key it holds (0 = none)
    std::string key;       // that key (empty when reg == 0)
    int32_t prev = -1;     // free-list links (valid while in_free)
    int32_t next = -1;
    bool in_free = false;
};

struct Sequence {
    uint64_t extra = 0;
    std::vector<int32_t> tokens;   // every known token id
    std::vector<int32_t> blocks;   // physical block of each logical block
    std::vector<uint64_t> chain;   // registration id that continues the key chain after each full block
    int32_t len = 0;               // tokens with slots
};

}  // namespace

struct pa_block_manager {
    int32_t bs = 16;
    bool caching = true;
    std::vector<BlockInfo> blocks;
    int32_t head = -1, tail = -1, nfree = 0;
    std::unordered_map<std::string, int32_t, Fnv1a> cached;   // key -> block holding it
    std::unordered_map<int64_t, Sequence> seqs;
    uint64_t next_reg = 1;

    // ---- free list -------------------------------------------------------
    void push_back(int32_t b) {
        BlockInfo& x = blocks[b];
        x.prev = tail;
        x.next = -1;
        x.in_free = true;
        if (tail >= 0) blocks[tail].next = b; else head = b;
        tail = b;
        ++nfree;
    }
    void unlink(int32_t b) {
        BlockInfo& x = blocks[b];
        if (x.prev >= 0) blocks[x.prev].next = x.next; else head = x.next;
        if (x.next >= 0) blocks[x.next].prev = x.prev; else tail = x.prev;
        x.prev = x.next = -1;
        x.in_free = false;
        --nfree;
    }
    // the least recently freed block; a key it still holds is evicted
    int32_t pop_front() {
        const int32_t b = head;
        unlink(b);
        unregister(b);
        blocks[b].ref = 1;
        return b;
    }

    // ---- prefix keys -----------------------------------------------------
    std::string make_key(uint64_t parent, uint64_t extra, const int32_t* toks) const {
        std::string k(16 + 4 * static_cast<size_t>(bs), '\0');
        std::memcpy(&k[0], &parent, 8);
        std::memcpy(&k[8], &extra, 8);
        std::memcpy(&k[16], toks, 4 * static_cast<size_t>(bs));
        return k;
    }
    void unregister(int32_t b) {
        BlockInfo& x = blocks[b];
        if (!x.reg) return;
        auto it = cached.find(x.key);
        if (it != cached.end() && it->second == b) cached.erase(it);
        x.reg = 0;
        x.key.clear();
    }
    // the key of logical block j of s (the chain before it must be known)
    std::string key_of(const Sequence& s, size_t j) const {
        const uint64_t parent = j == 0 ? 0 : s.chain[j - 1];
        return make_key(parent, j == 0 ? s.extra : 0, s.tokens.data() + j * bs);
    }
    // register the blocks of s that are full but not yet in its chain
    void register_full(Sequence& s) {
        if (!caching) return;
        const size_t full = static_cast<size_t>(s.len / bs);
        while (s.chain.size() < full) {
            const size_t j = s.chain.size();
            std::string k = key_of(s, j);
            auto it = cached.find(k);
            if (it != cached.end()) {
                // identical content is already cached under another block:
                // continue the chain through that registration
                s.chain.push_back(blocks[it->second].reg);
                continue;
            }
            const int32_t b = s.blocks[j];
            BlockInfo& x = blocks[b];
            if (x.reg) {
                // a shared block holds the key of other content (no path of
                // this manager leads here): leave it alone and continue the
                // chain with an id that no lookup can produce
                s.chain.push_back(next_reg++);
                continue;
            }
            x.reg = next_reg++;
            x.key = k;
            cached.emplace(std::move(k), b);
            s.chain.push_back(x.reg);
        }
    }

    void release(int32_t b) {
        if (--blocks[b].ref == 0) push_back(b);   // keeps its key until evicted
    }

    Sequence* find(int64_t id) {
        auto it = seqs.find(id);
        return it == seqs.end() ? nullptr : &it->second;
    }
    const Sequence* find(int64_t id) const {
        auto it = seqs.find(id);
        return it == seqs.end() ? nullptr : &it->second;
    }
};

extern "C" {

pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size, int32_t prefix_caching) {
    if (num_blocks <= 0 || block_size <= 0 || block_size > 4096) return nullptr;
    pa_block_manager* bm = new (std::nothrow) pa_block_manager;
    if (!bm) return nullptr;
    try {
        bm->bs = block_size;
        bm->caching = prefix_caching != 0;
        bm->blocks.resize(static_cast<size_t>(num_blocks));
        for (int32_t b = 0; b < num_blocks; ++b) bm->push_back(b);
    } catch (...) {
        delete bm;
        return nullptr;
    }
    return bm;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int32_t pa_bm_num_free_blocks(const pa_block_manager* bm) { return bm ? bm->nfree : -1; }

int pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, uint64_t extra_key, const int32_t* prompt,
                       int32_t prompt_len, int32_t* num_cached_tokens) {
    if (!bm || prompt_len < 0 || (prompt_len > 0 && !prompt) || !num_cached_tokens) return PA_BM_ERR_INVALID_ARG;
    if (bm->find(seq_id)) return PA_BM_ERR_INVALID_ARG;
    Sequence* s = nullptr;
    try {
        Sequence fresh;
        fresh.extra = extra_key;
        fresh.tokens.assign(prompt, prompt + prompt_len);
        // full blocks strictly before the one holding the last prompt token
        const size_t limit = bm->caching && prompt_len > 0 ? static_cast<size_t>((prompt_len - 1) / bm->bs) : 0;
        fresh.blocks.reserve(limit);
        fresh.chain.reserve(limit);
        for (size_t j = 0; j < limit; ++j) {
            auto it = bm->cached.find(bm->key_of(fresh, j));
            if (it == bm->cached.end()) break;
            fresh.blocks.push_back(it->second);
            fresh.chain.push_back(bm->blocks[it->second].reg);
        }
        s = &bm->seqs.emplace(seq_id, std::move(fresh)).first->second;
    } catch (...) {
        return PA_BM_ERR_NO_SPACE;
    }
    // the hits are shared from here on (nothing below can fail)
    for (int32_t b : s->blocks) {
        BlockInfo& x = bm->blocks[b];
        if (x.in_free) bm->unlink(b);   // a cached block with no holder comes back
        ++x.ref;
    }
    s->len = static_cast<int32_t>(s->blocks.size()) * bm->bs;
    *num_cached_tokens = s->len;
    return PA_BM_OK;
}

int pa_bm_append_tokens(pa_block_manager* bm, int64_t seq_id, const int32_t* token_ids, int32_t n) {
    if (!bm || n < 0 || (n > 0 && !token_ids)) return PA_BM_ERR_INVALID_ARG;
    Sequence* s = bm->find(seq_id);
    if (!s) return PA_BM_ERR_INVALID_ARG;
    if (static_cast<int64_t>(s->tokens.size()) + n > INT32_MAX) return PA_BM_ERR_INVALID_ARG;
    s->tokens.insert(s->tokens.end(), token_ids, token_ids + n);
    return PA_BM_OK;
}

int pa_bm_allocate_slots(pa_block_manager* bm, int64_t seq_id, int32_t num_new, int32_t* cow_src,
                         int32_t* cow_dst, int32_t* num_cow) {
    if (!bm || num_new < 0 || !cow_src || !cow_dst || !num_cow) return PA_BM_ERR_INVALID_ARG;
    Sequence* s = bm->find(seq_id);
    if (!s) return PA_BM_ERR_INVALID_ARG;
    const int64_t new_len = static_cast<int64_t>(s->len) + num_new;
    if (new_len > static_cast<int64_t>(s->tokens.size())) return PA_BM_ERR_INVALID_ARG;   // unknown tokens
    *num_cow = 0;
    if (num_new == 0) return PA_BM_OK;
    const int64_t have = static_cast<int64_t>(s->blocks.size());
    const int64_t want = (new_len + bm->bs - 1) / bm->bs;
    // the partial last block is written now: a shared one is copied first
    const bool cow = s->len % bm->bs != 0 && bm->blocks[s->blocks.back()].ref > 1;
    const int64_t need = (want - have) + (cow ? 1 : 0);
    if (need > bm->nfree) return PA_BM_ERR_NO_SPACE;
    try {
        s->blocks.reserve(static_cast<size_t>(want));
        s->chain.reserve(static_cast<size_t>(new_len / bm->bs));
    } catch (...) {
        return PA_BM_ERR_NO_SPACE;
    }
    if (cow) {
        const int32_t old = s->blocks.back();
        const int32_t fresh = bm->pop_front();
        --bm->blocks[old].ref;   // still > 0: another holder keeps it
        s->blocks.back() = fresh;
        *cow_src = old;
        *cow_dst = fresh;
        *num_cow = 1;
    }
    for (int64_t j = have; j < want; ++j) s->blocks.push_back(bm->pop_front());
    s->len = static_cast<int32_t>(new_len);
    bm->register_full(*s);
    return PA_BM_OK;
}

int pa_bm_truncate(pa_block_manager* bm, int64_t seq_id, int32_t new_len) {
    if (!bm || new_len < 0) return PA_BM_ERR_INVALID_ARG;
    Sequence* s = bm->find(seq_id);
    if (!s || new_len > s->len) return PA_BM_ERR_INVALID_ARG;
    const size_t keep = static_cast<size_t>((new_len + bm->bs - 1) / bm->bs);
    while (s->blocks.size() > keep) {
        bm->release(s->blocks.back());
        s->blocks.pop_back();
    }
    if (new_len % bm->bs != 0) {
        // the new last block will be written again from offset new_len % bs:
        // a key that describes its old full content must go, unless another
        // holder still needs that content (then the next write copies it)
        const int32_t b = s->blocks.back();
        if (bm->blocks[b].ref == 1) bm->unregister(b);
    }
    s->chain.resize(std::min(s->chain.size(), static_cast<size_t>(new_len / bm->bs)));
    s->tokens.resize(static_cast<size_t>(new_len));
    s->len = new_len;
    return PA_BM_OK;
}

int pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id) {
    if (!bm || parent_id == child_id) return PA_BM_ERR_INVALID_ARG;
    const Sequence* p = bm->find(parent_id);
    if (!p || bm->find(child_id)) return PA_BM_ERR_INVALID_ARG;
    try {
        Sequence c = *p;
        for (int32_t b : c.blocks) ++bm->blocks[b].ref;
        bm->seqs.emplace(child_id, std::move(c));
    } catch (...) {
        return PA_BM_ERR_NO_SPACE;
    }
    return PA_BM_OK;
}

int pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id) {
    if (!bm) return PA_BM_ERR_INVALID_ARG;
    auto it = bm->seqs.find(seq_id);
    if (it == bm->seqs.end()) return PA_BM_ERR_INVALID_ARG;
    const std::vector<int32_t>& blocks = it->second.blocks;
    for (auto r = blocks.rbegin(); r != blocks.rend(); ++r) bm->release(*r);
    bm->seqs.erase(it);
    return PA_BM_OK;
}

int32_t pa_bm_seq_len(const pa_block_manager* bm, int64_t seq_id) {
    const Sequence* s = bm ? bm->find(seq_id) : nullptr;
    return s ? s->len : -1;
}

int32_t pa_bm_block_table(const pa_block_manager* bm, int64_t seq_id, int32_t* out, int32_t cap) {
    const Sequence* s = bm ? bm->find(seq_id) : nullptr;
    if (!s) return -1;
    const int32_t n = static_cast<int32_t>(s->blocks.size());
    if (n > cap || (n > 0 && !out)) return -1;
    std::copy(s->blocks.begin(), s->blocks.end(), out);
    return n;
}

int32_t pa_bm_block_ref(const pa_block_manager* bm, int32_t block) {
    if (!bm || block < 0 || block >= static_cast<int32_t>(bm->blocks.size())) return -1;
    return bm->blocks[block].ref;
}

int32_t pa_bm_block_cached(const pa_block_manager* bm, int32_t block) {
    if (!bm || block < 0 || block >= static_cast<int32_t>(bm->blocks.size())) return -1;
    return bm->blocks[block].reg != 0;
}

int pa_bm_build_step(const pa_block_manager* bm, const int64_t* seq_ids, const int32_t* q_lens, int32_t num_seqs,
                     int32_t* block_tables, int32_t max_blocks, int32_t* seq_lens, int32_t* cu_q_lens,
                     int64_t* slot_mapping, int64_t slot_capacity) {
    if (!bm || num_seqs < 0 || max_blocks <= 0 || slot_capacity < 0) return PA_BM_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!seq_ids || !q_lens || !block_tables || !seq_lens)) return PA_BM_ERR_INVALID_ARG;
    if (!cu_q_lens) return PA_BM_ERR_INVALID_ARG;
    // validate everything before writing anything
    int64_t total = 0;
    for (int32_t i = 0; i < num_seqs; ++i) {
        const Sequence* s = bm->find(seq_ids[i]);
        if (!s || q_lens[i] < 1 || q_lens[i] > s->len) return PA_BM_ERR_INVALID_ARG;
        if (static_cast<int64_t>(s->blocks.size()) > max_blocks) return PA_BM_ERR_CAPACITY;
        total += q_lens[i];
    }
    if (total > slot_capacity || total > INT32_MAX) return PA_BM_ERR_CAPACITY;
    if (total > 0 && !slot_mapping) return PA_BM_ERR_INVALID_ARG;
    int64_t t = 0;
    cu_q_lens[0] = 0;
    for (int32_t i = 0; i < num_seqs; ++i) {
        const Sequence& s = *bm->find(seq_ids[i]);
        int32_t* row = block_tables + static_cast<int64_t>(i) * max_blocks;
        std::fill(row, row + max_blocks, -1);
        std::copy(s.blocks.begin(), s.blocks.end(), row);
        seq_lens[i] = s.len;
        for (int32_t pos = s.len - q_lens[i]; pos < s.len; ++pos)
            slot_mapping[t++] = static_cast<int64_t>(s.blocks[pos / bm->bs]) * bm->bs + pos % bm->bs;
        cu_q_lens[i + 1] = static_cast<int32_t>(t);
    }
    return PA_BM_OK;
}

}  // extern "C"
