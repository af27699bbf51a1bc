// pa_blocks.cpp -- host block manager of the paged KV pool with a
// content-hash prefix cache (declared in include/pa_blocks.h; sources:
// "11. 推理加速(一):vLLM 原理", §11.2 PagedAttention and §11.4 prefix caching).
//
// State: per physical block a reference count, whether it is cached
// (matchable by its prefix hash) and when it was released; a set of free
// blocks (unreferenced, not cached; lowest id first), a set of evictable
// blocks (unreferenced, cached; oldest release first) and the hash -> block
// map.  Per request: its token ids, how many of them are computed, its block
// table and the prefix hash of each computed full block.
#include <cstring>
#include <new>
#include <set>
#include <unordered_map>
#include <unordered_set>
#include <utility>
#include <vector>

#include "pa.h"
#include "pa_blocks.h"

namespace {

// 128-bit identity of a token prefix, built block by block: the hash of
// block i folds the hash of block i-1 with block i's token ids.  Two lanes
// with different constants; each step is a 64-bit finaliser of the
// xor-shift-multiply kind.
struct Hash128 {
    uint64_t a = 0, b = 0;
    bool operator==(const Hash128 &o) const { return a == o.a && b == o.b; }
};
struct Hash128Hasher {
    size_t operator()(const Hash128 &h) const {
        return static_cast<size_t>(h.a ^ (h.b * 0x9E3779B97F4A7C15ull));
    }
};

uint64_t fmix(uint64_t x) {
    x ^= x >> 31;
    x *= 0x7FB5D329728EA185ull;
    x ^= x >> 27;
    x *= 0x81DADEF4BC2DD44Dull;
    x ^= x >> 33;
    return x;
}

Hash128 chain(const Hash128 &parent, const int32_t *tokens, int32_t n) {
    uint64_t a = parent.a ^ 0x243F6A8885A308D3ull;
    uint64_t b = parent.b + 0x13198A2E03707344ull;
    for (int32_t i = 0; i < n; ++i) {
        const uint64_t x = static_cast<uint32_t>(tokens[i]);
        a = fmix(a ^ (x + 0xA4093822299F31D0ull));
        b = fmix(b + x * 0x9E3779B97F4A7C15ull + static_cast<uint64_t>(i));
    }
    Hash128 h;
    h.a = fmix(a ^ static_cast<uint64_t>(n));
    h.b = fmix(b ^ (static_cast<uint64_t>(n) << 32));
    return h;
}

struct Block {
    int32_t ref = 0;
    bool cached = false;
    Hash128 h;
    uint64_t released = 0;
};

struct Request {
    std::vector<int32_t> tokens;
    int32_t computed = 0;
    std::vector<int32_t> table;
    std::vector<Hash128> prefix;  // hash of each computed full block's prefix
};

}  // namespace

struct pa_block_manager {
    int32_t bs = 0;
    std::vector<Block> blocks;
    std::set<int32_t> free_ids;
    std::set<std::pair<uint64_t, int32_t>> evictable;
    std::unordered_map<Hash128, int32_t, Hash128Hasher> cache;
    std::unordered_map<int64_t, Request> reqs;
    uint64_t clock = 0;

    int32_t available() const {
        return static_cast<int32_t>(free_ids.size() + evictable.size());
    }

    // Caller has checked available() > 0.
    int32_t alloc() {
        int32_t b;
        if (!free_ids.empty()) {
            b = *free_ids.begin();
            free_ids.erase(free_ids.begin());
        } else {
            b = evictable.begin()->second;
            evictable.erase(evictable.begin());
            cache.erase(blocks[b].h);
            blocks[b].cached = false;
        }
        blocks[b].ref = 1;
        return b;
    }

    void take_ref(int32_t b) {
        if (blocks[b].ref == 0) evictable.erase({blocks[b].released, b});
        ++blocks[b].ref;
    }

    void release(int32_t b) {
        if (--blocks[b].ref > 0) return;
        if (blocks[b].cached) {
            blocks[b].released = ++clock;
            evictable.insert({blocks[b].released, b});
        } else {
            free_ids.insert(b);
        }
    }
};

extern "C" {

pa_block_manager *pa_bm_create(int32_t num_blocks, int32_t block_size) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pa_block_manager *bm = new (std::nothrow) pa_block_manager;
    if (!bm) return nullptr;
    try {
        bm->bs = block_size;
        bm->blocks.resize(static_cast<size_t>(num_blocks));
        for (int32_t b = 0; b < num_blocks; ++b) bm->free_ids.insert(bm->free_ids.end(), b);
    } catch (...) {
        delete bm;
        return nullptr;
    }
    return bm;
}

void pa_bm_destroy(pa_block_manager *bm) { delete bm; }

int pa_bm_add_request(pa_block_manager *bm, int64_t req_id, const int32_t *token_ids,
                      int32_t num_tokens, int32_t *num_cached_tokens) {
    if (!bm || !token_ids || num_tokens < 1 || bm->reqs.count(req_id)) return PA_ERR_INVALID_ARG;
    Request r;
    r.tokens.assign(token_ids, token_ids + num_tokens);
    // the prompt's last token is always computed: match at most the full
    // blocks that end before it
    const int32_t max_hits = (num_tokens - 1) / bm->bs;
    Hash128 h;
    for (int32_t i = 0; i < max_hits; ++i) {
        h = chain(h, token_ids + static_cast<int64_t>(i) * bm->bs, bm->bs);
        auto it = bm->cache.find(h);
        if (it == bm->cache.end()) break;
        bm->take_ref(it->second);
        r.table.push_back(it->second);
        r.prefix.push_back(h);
    }
    r.computed = static_cast<int32_t>(r.table.size()) * bm->bs;
    if (num_cached_tokens) *num_cached_tokens = r.computed;
    bm->reqs.emplace(req_id, std::move(r));
    return PA_OK;
}

int pa_bm_append_tokens(pa_block_manager *bm, int64_t req_id, const int32_t *token_ids,
                        int32_t num_tokens) {
    if (!bm || num_tokens < 0 || (num_tokens > 0 && !token_ids)) return PA_ERR_INVALID_ARG;
    auto it = bm->reqs.find(req_id);
    if (it == bm->reqs.end()) return PA_ERR_INVALID_ARG;
    it->second.tokens.insert(it->second.tokens.end(), token_ids, token_ids + num_tokens);
    return PA_OK;
}

int pa_bm_fork(pa_block_manager *bm, int64_t src_id, int64_t dst_id) {
    if (!bm || src_id == dst_id || bm->reqs.count(dst_id)) return PA_ERR_INVALID_ARG;
    auto it = bm->reqs.find(src_id);
    if (it == bm->reqs.end()) return PA_ERR_INVALID_ARG;
    Request r = it->second;
    for (int32_t b : r.table) bm->take_ref(b);
    bm->reqs.emplace(dst_id, std::move(r));
    return PA_OK;
}

int pa_bm_schedule(pa_block_manager *bm, int32_t num_reqs, const int64_t *req_ids,
                   const int32_t *num_new_tokens, int32_t max_blocks_per_seq,
                   int32_t *block_tables, int32_t *query_start_loc, int32_t *context_lens,
                   int32_t *seq_lens, int64_t *slot_mapping, int32_t max_copies,
                   int32_t *copies, int32_t *num_copies) {
    if (!bm || num_reqs < 0 || max_blocks_per_seq < 1 || max_copies < 0 || !query_start_loc)
        return PA_ERR_INVALID_ARG;
    if (num_reqs > 0 && (!req_ids || !num_new_tokens || !block_tables || !context_lens ||
                         !seq_lens || !slot_mapping))
        return PA_ERR_INVALID_ARG;
    const int32_t bs = bm->bs;
    // 1. validate everything and count the blocks needed, changing nothing
    std::vector<Request *> rs(static_cast<size_t>(num_reqs));
    std::unordered_set<int64_t> seen;
    int64_t need = 0, n_copies = 0;
    for (int32_t i = 0; i < num_reqs; ++i) {
        auto it = bm->reqs.find(req_ids[i]);
        if (it == bm->reqs.end() || !seen.insert(req_ids[i]).second || num_new_tokens[i] < 1)
            return PA_ERR_INVALID_ARG;
        Request &r = it->second;
        const int64_t end = static_cast<int64_t>(r.computed) + num_new_tokens[i];
        if (end > static_cast<int64_t>(r.tokens.size())) return PA_ERR_INVALID_ARG;
        const int64_t nblk = (end + bs - 1) / bs;
        if (nblk > max_blocks_per_seq) return PA_ERR_INVALID_ARG;
        const bool cow = r.computed % bs != 0 && bm->blocks[r.table[r.computed / bs]].ref > 1;
        need += (nblk - static_cast<int64_t>(r.table.size())) + (cow ? 1 : 0);
        n_copies += cow ? 1 : 0;
        rs[static_cast<size_t>(i)] = &r;
    }
    if (n_copies > max_copies || (n_copies > 0 && !copies)) return PA_ERR_INVALID_ARG;
    if (need > bm->available()) return PA_ERR_WORKSPACE;

    // 2. allocate, emit the metadata, advance, cache newly filled blocks
    int32_t nc = 0;
    int64_t t = 0;
    query_start_loc[0] = 0;
    for (int32_t i = 0; i < num_reqs; ++i) {
        Request &r = *rs[static_cast<size_t>(i)];
        const int32_t n = num_new_tokens[i];
        if (r.computed % bs != 0) {
            const int32_t idx = r.computed / bs;
            const int32_t old = r.table[static_cast<size_t>(idx)];
            if (bm->blocks[old].ref > 1) {  // copy-on-write
                const int32_t fresh = bm->alloc();
                copies[2 * nc] = old;
                copies[2 * nc + 1] = fresh;
                ++nc;
                bm->release(old);
                r.table[static_cast<size_t>(idx)] = fresh;
            }
        }
        const int32_t end = r.computed + n;
        while (static_cast<int64_t>(r.table.size()) * bs < end) r.table.push_back(bm->alloc());
        int32_t *row = block_tables + static_cast<int64_t>(i) * max_blocks_per_seq;
        for (int32_t j = 0; j < max_blocks_per_seq; ++j)
            row[j] = j < static_cast<int32_t>(r.table.size()) ? r.table[static_cast<size_t>(j)] : -1;
        context_lens[i] = r.computed;
        seq_lens[i] = end;
        query_start_loc[i + 1] = query_start_loc[i] + n;
        for (int32_t p = r.computed; p < end; ++p)
            slot_mapping[t++] = static_cast<int64_t>(r.table[static_cast<size_t>(p / bs)]) * bs + p % bs;
        r.computed = end;
        while (static_cast<int64_t>(r.prefix.size() + 1) * bs <= r.computed) {
            const size_t k = r.prefix.size();
            const Hash128 parent = k > 0 ? r.prefix[k - 1] : Hash128();
            const Hash128 h = chain(parent, r.tokens.data() + k * bs, bs);
            r.prefix.push_back(h);
            const int32_t blk = r.table[k];
            if (!bm->blocks[blk].cached && !bm->cache.count(h)) {
                bm->cache.emplace(h, blk);
                bm->blocks[blk].cached = true;
                bm->blocks[blk].h = h;
            }
        }
    }
    if (num_copies) *num_copies = nc;
    return PA_OK;
}

int pa_bm_free_request(pa_block_manager *bm, int64_t req_id) {
    if (!bm) return PA_ERR_INVALID_ARG;
    auto it = bm->reqs.find(req_id);
    if (it == bm->reqs.end()) return PA_ERR_INVALID_ARG;
    const std::vector<int32_t> &tab = it->second.table;
    for (size_t j = tab.size(); j-- > 0;) bm->release(tab[j]);
    bm->reqs.erase(it);
    return PA_OK;
}

int32_t pa_bm_num_free_blocks(const pa_block_manager *bm) { return bm ? bm->available() : -1; }

int32_t pa_bm_num_cached_blocks(const pa_block_manager *bm) {
    return bm ? static_cast<int32_t>(bm->cache.size()) : -1;
}

int32_t pa_bm_block_ref_count(const pa_block_manager *bm, int32_t block) {
    if (!bm || block < 0 || block >= static_cast<int32_t>(bm->blocks.size())) return -1;
    return bm->blocks[block].ref;
}

int32_t pa_bm_request_blocks(const pa_block_manager *bm, int64_t req_id, int32_t *out,
                             int32_t cap) {
    if (!bm) return -1;
    auto it = bm->reqs.find(req_id);
    if (it == bm->reqs.end()) return -1;
    const std::vector<int32_t> &tab = it->second.table;
    for (int32_t j = 0; j < cap && j < static_cast<int32_t>(tab.size()); ++j)
        out[j] = tab[static_cast<size_t>(j)];
    return static_cast<int32_t>(tab.size());
}

int32_t pa_bm_num_computed(const pa_block_manager *bm, int64_t req_id) {
    if (!bm) return -1;
    auto it = bm->reqs.find(req_id);
    return it == bm->reqs.end() ? -1 : it->second.computed;
}

}  // extern "C"
