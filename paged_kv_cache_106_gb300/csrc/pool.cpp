// Host-side block manager of the paged KV cache: a fixed pool of physical
// blocks, a FIFO free-block queue, a reference count per physical block and
// one block table per sequence, with fork / append / free and copy-on-write
// of a shared, partly filled last block.
//
// Steps follow the pages:
//  - pool sized once, blocks taken from the head of a free queue (vLLM
//    teardown, arcyou.ai, "PagedAttention" section; vLLM paper review,
//    mz-moonzoo.tistory.com/116, §4.2);
//  - on-demand growth: a prompt of n tokens takes ceil(n/B) blocks; a new
//    token fills the last block's free slot, else a new block is appended
//    (review §4.3 decoding example; KV cache management and PagedAttention
//    tutorial, llm-systems-engineering.pages.dev, Fig. 1-3);
//  - slot of position p: table[p / B] * B + p % B (tutorial, Fig. 2);
//  - copy-on-write on a shared partly filled last block, a shared full block
//    is never copied, the last holder writes in place (tutorial, Fig. 5-6;
//    PagedAttention notes, unpurerationalist.github.io, §3.4.1);
//  - free drops one reference per block and returns blocks at count 0, tail
//    blocks first (tutorial, "returning blocks"; notes §3.4.2, §4.2;
//    teardown, "when blocks run out");
//  - an allocation the queue cannot cover fails with no change (teardown:
//    allocate_slots returns None).
//
// A sequence's #filled is kept as its token count: every table entry but
// the last holds B tokens, the last holds num_tokens - (entries - 1) * B.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstring>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pa_internal.h"

namespace {

struct Seq {
    std::vector<int32_t> table;
    int32_t num_tokens = 0;
    uint64_t stamp = 0;   // the batched call that last listed it (duplicate check)
    uint64_t tver = 0;    // table version: a new value at every change of the table
};

// Table versions, unique in the process (a sequence keeps its version when
// it moves between pools); 0 is never handed out.
std::atomic<uint64_t> g_table_version{0};
uint64_t next_table_version() { return ++g_table_version; }

}  // namespace

struct pa_pool {
    int32_t num_blocks = 0;
    int32_t block_size = 1;
    pa_pool_desc desc{};
    bool caching = false;
    // FIFO free queue as a doubly linked list over block ids (-1 = none), so
    // that a cached free block can leave the middle of the queue when a new
    // request reuses it.
    std::vector<int32_t> nxt, prv;
    std::vector<char> in_queue;
    int32_t head = -1, tail = -1;
    int64_t count = 0;
    std::vector<int32_t> ref;
    std::unordered_map<int32_t, Seq> seqs;
    // Scratch of the batched appends, kept between calls so that a call
    // allocates nothing: a call number for the duplicate check, reference
    // decrements planned per block (zero between calls) and the blocks they
    // touched, the sequences of the call.
    uint64_t epoch = 0;
    std::vector<int32_t> plan_dec;
    std::vector<int32_t> plan_touched;
    std::vector<Seq *> plan_seqs;
    std::vector<int32_t> beam_row;   // pa_beam_prune: a group's new beams
    // Prefix cache: full prompt blocks keyed by a hash chain over
    // (parent key, the block's token ids, extra key).  Per block: its key,
    // its parent's key, the extra key and its token ids, to verify a hit.
    std::unordered_map<uint64_t, int32_t> cache;
    std::vector<char> cached;
    std::vector<uint64_t> key, parent_key;
    std::vector<int64_t> extra;
    std::vector<int32_t> tokens;   // [num_blocks][block_size]

    void queue_push_tail(int32_t b) {
        prv[(size_t)b] = tail;
        nxt[(size_t)b] = -1;
        if (tail >= 0) nxt[(size_t)tail] = b; else head = b;
        tail = b;
        in_queue[(size_t)b] = 1;
        ++count;
    }
    void queue_remove(int32_t b) {
        const int32_t p = prv[(size_t)b], n = nxt[(size_t)b];
        if (p >= 0) nxt[(size_t)p] = n; else head = n;
        if (n >= 0) prv[(size_t)n] = p; else tail = p;
        in_queue[(size_t)b] = 0;
        --count;
    }
    void uncache(int32_t b) {
        if (!cached[(size_t)b]) return;
        cache.erase(key[(size_t)b]);
        cached[(size_t)b] = 0;
    }
    // Take the block at the head of the free queue; a cached block there is
    // evicted from the prefix cache (it was the least recently freed).
    int32_t pop_free() {
        const int32_t b = head;
        queue_remove(b);
        uncache(b);
        ref[(size_t)b] = 1;
        return b;
    }
    void release(int32_t b) {
        if (--ref[(size_t)b] == 0) queue_push_tail(b);
    }
    int32_t last_filled(const Seq &s) const {
        return s.num_tokens - (int32_t)(s.table.size() - 1) * block_size;
    }
};

namespace {

// 64-bit mixing (splitmix64 finaliser) and the block key chain.
uint64_t mix64(uint64_t x) {
    x += 0x9e3779b97f4a7c15ull;
    x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
    x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
    return x ^ (x >> 31);
}

uint64_t block_key(uint64_t parent, const int32_t *tok, int32_t n, int64_t extra) {
    uint64_t h = mix64(parent ^ 0x5bd1e995u);
    h = mix64(h ^ (uint64_t)extra);
    for (int32_t i = 0; i < n; ++i) h = mix64(h ^ (uint32_t)tok[i]);
    return h;
}

constexpr uint64_t kRootKey = 0x243f6a8885a308d3ull;

}  // namespace

using pagedkv::fail;

extern "C" {

int pa_pool_create(const pa_pool_desc *desc, pa_pool **out) {
    if (!desc || !out) return fail(PA_ERR_INVALID_ARG, "pa_pool_create: NULL argument");
    *out = nullptr;
    if (desc->num_blocks < 0 || desc->block_size < 1 || desc->num_layers < 1 ||
        desc->num_heads < 1 || desc->head_dim < 1 || desc->dtype != PA_DTYPE_F16 ||
        (desc->flags & ~PA_POOL_PREFIX_CACHING) != 0)
        return fail(PA_ERR_INVALID_ARG,
                    "pa_pool_create: bad geometry (num_blocks=%d block_size=%d num_layers=%d "
                    "num_heads=%d head_dim=%d dtype=%d flags=%d)",
                    desc->num_blocks, desc->block_size, desc->num_layers, desc->num_heads,
                    desc->head_dim, desc->dtype, desc->flags);
    pa_pool *p = new (std::nothrow) pa_pool();
    if (!p) return fail(PA_ERR_INVALID_ARG, "pa_pool_create: out of host memory");
    p->num_blocks = desc->num_blocks;
    p->block_size = desc->block_size;
    p->desc = *desc;
    p->desc.free_order = nullptr;
    const size_t nb = (size_t)desc->num_blocks;
    p->nxt.assign(nb, -1);
    p->prv.assign(nb, -1);
    p->in_queue.assign(nb, 0);
    p->ref.assign(nb, 0);
    p->plan_dec.assign(nb, 0);
    p->caching = (desc->flags & PA_POOL_PREFIX_CACHING) != 0;
    if (p->caching) {
        p->cached.assign(nb, 0);
        p->key.assign(nb, 0);
        p->parent_key.assign(nb, 0);
        p->extra.assign(nb, 0);
        p->tokens.assign(nb * (size_t)desc->block_size, 0);
    } else {
        p->cached.assign(nb, 0);
    }
    if (desc->free_order) {
        std::vector<char> seen(nb, 0);
        for (int32_t i = 0; i < desc->num_blocks; ++i) {
            int32_t b = desc->free_order[i];
            if (b < 0 || b >= desc->num_blocks || seen[(size_t)b]) {
                delete p;
                return fail(PA_ERR_INVALID_ARG,
                            "pa_pool_create: free_order is not a permutation (entry %d = %d)", i,
                            b);
            }
            seen[(size_t)b] = 1;
            p->queue_push_tail(b);
        }
    } else {
        for (int32_t i = 0; i < desc->num_blocks; ++i) p->queue_push_tail(i);
    }
    *out = p;
    return PA_OK;
}

int pa_pool_destroy(pa_pool *pool) {
    delete pool;
    return PA_OK;
}

int pa_seq_add(pa_pool *pool, int32_t seq_id, int32_t n_tokens, int64_t *slots_out) {
    if (!pool) return fail(PA_ERR_INVALID_ARG, "pa_seq_add: NULL pool");
    if (n_tokens < 0) return fail(PA_ERR_INVALID_ARG, "pa_seq_add: n_tokens < 0");
    if (pool->seqs.count(seq_id))
        return fail(PA_ERR_NO_SEQ, "pa_seq_add: sequence %d already exists", seq_id);
    const int32_t B = pool->block_size;
    int64_t need = ((int64_t)n_tokens + B - 1) / B;
    if (need > pool->count)
        return fail(PA_ERR_OUT_OF_BLOCKS, "pa_seq_add: need %lld blocks, %lld free",
                    (long long)need, (long long)pool->count);
    Seq s;
    s.table.reserve((size_t)need);
    for (int64_t i = 0; i < need; ++i) s.table.push_back(pool->pop_free());
    s.num_tokens = n_tokens;
    s.tver = next_table_version();
    if (slots_out)
        for (int32_t p = 0; p < n_tokens; ++p)
            slots_out[p] = (int64_t)s.table[(size_t)(p / B)] * B + p % B;
    pool->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
}

int pa_seq_add_tokens(pa_pool *pool, int32_t seq_id, int32_t n_tokens, const int32_t *token_ids,
                      int64_t extra_key, int64_t *slots_out, int32_t *n_cached_out) {
    if (!pool) return fail(PA_ERR_INVALID_ARG, "pa_seq_add_tokens: NULL pool");
    if (n_tokens < 0 || (n_tokens > 0 && !token_ids))
        return fail(PA_ERR_INVALID_ARG, "pa_seq_add_tokens: bad arguments");
    if (pool->seqs.count(seq_id))
        return fail(PA_ERR_NO_SEQ, "pa_seq_add_tokens: sequence %d already exists", seq_id);
    const int32_t B = pool->block_size;
    const int32_t total = (int32_t)(((int64_t)n_tokens + B - 1) / B);
    const int32_t full = n_tokens / B;
    // 1. the longest run of leading full blocks already in the cache, short
    // of the block holding the last prompt token: that token's query must be
    // computed, so its block is always new and written by the caller
    const int32_t reusable = n_tokens > 0 ? (n_tokens - 1) / B : 0;
    std::vector<int32_t> hit;
    std::vector<uint64_t> keys((size_t)full);
    uint64_t parent = kRootKey;
    bool chain = pool->caching;
    for (int32_t j = 0; j < full; ++j) {
        const int32_t *tok = token_ids + (int64_t)j * B;
        keys[(size_t)j] = block_key(parent, tok, B, extra_key);
        if (chain && j >= reusable) chain = false;
        if (chain) {
            auto it = pool->cache.find(keys[(size_t)j]);
            const int32_t b = it == pool->cache.end() ? -1 : it->second;
            if (b >= 0 && pool->cached[(size_t)b] && pool->parent_key[(size_t)b] == parent &&
                pool->extra[(size_t)b] == extra_key &&
                std::memcmp(&pool->tokens[(size_t)b * B], tok, sizeof(int32_t) * B) == 0)
                hit.push_back(b);
            else
                chain = false;
        }
        parent = keys[(size_t)j];
    }
    // 2. room for the rest: hits that sit in the free queue leave it
    int64_t hits_free = 0;
    for (int32_t b : hit) hits_free += pool->ref[(size_t)b] == 0;
    const int64_t need = total - (int64_t)hit.size();
    if (need > pool->count - hits_free)
        return fail(PA_ERR_OUT_OF_BLOCKS, "pa_seq_add_tokens: need %lld new blocks, %lld free",
                    (long long)need, (long long)(pool->count - hits_free));
    // 3. touch the hits, take new blocks, register the new full blocks
    Seq s;
    s.table.reserve((size_t)total);
    for (int32_t b : hit) {
        if (pool->ref[(size_t)b] == 0) pool->queue_remove(b);
        ++pool->ref[(size_t)b];
        s.table.push_back(b);
    }
    for (int64_t i = 0; i < need; ++i) s.table.push_back(pool->pop_free());
    if (pool->caching) {
        for (int32_t j = (int32_t)hit.size(); j < full; ++j) {
            const int32_t b = s.table[(size_t)j];
            const uint64_t k = keys[(size_t)j];
            if (pool->cache.count(k)) continue;   // a different block holds this key
            pool->cache.emplace(k, b);
            pool->cached[(size_t)b] = 1;
            pool->key[(size_t)b] = k;
            pool->parent_key[(size_t)b] = j ? keys[(size_t)j - 1] : kRootKey;
            pool->extra[(size_t)b] = extra_key;
            std::memcpy(&pool->tokens[(size_t)b * B], token_ids + (int64_t)j * B,
                        sizeof(int32_t) * B);
        }
    }
    s.num_tokens = n_tokens;
    s.tver = next_table_version();
    if (slots_out)
        for (int32_t p = 0; p < n_tokens; ++p)
            slots_out[p] = (int64_t)s.table[(size_t)(p / B)] * B + p % B;
    if (n_cached_out) *n_cached_out = (int32_t)hit.size() * B;
    pool->seqs.emplace(seq_id, std::move(s));
    return PA_OK;
}

int pa_pool_cached_blocks(const pa_pool *pool, int32_t *n_cached) {
    if (!pool || !n_cached) return fail(PA_ERR_INVALID_ARG, "pa_pool_cached_blocks: NULL argument");
    *n_cached = (int32_t)pool->cache.size();
    return PA_OK;
}

// Move a group of sequences from pool `from` to pool `to` (swapping).
static int move_group(const char *who, pa_pool *from, pa_pool *to, int32_t n_seqs,
                      const int32_t *seq_ids, int32_t *pairs_out, int32_t pairs_cap,
                      int32_t *n_pairs_out) {
    if (!from || !to || from == to || n_seqs < 0 || (n_seqs > 0 && !seq_ids) || pairs_cap < 0 ||
        (pairs_cap > 0 && !pairs_out))
        return fail(PA_ERR_INVALID_ARG, "%s: bad arguments", who);
    if (from->block_size != to->block_size)
        return fail(PA_ERR_INVALID_ARG, "%s: the pools' block sizes differ", who);
    // blocks of the group in first-use order, with their reference counts
    std::unordered_set<int32_t> ids;
    std::unordered_map<int32_t, int32_t> uses;   // block -> references from the group
    std::vector<int32_t> blocks;
    for (int32_t i = 0; i < n_seqs; ++i) {
        auto it = from->seqs.find(seq_ids[i]);
        if (it == from->seqs.end())
            return fail(PA_ERR_NO_SEQ, "%s: no sequence %d", who, seq_ids[i]);
        if (!ids.insert(seq_ids[i]).second)
            return fail(PA_ERR_INVALID_ARG, "%s: sequence %d listed twice", who, seq_ids[i]);
        if (to->seqs.count(seq_ids[i]))
            return fail(PA_ERR_NO_SEQ, "%s: sequence %d already in the target pool", who,
                        seq_ids[i]);
        for (int32_t b : it->second.table)
            if (uses[b]++ == 0) blocks.push_back(b);
    }
    for (int32_t b : blocks)
        if (from->ref[(size_t)b] != uses[b])
            return fail(PA_ERR_INVALID_ARG,
                        "%s: block %d is shared with a sequence outside the group", who, b);
    if ((int64_t)blocks.size() > to->count)
        return fail(PA_ERR_OUT_OF_BLOCKS, "%s: need %zu blocks, %lld free", who, blocks.size(),
                    (long long)to->count);
    if ((int64_t)blocks.size() > pairs_cap)
        return fail(PA_ERR_INVALID_ARG, "%s: %zu copies, pairs_cap is %d", who, blocks.size(),
                    pairs_cap);
    std::unordered_map<int32_t, int32_t> moved;
    for (size_t k = 0; k < blocks.size(); ++k) {
        const int32_t b = blocks[k], nb = to->pop_free();
        to->ref[(size_t)nb] = uses[b];
        moved[b] = nb;
        pairs_out[2 * k] = b;
        pairs_out[2 * k + 1] = nb;
    }
    for (int32_t i = 0; i < n_seqs; ++i) {
        auto it = from->seqs.find(seq_ids[i]);
        Seq s = std::move(it->second);
        from->seqs.erase(it);
        for (int32_t &b : s.table) b = moved[b];
        s.tver = next_table_version();
        to->seqs.emplace(seq_ids[i], std::move(s));
    }
    // the source blocks go back to their free queue, last-used first
    for (size_t k = blocks.size(); k-- > 0;) {
        from->ref[(size_t)blocks[k]] = 0;
        from->queue_push_tail(blocks[k]);
    }
    if (n_pairs_out) *n_pairs_out = (int32_t)blocks.size();
    return PA_OK;
}

int pa_swap_out(pa_pool *gpu, pa_pool *cpu, int32_t n_seqs, const int32_t *seq_ids,
                int32_t *pairs_out, int32_t pairs_cap, int32_t *n_pairs_out) {
    return move_group("pa_swap_out", gpu, cpu, n_seqs, seq_ids, pairs_out, pairs_cap, n_pairs_out);
}

int pa_swap_in(pa_pool *cpu, pa_pool *gpu, int32_t n_seqs, const int32_t *seq_ids,
               int32_t *pairs_out, int32_t pairs_cap, int32_t *n_pairs_out) {
    return move_group("pa_swap_in", cpu, gpu, n_seqs, seq_ids, pairs_out, pairs_cap, n_pairs_out);
}

int pa_seq_fork(pa_pool *pool, int32_t parent, int32_t child) {
    if (!pool) return fail(PA_ERR_INVALID_ARG, "pa_seq_fork: NULL pool");
    auto it = pool->seqs.find(parent);
    if (it == pool->seqs.end()) return fail(PA_ERR_NO_SEQ, "pa_seq_fork: no sequence %d", parent);
    if (pool->seqs.count(child))
        return fail(PA_ERR_NO_SEQ, "pa_seq_fork: sequence %d already exists", child);
    Seq c = it->second;
    for (int32_t b : c.table) ++pool->ref[(size_t)b];
    c.tver = next_table_version();
    pool->seqs.emplace(child, std::move(c));
    return PA_OK;
}

int pa_seq_fork_batch(pa_pool *pool, int32_t n, const int32_t *parents, const int32_t *children) {
    if (!pool || n < 0 || (n > 0 && (!parents || !children)))
        return fail(PA_ERR_INVALID_ARG, "pa_seq_fork_batch: bad arguments");
    std::unordered_set<int32_t> born;
    for (int32_t i = 0; i < n; ++i) {
        if (!pool->seqs.count(parents[i]) && !born.count(parents[i]))
            return fail(PA_ERR_NO_SEQ, "pa_seq_fork_batch: no sequence %d", parents[i]);
        if (pool->seqs.count(children[i]) || !born.insert(children[i]).second)
            return fail(PA_ERR_NO_SEQ, "pa_seq_fork_batch: sequence %d already exists",
                        children[i]);
    }
    for (int32_t i = 0; i < n; ++i) pa_seq_fork(pool, parents[i], children[i]);
    return PA_OK;
}

int pa_seq_free_batch(pa_pool *pool, int32_t n, const int32_t *seq_ids) {
    if (!pool || n < 0 || (n > 0 && !seq_ids))
        return fail(PA_ERR_INVALID_ARG, "pa_seq_free_batch: bad arguments");
    std::unordered_set<int32_t> seen;
    for (int32_t i = 0; i < n; ++i) {
        if (!pool->seqs.count(seq_ids[i]))
            return fail(PA_ERR_NO_SEQ, "pa_seq_free_batch: no sequence %d", seq_ids[i]);
        if (!seen.insert(seq_ids[i]).second)
            return fail(PA_ERR_INVALID_ARG, "pa_seq_free_batch: sequence %d listed twice",
                        seq_ids[i]);
    }
    for (int32_t i = 0; i < n; ++i) pa_seq_free(pool, seq_ids[i]);
    return PA_OK;
}

int pa_beam_prune(pa_pool *pool, int32_t n_groups, int32_t width, int32_t *beams,
                  const int32_t *counts, int32_t *next_id) {
    const char *who = "pa_beam_prune";
    if (!pool || n_groups < 0 || width < 1 || !next_id ||
        (n_groups > 0 && (!beams || !counts)))
        return fail(PA_ERR_INVALID_ARG, "%s: bad arguments", who);
    // check everything first: every beam exists once, each group keeps
    // `width` survivors, the new ids are unused
    const uint64_t epoch = ++pool->epoch;
    int64_t forks = 0;
    for (int32_t g = 0; g < n_groups; ++g) {
        int64_t kept = 0;
        for (int32_t i = 0; i < width; ++i) {
            const int32_t c = counts[(int64_t)g * width + i], id = beams[(int64_t)g * width + i];
            if (c < 0) return fail(PA_ERR_INVALID_ARG, "%s: negative count", who);
            auto it = pool->seqs.find(id);
            if (it == pool->seqs.end()) return fail(PA_ERR_NO_SEQ, "%s: no sequence %d", who, id);
            if (it->second.stamp == epoch)
                return fail(PA_ERR_INVALID_ARG, "%s: sequence %d listed twice", who, id);
            it->second.stamp = epoch;
            kept += c;
            if (c > 1) forks += c - 1;
        }
        if (kept != width)
            return fail(PA_ERR_INVALID_ARG, "%s: group %d keeps %lld beams, not %d", who, g,
                        (long long)kept, width);
    }
    if ((int64_t)*next_id + forks > INT32_MAX)
        return fail(PA_ERR_INVALID_ARG, "%s: sequence ids run out", who);
    for (int64_t k = 0; k < forks; ++k)
        if (pool->seqs.count((int32_t)(*next_id + k)))
            return fail(PA_ERR_NO_SEQ, "%s: sequence %lld already exists", who,
                        (long long)(*next_id + k));
    // apply, group by group: the survivors in beam order, each followed by its
    // forks; then the pruned beams are freed, in beam order
    std::vector<int32_t> &nb = pool->beam_row;
    int32_t nid = *next_id;
    for (int32_t g = 0; g < n_groups; ++g) {
        int32_t *row = beams + (int64_t)g * width;
        const int32_t *cnt = counts + (int64_t)g * width;
        nb.clear();
        for (int32_t i = 0; i < width; ++i) {
            if (cnt[i] == 0) continue;
            nb.push_back(row[i]);
            for (int32_t c = 1; c < cnt[i]; ++c) {
                pa_seq_fork(pool, row[i], nid);
                nb.push_back(nid++);
            }
        }
        for (int32_t i = 0; i < width; ++i)
            if (cnt[i] == 0) pa_seq_free(pool, row[i]);
        std::copy(nb.begin(), nb.end(), row);
    }
    nb.clear();
    *next_id = nid;
    return PA_OK;
}

int pa_seq_free(pa_pool *pool, int32_t seq_id) {
    if (!pool) return fail(PA_ERR_INVALID_ARG, "pa_seq_free: NULL pool");
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end()) return fail(PA_ERR_NO_SEQ, "pa_seq_free: no sequence %d", seq_id);
    const std::vector<int32_t> &t = it->second.table;
    for (size_t i = t.size(); i-- > 0;) pool->release(t[i]);
    pool->seqs.erase(it);
    return PA_OK;
}

}  // extern "C"

namespace {

// Dry run of one appended token for each of seq_ids (pa_alloc_slots): looks
// the sequences up into pool->plan_seqs and counts the new blocks and the
// copies.  Only the reference counts of shared last blocks change between
// the sequences of one call (each sequence appears once, new blocks belong
// to one sequence), so tracking those decrements reproduces the real pass
// exactly.  With max_blocks >= 0, a table that would grow beyond it fails
// the call.  Changes no state but the scratch.
int plan_append(pa_pool *pool, const char *who, int32_t n_seqs, const int32_t *seq_ids,
                int32_t max_blocks, int64_t *need_out, int32_t *n_copies_out) {
    const int32_t B = pool->block_size;
    const uint64_t epoch = ++pool->epoch;
    pool->plan_seqs.resize((size_t)n_seqs);
    pool->plan_touched.clear();
    int64_t need = 0;
    int32_t n_copies = 0;
    int rc = PA_OK;
    for (int32_t i = 0; i < n_seqs; ++i) {
        auto it = pool->seqs.find(seq_ids[i]);
        if (it == pool->seqs.end()) {
            rc = fail(PA_ERR_NO_SEQ, "%s: no sequence %d", who, seq_ids[i]);
            break;
        }
        Seq &s = it->second;
        if (s.stamp == epoch) {
            rc = fail(PA_ERR_INVALID_ARG, "%s: sequence %d listed twice", who, seq_ids[i]);
            break;
        }
        s.stamp = epoch;
        pool->plan_seqs[(size_t)i] = &s;
        size_t blocks_after = s.table.size();
        if (s.table.empty() || pool->last_filled(s) == B) {
            ++need;
            ++blocks_after;
        } else {
            const int32_t last = s.table.back();
            int32_t &d = pool->plan_dec[(size_t)last];
            if (pool->ref[(size_t)last] - d > 1) {
                if (d == 0) pool->plan_touched.push_back(last);
                ++need;
                ++n_copies;
                ++d;
            }
        }
        if (max_blocks >= 0 && (int64_t)blocks_after > max_blocks) {
            rc = fail(PA_ERR_INVALID_ARG, "%s: sequence %d would have %zu blocks > max_blocks %d",
                      who, seq_ids[i], blocks_after, max_blocks);
            break;
        }
    }
    for (int32_t b : pool->plan_touched) pool->plan_dec[(size_t)b] = 0;
    pool->plan_touched.clear();
    *need_out = need;
    *n_copies_out = n_copies;
    return rc;
}

// The real pass over pool->plan_seqs, after a successful plan_append.
int32_t commit_append(pa_pool *pool, int32_t n_seqs, int64_t *slot_mapping_out,
                      int32_t *copies_out) {
    const int32_t B = pool->block_size;
    int32_t c = 0;
    for (int32_t i = 0; i < n_seqs; ++i) {
        Seq &s = *pool->plan_seqs[(size_t)i];
        if (s.table.empty() || pool->last_filled(s) == B) {
            s.table.push_back(pool->pop_free());
            s.tver = next_table_version();
        } else {
            const int32_t last = s.table.back();
            if (pool->ref[(size_t)last] > 1) {
                const int32_t nb = pool->pop_free();
                copies_out[2 * c] = last;
                copies_out[2 * c + 1] = nb;
                ++c;
                --pool->ref[(size_t)last];
                s.table.back() = nb;
                s.tver = next_table_version();
            }
        }
        const int32_t off = s.num_tokens - (int32_t)(s.table.size() - 1) * B;
        slot_mapping_out[i] = (int64_t)s.table.back() * B + off;
        ++s.num_tokens;
    }
    return c;
}

// The decode step: append one token to each listed sequence (plan, then
// commit), then its slot, context length and padded table row.  With
// row_versions, row i is written only when the sequence's table version
// differs from row_versions[i] (then stored there).
int decode_step_prepare(pa_pool *pool, const char *who, int32_t n_seqs, const int32_t *seq_ids,
                        int32_t max_blocks, int64_t *slot_mapping_out, int32_t *ctx_lens_out,
                        int32_t *tables_out, uint64_t *row_versions, int32_t *copies_out,
                        int32_t copies_cap, int32_t *n_copies_out) {
    if (!pool) return fail(PA_ERR_INVALID_ARG, "%s: NULL pool", who);
    if (n_seqs < 0 || max_blocks < 0 || copies_cap < 0 || (copies_cap > 0 && !copies_out) ||
        (n_seqs > 0 && (!seq_ids || !slot_mapping_out || !ctx_lens_out ||
                        (max_blocks > 0 && !tables_out))))
        return fail(PA_ERR_INVALID_ARG, "%s: bad arguments", who);
    int64_t need = 0;
    int32_t n_copies = 0;
    int rc = plan_append(pool, who, n_seqs, seq_ids, max_blocks, &need, &n_copies);
    if (rc != PA_OK) return rc;
    if (need > pool->count)
        return fail(PA_ERR_OUT_OF_BLOCKS, "%s: need %lld blocks, %lld free", who,
                    (long long)need, (long long)pool->count);
    if (n_copies > copies_cap)
        return fail(PA_ERR_INVALID_ARG, "%s: %d copies needed, copies_cap is %d", who, n_copies,
                    copies_cap);
    const int32_t c = commit_append(pool, n_seqs, slot_mapping_out, copies_out);
    for (int32_t i = 0; i < n_seqs; ++i) {
        const Seq &s = *pool->plan_seqs[(size_t)i];
        ctx_lens_out[i] = s.num_tokens;
        if (row_versions) {
            if (row_versions[i] == s.tver) continue;   // the row already holds this table
            row_versions[i] = s.tver;
        }
        int32_t *row = tables_out + (int64_t)i * max_blocks;
        const size_t n = s.table.size();   // >= 1: the call appended a token
        std::memcpy(row, s.table.data(), n * sizeof(int32_t));
        for (int32_t j = (int32_t)n; j < max_blocks; ++j) row[j] = -1;
    }
    if (n_copies_out) *n_copies_out = c;
    return PA_OK;
}

}  // namespace

extern "C" {

int pa_alloc_slots(pa_pool *pool, int32_t n_seqs, const int32_t *seq_ids,
                   int64_t *slot_mapping_out, int32_t *copies_out, int32_t copies_cap,
                   int32_t *n_copies_out) {
    if (!pool) return fail(PA_ERR_INVALID_ARG, "pa_alloc_slots: NULL pool");
    if (n_seqs < 0 || (n_seqs > 0 && (!seq_ids || !slot_mapping_out)) || copies_cap < 0 ||
        (copies_cap > 0 && !copies_out))
        return fail(PA_ERR_INVALID_ARG, "pa_alloc_slots: bad arguments");
    int64_t need = 0;
    int32_t n_copies = 0;
    int rc = plan_append(pool, "pa_alloc_slots", n_seqs, seq_ids, -1, &need, &n_copies);
    if (rc != PA_OK) return rc;
    if (need > pool->count)
        return fail(PA_ERR_OUT_OF_BLOCKS, "pa_alloc_slots: need %lld blocks, %lld free",
                    (long long)need, (long long)pool->count);
    if (n_copies > copies_cap)
        return fail(PA_ERR_INVALID_ARG, "pa_alloc_slots: %d copies needed, copies_cap is %d",
                    n_copies, copies_cap);
    const int32_t c = commit_append(pool, n_seqs, slot_mapping_out, copies_out);
    if (n_copies_out) *n_copies_out = c;
    return PA_OK;
}

int pa_decode_step_prepare(pa_pool *pool, int32_t n_seqs, const int32_t *seq_ids,
                           int32_t max_blocks, int64_t *slot_mapping_out, int32_t *ctx_lens_out,
                           int32_t *tables_out, int32_t *copies_out, int32_t copies_cap,
                           int32_t *n_copies_out) {
    return decode_step_prepare(pool, "pa_decode_step_prepare", n_seqs, seq_ids, max_blocks,
                               slot_mapping_out, ctx_lens_out, tables_out, nullptr, copies_out,
                               copies_cap, n_copies_out);
}

int pa_decode_step_prepare_rows(pa_pool *pool, int32_t n_seqs, const int32_t *seq_ids,
                                int32_t max_blocks, int64_t *slot_mapping_out,
                                int32_t *ctx_lens_out, int32_t *tables_out,
                                uint64_t *row_versions, int32_t *copies_out, int32_t copies_cap,
                                int32_t *n_copies_out) {
    if (n_seqs > 0 && max_blocks > 0 && !row_versions)
        return fail(PA_ERR_INVALID_ARG, "pa_decode_step_prepare_rows: NULL row_versions");
    return decode_step_prepare(pool, "pa_decode_step_prepare_rows", n_seqs, seq_ids, max_blocks,
                               slot_mapping_out, ctx_lens_out, tables_out, row_versions,
                               copies_out, copies_cap, n_copies_out);
}

int pa_alloc_slots_n(pa_pool *pool, int32_t n_seqs, const int32_t *seq_ids,
                     const int32_t *counts, int64_t *slot_mapping_out, int32_t *copies_out,
                     int32_t copies_cap, int32_t *n_copies_out) {
    if (!pool) return fail(PA_ERR_INVALID_ARG, "pa_alloc_slots_n: NULL pool");
    if (n_seqs < 0 || (n_seqs > 0 && (!seq_ids || !counts)) || copies_cap < 0 ||
        (copies_cap > 0 && !copies_out))
        return fail(PA_ERR_INVALID_ARG, "pa_alloc_slots_n: bad arguments");
    const int32_t B = pool->block_size;
    // Dry run, as in pa_alloc_slots: only a shared, partly filled last block
    // (its count decremented by earlier copies in this call) needs a copy.
    std::vector<Seq *> seq(static_cast<size_t>(n_seqs));
    std::unordered_set<int32_t> ids;
    std::unordered_map<int32_t, int32_t> dec;
    int64_t need = 0, total = 0;
    int32_t n_copies = 0;
    for (int32_t i = 0; i < n_seqs; ++i) {
        auto it = pool->seqs.find(seq_ids[i]);
        if (it == pool->seqs.end())
            return fail(PA_ERR_NO_SEQ, "pa_alloc_slots_n: no sequence %d", seq_ids[i]);
        if (!ids.insert(seq_ids[i]).second)
            return fail(PA_ERR_INVALID_ARG, "pa_alloc_slots_n: sequence %d listed twice",
                        seq_ids[i]);
        if (counts[i] < 0) return fail(PA_ERR_INVALID_ARG, "pa_alloc_slots_n: negative count");
        Seq &s = it->second;
        seq[(size_t)i] = &s;
        total += counts[i];
        if (counts[i] == 0) continue;
        int64_t room = 0;   // free slots in the last block usable in place
        if (!s.table.empty() && pool->last_filled(s) < B) {
            const int32_t last = s.table.back();
            int32_t &d = dec[last];
            if (pool->ref[(size_t)last] - d > 1) {
                ++need;       // copy-on-write block, then filled
                ++n_copies;
                ++d;
            }
            room = B - pool->last_filled(s);
        }
        if (counts[i] > room) need += (counts[i] - room + B - 1) / B;
    }
    if (need > pool->count)
        return fail(PA_ERR_OUT_OF_BLOCKS, "pa_alloc_slots_n: need %lld blocks, %lld free",
                    (long long)need, (long long)pool->count);
    if (n_copies > copies_cap)
        return fail(PA_ERR_INVALID_ARG, "pa_alloc_slots_n: %d copies needed, copies_cap is %d",
                    n_copies, copies_cap);
    if (total > 0 && !slot_mapping_out)
        return fail(PA_ERR_INVALID_ARG, "pa_alloc_slots_n: NULL slot_mapping_out");
    int32_t c = 0;
    int64_t o = 0;
    for (int32_t i = 0; i < n_seqs; ++i) {
        Seq &s = *seq[(size_t)i];
        for (int32_t t = 0; t < counts[i]; ++t) {
            if (s.table.empty() || pool->last_filled(s) == B) {
                s.table.push_back(pool->pop_free());
                s.tver = next_table_version();
            } else if (t == 0 && pool->ref[(size_t)s.table.back()] > 1) {
                const int32_t last = s.table.back();
                const int32_t nb = pool->pop_free();
                copies_out[2 * c] = last;
                copies_out[2 * c + 1] = nb;
                ++c;
                --pool->ref[(size_t)last];
                s.table.back() = nb;
                s.tver = next_table_version();
            }
            const int32_t off = s.num_tokens - (int32_t)(s.table.size() - 1) * B;
            slot_mapping_out[o++] = (int64_t)s.table.back() * B + off;
            ++s.num_tokens;
        }
    }
    if (n_copies_out) *n_copies_out = c;
    return PA_OK;
}

int pa_get_block_tables(const pa_pool *pool, int32_t n_seqs, const int32_t *seq_ids,
                        int32_t max_blocks, int32_t *tables_out, int32_t *ctx_lens_out) {
    if (!pool) return fail(PA_ERR_INVALID_ARG, "pa_get_block_tables: NULL pool");
    if (n_seqs < 0 || max_blocks < 0 ||
        (n_seqs > 0 && (!seq_ids || (max_blocks > 0 && !tables_out))))
        return fail(PA_ERR_INVALID_ARG, "pa_get_block_tables: bad arguments");
    for (int32_t i = 0; i < n_seqs; ++i) {
        auto it = pool->seqs.find(seq_ids[i]);
        if (it == pool->seqs.end())
            return fail(PA_ERR_NO_SEQ, "pa_get_block_tables: no sequence %d", seq_ids[i]);
        const Seq &s = it->second;
        if ((int64_t)s.table.size() > max_blocks)
            return fail(PA_ERR_INVALID_ARG,
                        "pa_get_block_tables: sequence %d has %zu blocks > max_blocks %d",
                        seq_ids[i], s.table.size(), max_blocks);
        int32_t *row = tables_out + (int64_t)i * max_blocks;
        size_t n = s.table.size();
        if (n) std::memcpy(row, s.table.data(), n * sizeof(int32_t));
        for (int32_t j = (int32_t)n; j < max_blocks; ++j) row[j] = -1;
        if (ctx_lens_out) ctx_lens_out[i] = s.num_tokens;
    }
    return PA_OK;
}

int pa_seq_info(const pa_pool *pool, int32_t seq_id, int32_t *num_tokens, int32_t *num_blocks) {
    if (!pool) return fail(PA_ERR_INVALID_ARG, "pa_seq_info: NULL pool");
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end()) return fail(PA_ERR_NO_SEQ, "pa_seq_info: no sequence %d", seq_id);
    if (num_tokens) *num_tokens = it->second.num_tokens;
    if (num_blocks) *num_blocks = (int32_t)it->second.table.size();
    return PA_OK;
}

int pa_pool_num_free(const pa_pool *pool, int32_t *n_free) {
    if (!pool || !n_free) return fail(PA_ERR_INVALID_ARG, "pa_pool_num_free: NULL argument");
    *n_free = (int32_t)pool->count;
    return PA_OK;
}

int pa_pool_free_queue(const pa_pool *pool, int32_t *out, int32_t cap, int32_t *n_out) {
    if (!pool || (!out && cap > 0) || cap < 0)
        return fail(PA_ERR_INVALID_ARG, "pa_pool_free_queue: bad arguments");
    if (n_out) *n_out = (int32_t)pool->count;
    if (pool->count > cap)
        return fail(PA_ERR_INVALID_ARG, "pa_pool_free_queue: cap %d < queue length %lld", cap,
                    (long long)pool->count);
    int64_t i = 0;
    for (int32_t b = pool->head; b >= 0; b = pool->nxt[(size_t)b]) out[i++] = b;
    return PA_OK;
}

int pa_pool_refcounts(const pa_pool *pool, int32_t *out) {
    if (!pool || (!out && pool->num_blocks > 0))
        return fail(PA_ERR_INVALID_ARG, "pa_pool_refcounts: NULL argument");
    if (pool->num_blocks)
        std::memcpy(out, pool->ref.data(), sizeof(int32_t) * (size_t)pool->num_blocks);
    return PA_OK;
}

}  // extern "C"
