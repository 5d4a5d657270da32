// Host block allocator of the paged KV cache (C ABI in include/pa.h).
//
// Pages: "Q32: vLLM PagedAttention 原理" §2 (分块管理, Block Table映射, 非连续存储)
// and §3 (Copy-on-Write); data.6616ai.com "把虚拟内存搬进 KV Cache" and
// "Copy-on-write 共享"; ohmygp.com "破局思路" (按需分配, 块表映射, 写时共享).
//
// State: a FIFO free list kept as a ring buffer over num_blocks entries (each
// free block appears exactly once), one refcount per block, and per sequence
// its block table and length.  Every public call first checks that it can
// succeed (a dry run of the block demand) and only then mutates, so a failing
// call leaves the allocator unchanged.
#include <algorithm>
#include <cstring>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pa.h"

namespace {

struct Sequence {
    std::vector<int32_t> table;  // logical block -> physical block
    int32_t len = 0;             // tokens written
    bool swapped = false;        // blocks released to the host by pa_seq_swap_out; len kept
    // dry-run state of the current pa_append_batch call (valid while mark
    // equals the allocator's batch epoch)
    uint64_t mark = 0;
    int32_t dry_len = 0;
    bool dry_private = false;  // the tail is known to have refcount 1 at this point
};

// A full block registered in the prefix cache: the chained hash of the token
// prefix it completes, and (to verify a hit exactly) its parent's hash and its
// own token ids.
struct CachedBlock {
    uint64_t hash = 0, parent = 0;
    std::vector<int32_t> tokens;
    bool evictable = false;            // refcount 0: kept for reuse until its slot is needed
    std::list<int32_t>::iterator lru;  // position in the evictable list while evictable
};

// Chained hash of block i: mixes the previous block's hash with this block's
// token ids (splitmix64 finaliser as the mixing step).
uint64_t mix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}
uint64_t block_hash(uint64_t parent, const int32_t* tokens, int32_t n) {
    uint64_t h = mix64(parent ^ 0x5052454649584B56ull);
    for (int32_t i = 0; i < n; ++i) h = mix64(h ^ (uint64_t)(uint32_t)tokens[i]);
    return h;
}

}  // namespace

struct pa_allocator {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    int32_t max_refcount = 0;  // 0 = no cap
    std::vector<int32_t> ring;  // free list storage
    int32_t head = 0;           // index of the next block to pop
    int32_t free_count = 0;
    std::vector<int32_t> refcount;
    std::unordered_map<int64_t, Sequence> seqs;
    int64_t cow_copies = 0;
    // scratch of pa_append_batch, reused across calls so a batch allocates nothing
    uint64_t epoch = 0;               // batch calls so far
    std::vector<uint64_t> drop_mark;  // per block: the epoch drop_count belongs to
    std::vector<int32_t> drop_count;  // copies of a shared block planned in this call
    std::vector<Sequence*> batch;     // the call's sequences, in order

    // prefix cache: chained hash -> block, registered blocks, evictable ones oldest first
    std::unordered_map<uint64_t, int32_t> prefix_map;
    std::unordered_map<int32_t, CachedBlock> cached;
    std::list<int32_t> lru;

    // Blocks an allocation may take: the free list, then evictable cached blocks.
    int64_t available() const { return (int64_t)free_count + (int64_t)lru.size(); }
    int32_t pop_free() {
        int32_t b;
        if (free_count > 0) {
            b = ring[head];
            head = (head + 1) % num_blocks;
            --free_count;
        } else {  // evict the least recently released cached block
            b = lru.front();
            lru.pop_front();
            auto it = cached.find(b);
            prefix_map.erase(it->second.hash);
            cached.erase(it);
        }
        refcount[b] = 1;
        return b;
    }
    void push_free(int32_t b) {
        ring[(head + free_count) % num_blocks] = b;
        ++free_count;
    }
    // A block whose last reference went: a cached block stays cached (evictable,
    // most recent at the back); any other returns to the back of the free list.
    void release(int32_t b) {
        auto it = cached.find(b);
        if (it == cached.end()) {
            push_free(b);
            return;
        }
        it->second.evictable = true;
        it->second.lru = lru.insert(lru.end(), b);
    }
    // Blocks one append of n tokens to `s` will take: the blocks newly
    // started plus one copy if the first token lands in a shared tail.
    int64_t demand(const Sequence& s, int32_t n, int32_t tail_refs) const {
        if (n <= 0) return 0;
        int64_t before = (s.len + block_size - 1) / block_size;
        int64_t after = ((int64_t)s.len + n + block_size - 1) / block_size;
        int64_t copy = (s.len % block_size != 0 && tail_refs > 1) ? 1 : 0;
        return (after - before) + copy;
    }
    // One token; caller guarantees a free block is available when needed.
    void append_one(Sequence& s, int64_t* slot, int32_t* pairs, int32_t* n_pairs) {
        const int32_t off = s.len % block_size;
        if (off == 0) {
            s.table.push_back(pop_free());
        } else {
            int32_t& tail = s.table.back();
            if (refcount[tail] > 1) {
                int32_t fresh = pop_free();
                pairs[2 * *n_pairs] = tail;
                pairs[2 * *n_pairs + 1] = fresh;
                ++*n_pairs;
                --refcount[tail];
                tail = fresh;
                ++cow_copies;
            }
        }
        *slot = (int64_t)s.table[s.len / block_size] * block_size + off;
        ++s.len;
    }
};

#define PA_GUARD_BEGIN try {
#define PA_GUARD_END                \
    }                               \
    catch (const std::bad_alloc&) { \
        return PA_ERR_INTERNAL;     \
    }                               \
    catch (...) {                   \
        return PA_ERR_INTERNAL;     \
    }

extern "C" {

pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order, pa_allocator** out) {
    if (!out || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
    *out = nullptr;
    PA_GUARD_BEGIN
    pa_allocator* a = new pa_allocator();
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->ring.resize(num_blocks);
    a->refcount.assign(num_blocks, 0);
    a->drop_mark.assign(num_blocks, 0);
    a->drop_count.assign(num_blocks, 0);
    if (free_order) {
        std::vector<char> seen(num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[b]) {
                delete a;
                return PA_ERR_INVALID_ARG;
            }
            seen[b] = 1;
            a->ring[i] = b;
        }
    } else {
        for (int32_t i = 0; i < num_blocks; ++i) a->ring[i] = i;
    }
    a->head = 0;
    a->free_count = num_blocks;
    *out = a;
    return PA_OK;
    PA_GUARD_END
}

void pa_alloc_destroy(pa_allocator* a) { delete a; }

pa_status pa_alloc_set_max_refcount(pa_allocator* a, int32_t max_refcount) {
    if (!a || max_refcount < 0) return PA_ERR_INVALID_ARG;
    a->max_refcount = max_refcount;
    return PA_OK;
}

pa_status pa_seq_create(pa_allocator* a, int64_t seq_id) {
    if (!a) return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    if (a->seqs.count(seq_id)) return PA_ERR_SEQ_EXISTS;
    a->seqs.emplace(seq_id, Sequence());
    return PA_OK;
    PA_GUARD_END
}

pa_status pa_seq_append(pa_allocator* a, int64_t seq_id, int32_t n_tokens, int64_t* slots_out,
                        int32_t* cow_pairs_out, int32_t* n_cow_out) {
    if (!a || n_tokens < 0 || (n_tokens > 0 && (!slots_out || !cow_pairs_out)) || !n_cow_out)
        return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NO_SUCH_SEQ;
    Sequence& s = it->second;
    if (s.swapped) return PA_ERR_SEQ_SWAPPED;
    if ((int64_t)s.len + n_tokens > INT32_MAX) return PA_ERR_INVALID_ARG;
    int32_t tail_refs = s.table.empty() ? 0 : a->refcount[s.table.back()];
    if (a->demand(s, n_tokens, tail_refs) > a->available()) return PA_ERR_OUT_OF_BLOCKS;
    s.table.reserve((s.len + n_tokens + a->block_size - 1) / a->block_size);
    *n_cow_out = 0;
    for (int32_t i = 0; i < n_tokens; ++i) a->append_one(s, &slots_out[i], cow_pairs_out, n_cow_out);
    return PA_OK;
    PA_GUARD_END
}

pa_status pa_append_batch(pa_allocator* a, const int64_t* seq_ids, int32_t n, int64_t* slots_out,
                          int32_t* cow_pairs_out, int32_t* n_cow_out) {
    if (!a || n < 0 || (n > 0 && (!seq_ids || !slots_out || !cow_pairs_out)) || !n_cow_out)
        return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    // Dry run: the same id may appear more than once, and a copy made for an
    // earlier id lowers the refcount a later sharer sees.  Per-call state lives
    // in the sequences and in per-block arrays, stamped with this call's epoch.
    const uint64_t ep = ++a->epoch;
    const int32_t bs = a->block_size;
    a->batch.resize(n);
    int64_t need = 0;
    for (int32_t i = 0; i < n; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return PA_ERR_NO_SUCH_SEQ;
        Sequence* s = &it->second;
        if (s->swapped) return PA_ERR_SEQ_SWAPPED;
        a->batch[i] = s;
        if (s->mark != ep) {
            s->mark = ep;
            s->dry_len = s->len;
            s->dry_private = false;
        }
        if (s->dry_len % bs == 0) {
            ++need;
            s->dry_private = true;
        } else if (!s->dry_private) {
            const int32_t tail = s->table.back();
            const int32_t drop = a->drop_mark[tail] == ep ? a->drop_count[tail] : 0;
            if (a->refcount[tail] - drop > 1) {
                ++need;
                a->drop_mark[tail] = ep;
                a->drop_count[tail] = drop + 1;
            }
            s->dry_private = true;
        }
        if (s->dry_len == INT32_MAX) return PA_ERR_INVALID_ARG;
        ++s->dry_len;
    }
    if (need > a->available()) return PA_ERR_OUT_OF_BLOCKS;
    for (int32_t i = 0; i < n; ++i)  // so that the mutating loop below cannot fail half-way
        a->batch[i]->table.reserve((a->batch[i]->dry_len + bs - 1) / bs);
    *n_cow_out = 0;
    for (int32_t i = 0; i < n; ++i) a->append_one(*a->batch[i], &slots_out[i], cow_pairs_out, n_cow_out);
    return PA_OK;
    PA_GUARD_END
}

pa_status pa_seq_fork(pa_allocator* a, int64_t parent, int64_t child) {
    if (!a) return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end()) return PA_ERR_NO_SUCH_SEQ;
    if (it->second.swapped) return PA_ERR_SEQ_SWAPPED;
    if (a->seqs.count(child)) return PA_ERR_SEQ_EXISTS;
    if (a->max_refcount > 0)
        for (int32_t b : it->second.table)
            if (a->refcount[b] + 1 > a->max_refcount) return PA_ERR_REFCOUNT_LIMIT;
    Sequence copy = it->second;  // may throw before any state changes
    for (int32_t b : copy.table) ++a->refcount[b];
    a->seqs.emplace(child, std::move(copy));
    return PA_OK;
    PA_GUARD_END
}

pa_status pa_seq_free(pa_allocator* a, int64_t seq_id) {
    if (!a) return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NO_SUCH_SEQ;
    for (int32_t b : it->second.table)
        if (--a->refcount[b] == 0) a->release(b);
    a->seqs.erase(it);
    return PA_OK;
    PA_GUARD_END
}

pa_status pa_seq_swap_out(pa_allocator* a, int64_t seq_id, int32_t* blocks_out, int32_t cap, int32_t* n_out) {
    if (!a || !n_out || cap < 0 || (cap > 0 && !blocks_out)) return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NO_SUCH_SEQ;
    Sequence& s = it->second;
    if (s.swapped) return PA_ERR_SEQ_SWAPPED;
    *n_out = (int32_t)s.table.size();
    if ((int32_t)s.table.size() > cap) return PA_ERR_BUFFER_TOO_SMALL;
    std::copy(s.table.begin(), s.table.end(), blocks_out);
    // the sequence's references go, as in pa_seq_free; its length stays
    for (int32_t b : s.table)
        if (--a->refcount[b] == 0) a->release(b);
    s.table.clear();
    s.swapped = true;
    return PA_OK;
    PA_GUARD_END
}

pa_status pa_seq_swap_in(pa_allocator* a, int64_t seq_id, int32_t* blocks_out, int32_t cap, int32_t* n_out) {
    if (!a || !n_out || cap < 0 || (cap > 0 && !blocks_out)) return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NO_SUCH_SEQ;
    Sequence& s = it->second;
    if (!s.swapped) return PA_ERR_INVALID_ARG;
    const int32_t need = (int32_t)(((int64_t)s.len + a->block_size - 1) / a->block_size);
    *n_out = need;
    if (need > cap) return PA_ERR_BUFFER_TOO_SMALL;
    if (need > a->available()) return PA_ERR_OUT_OF_BLOCKS;
    s.table.reserve(need);  // may throw before any state changes
    for (int32_t i = 0; i < need; ++i) s.table.push_back(a->pop_free());
    std::copy(s.table.begin(), s.table.end(), blocks_out);
    s.swapped = false;
    return PA_OK;
    PA_GUARD_END
}

pa_status pa_seq_create_cached(pa_allocator* a, int64_t seq_id, const int32_t* tokens, int32_t n_tokens,
                               int32_t* n_cached_out) {
    if (!a || n_tokens < 0 || (n_tokens > 0 && !tokens) || !n_cached_out) return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    if (a->seqs.count(seq_id)) return PA_ERR_SEQ_EXISTS;
    const int32_t bs = a->block_size;
    // the longest run of cached full blocks; at least one prompt token is left to compute
    const int32_t max_blocks = n_tokens > 0 ? (n_tokens - 1) / bs : 0;
    std::vector<int32_t> hits;
    hits.reserve(max_blocks);
    uint64_t h = 0;
    for (int32_t i = 0; i < max_blocks; ++i) {
        const int32_t* tk = tokens + (size_t)i * bs;
        const uint64_t hi = block_hash(h, tk, bs);
        auto m = a->prefix_map.find(hi);
        if (m == a->prefix_map.end()) break;
        const CachedBlock& cb = a->cached.find(m->second)->second;
        if (cb.parent != h || !std::equal(cb.tokens.begin(), cb.tokens.end(), tk)) break;
        if (a->max_refcount > 0 && a->refcount[m->second] + 1 > a->max_refcount) break;
        hits.push_back(m->second);
        h = hi;
    }
    Sequence s;
    s.table = hits;  // may throw before any state changes
    s.len = (int32_t)hits.size() * bs;
    auto it = a->seqs.emplace(seq_id, std::move(s)).first;
    for (int32_t b : it->second.table) {
        CachedBlock& cb = a->cached.find(b)->second;
        if (cb.evictable) {  // revived: leaves the evictable list
            a->lru.erase(cb.lru);
            cb.evictable = false;
        }
        ++a->refcount[b];
    }
    *n_cached_out = it->second.len;
    return PA_OK;
    PA_GUARD_END
}

pa_status pa_seq_cache_prefix(pa_allocator* a, int64_t seq_id, const int32_t* tokens, int32_t n_tokens) {
    if (!a || n_tokens < 0 || (n_tokens > 0 && !tokens)) return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NO_SUCH_SEQ;
    const Sequence& s = it->second;
    if (s.swapped) return PA_ERR_SEQ_SWAPPED;
    if (n_tokens > s.len) return PA_ERR_INVALID_ARG;
    const int32_t bs = a->block_size, nfull = n_tokens / bs;
    // register the full blocks in order; a prefix already cached (the same block,
    // or another block with the same content) keeps its entry
    std::vector<CachedBlock> fresh;
    std::vector<int32_t> fresh_blocks;
    uint64_t h = 0;
    for (int32_t i = 0; i < nfull; ++i) {
        const int32_t* tk = tokens + (size_t)i * bs;
        const uint64_t hi = block_hash(h, tk, bs);
        const int32_t b = s.table[i];
        bool dup = a->prefix_map.count(hi) || a->cached.count(b);
        for (const CachedBlock& f : fresh) dup = dup || f.hash == hi;
        if (!dup && std::find(fresh_blocks.begin(), fresh_blocks.end(), b) == fresh_blocks.end()) {
            CachedBlock cb;
            cb.hash = hi;
            cb.parent = h;
            cb.tokens.assign(tk, tk + bs);
            fresh.push_back(std::move(cb));
            fresh_blocks.push_back(b);
        }
        h = hi;
    }
    a->prefix_map.reserve(a->prefix_map.size() + fresh.size());  // may throw before any state changes
    a->cached.reserve(a->cached.size() + fresh.size());
    for (size_t k = 0; k < fresh.size(); ++k) {
        a->prefix_map.emplace(fresh[k].hash, fresh_blocks[k]);
        a->cached.emplace(fresh_blocks[k], std::move(fresh[k]));
    }
    return PA_OK;
    PA_GUARD_END
}

pa_status pa_prefix_cache_stats(const pa_allocator* a, int32_t* cached_blocks, int32_t* evictable_blocks) {
    if (!a) return PA_ERR_INVALID_ARG;
    if (cached_blocks) *cached_blocks = (int32_t)a->cached.size();
    if (evictable_blocks) *evictable_blocks = (int32_t)a->lru.size();
    return PA_OK;
}

pa_status pa_seq_block_table(const pa_allocator* a, int64_t seq_id, int32_t* out, int32_t cap, int32_t* n_out) {
    if (!a || !n_out || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NO_SUCH_SEQ;
    if (it->second.swapped) return PA_ERR_SEQ_SWAPPED;
    const auto& t = it->second.table;
    *n_out = (int32_t)t.size();
    if ((int32_t)t.size() > cap) return PA_ERR_BUFFER_TOO_SMALL;
    std::copy(t.begin(), t.end(), out);
    return PA_OK;
    PA_GUARD_END
}

pa_status pa_seq_len(const pa_allocator* a, int64_t seq_id, int32_t* len_out) {
    if (!a || !len_out) return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return PA_ERR_NO_SUCH_SEQ;
    *len_out = it->second.len;
    return PA_OK;
    PA_GUARD_END
}

pa_status pa_export_tables(const pa_allocator* a, const int64_t* seq_ids, int32_t n, int32_t max_blocks_per_seq,
                           int32_t* tables_out, int32_t* lens_out) {
    if (!a || n < 0 || max_blocks_per_seq <= 0 || (n > 0 && (!seq_ids || !tables_out || !lens_out)))
        return PA_ERR_INVALID_ARG;
    PA_GUARD_BEGIN
    for (int32_t i = 0; i < n; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end()) return PA_ERR_NO_SUCH_SEQ;
        if (it->second.swapped) return PA_ERR_SEQ_SWAPPED;
        if ((int32_t)it->second.table.size() > max_blocks_per_seq) return PA_ERR_BUFFER_TOO_SMALL;
    }
    for (int32_t i = 0; i < n; ++i) {
        const Sequence& s = a->seqs.find(seq_ids[i])->second;
        int32_t* row = tables_out + (size_t)i * max_blocks_per_seq;
        std::copy(s.table.begin(), s.table.end(), row);
        std::fill(row + s.table.size(), row + max_blocks_per_seq, 0);
        lens_out[i] = s.len;
    }
    return PA_OK;
    PA_GUARD_END
}

int32_t pa_block_refcount(const pa_allocator* a, int32_t block) {
    if (!a || block < 0 || block >= a->num_blocks) return -1;
    return a->refcount[block];
}

pa_status pa_alloc_stats(const pa_allocator* a, pa_alloc_stats_t* out) {
    if (!a || !out) return PA_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof *out);
    out->num_blocks = a->num_blocks;
    out->block_size = a->block_size;
    out->free_blocks = a->free_count;
    for (int32_t r : a->refcount) out->used_blocks += (r > 0);
    for (int32_t r : a->refcount) out->shared_blocks += (r > 1);
    out->num_seqs = (int32_t)a->seqs.size();
    for (const auto& kv : a->seqs) out->tokens += kv.second.len;
    out->slots = (int64_t)out->used_blocks * a->block_size;
    out->cow_copies = a->cow_copies;
    return PA_OK;
}

pa_status pa_alloc_free_list(const pa_allocator* a, int32_t* out, int32_t cap, int32_t* n_out) {
    if (!a || !n_out || cap < 0 || (cap > 0 && !out)) return PA_ERR_INVALID_ARG;
    *n_out = a->free_count;
    if (a->free_count > cap) return PA_ERR_BUFFER_TOO_SMALL;
    for (int32_t i = 0; i < a->free_count; ++i) out[i] = a->ring[(a->head + i) % a->num_blocks];
    return PA_OK;
}

const char* pa_status_str(pa_status s) {
    switch (s) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PA_ERR_OUT_OF_BLOCKS: return "out of free blocks";
        case PA_ERR_NO_SUCH_SEQ: return "no such sequence";
        case PA_ERR_SEQ_EXISTS: return "sequence already exists";
        case PA_ERR_REFCOUNT_LIMIT: return "refcount limit reached";
        case PA_ERR_WORKSPACE_TOO_SMALL: return "decode workspace too small";
        case PA_ERR_BUFFER_TOO_SMALL: return "output buffer too small";
        case PA_ERR_CUDA: return "CUDA error";
        case PA_ERR_INTERNAL: return "internal error";
        case PA_ERR_SEQ_SWAPPED: return "sequence is swapped out";
    }
    return "unknown status";
}

int32_t pa_abi_version(void) { return PA_ABI_VERSION; }

}  // extern "C"
