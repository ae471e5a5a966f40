// Host block allocator for the paged KV cache (C ABI in include/pkv.h).
//
// What it keeps, following the PagedAttention pages:
//  - a pool of fixed-size physical blocks and, per sequence, a block table
//    mapping logical block i to a physical block (aiplusplus page, "core
//    idea" 1-3);
//  - on-demand allocation: blocks for the prompt on arrival, one more when a
//    new token starts a block; any free block serves (same page, "core idea"
//    4 and "effects"); a finished sequence returns its blocks at once
//    ("continuous batching");
//  - reference counts for blocks shared between tables (prefix sharing, beam
//    search) and a copy-on-write decision when a sequence writes into a
//    shared block that is not full (auturnal guide, section 3; cayang0802
//    walkthrough, beam search of width 4).
//  - an index of full blocks by content for automatic prefix caching
//    (cayang0802 walkthrough, prefix caching): a full block's key is a hash
//    of its own tokens and of every token before it, so equal keys mean equal
//    KV; a new sequence reuses the cached blocks of its longest matching
//    prefix.  A registered block whose count drops to zero is kept, still
//    findable, in a least-recently-freed list, and is only evicted (and
//    unregistered) when the plain free list is empty.
// Every operation either completes or leaves the state untouched (OOM and
// bad arguments included), as the auturnal guide's section 6 asks of OOM.
#include <cstdint>
#include <cstring>
#include <list>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

// FNV-1a, 64-bit (Fowler, Noll, Vo): offset basis 14695981039346656037,
// prime 1099511628211, over bytes.
struct Fnv1a {
    uint64_t h = 14695981039346656037ull;
    void byte(uint8_t b)
    {
        h ^= b;
        h *= 1099511628211ull;
    }
    void u64(uint64_t v)
    {
        for (int i = 0; i < 8; ++i) byte((uint8_t)(v >> (8 * i)));
    }
    void i32(int32_t v)
    {
        const uint32_t u = (uint32_t)v;
        for (int i = 0; i < 4; ++i) byte((uint8_t)(u >> (8 * i)));
    }
};

// Key of a full block: FNV-1a over the parent block's key (0 for the first
// block, 8 bytes little-endian) followed by the block's B token ids (4 bytes
// little-endian each).
uint64_t block_key(uint64_t parent, const int32_t* tokens, int block_size)
{
    Fnv1a f;
    f.u64(parent);
    for (int i = 0; i < block_size; ++i) f.i32(tokens[i]);
    return f.h;
}

}  // namespace

struct pkv_allocator {
    int num_blocks = 0;
    int block_size = 0;
    std::vector<int32_t> free_stack;  // back() is handed out next
    std::vector<int32_t> ref;         // reference count per physical block
    struct Seq {
        std::vector<int32_t> table;
        int64_t len = 0;
        // a decode step's plan (plan_step): valid while mark == the step's stamp
        uint64_t mark = 0;
        int64_t sim_len = 0, sim_blocks = 0;
        int32_t sim_last = -1;  // -1: a block taken in this step (private)
    };
    std::unordered_map<int64_t, Seq> seqs;

    // ---- scratch of a decode step, kept across steps so a step allocates
    // nothing: the stamp of the current plan, the sequences of the step, and
    // per block the count drops earlier appends of the step make (valid
    // where dref_mark == stamp)
    uint64_t stamp = 0;
    std::vector<Seq*> step_seqs;
    std::vector<int32_t> dref;
    std::vector<uint64_t> dref_mark;

    // ---- prefix cache: registered full blocks
    std::unordered_map<uint64_t, int32_t> index;  // key -> block
    std::vector<char> registered;                 // per block
    std::vector<uint64_t> key, parent_key;        // per registered block
    std::vector<int32_t> tokens;                  // [num_blocks][block_size]
    std::list<int32_t> cached_free;               // count 0, still findable; front = oldest
    std::vector<std::list<int32_t>::iterator> cached_pos;
    int64_t prefix_hits = 0;

    size_t available() const { return free_stack.size() + cached_free.size(); }

    void unregister(int32_t b)
    {
        auto it = index.find(key[b]);
        if (it != index.end() && it->second == b) index.erase(it);
        registered[b] = 0;
    }
    int32_t pop()
    {
        int32_t b;
        if (!free_stack.empty()) {
            b = free_stack.back();
            free_stack.pop_back();
        } else {  // evict the least recently freed cached block
            b = cached_free.front();
            cached_free.pop_front();
            unregister(b);
        }
        ref[b] = 1;
        return b;
    }
    void release(int32_t b)
    {
        if (--ref[b] == 0) {
            if (registered[b]) {
                cached_free.push_back(b);
                cached_pos[b] = std::prev(cached_free.end());
            } else {
                free_stack.push_back(b);
            }
        }
    }
    void take(int32_t b)  // one more user of a registered block
    {
        if (ref[b] == 0) cached_free.erase(cached_pos[b]);
        ref[b] += 1;
    }
    // Block cached for (parent key, tokens), or -1.
    int32_t lookup(uint64_t k, uint64_t parent, const int32_t* toks) const
    {
        auto it = index.find(k);
        if (it == index.end()) return -1;
        const int32_t b = it->second;
        if (parent_key[b] != parent ||
            std::memcmp(&tokens[(size_t)b * block_size], toks, sizeof(int32_t) * block_size))
            return -1;  // a key collision: contents differ
        return b;
    }
    void append_one(Seq& s, int64_t* slot, int64_t* src, int64_t* dst)
    {
        *src = *dst = -1;
        int64_t p = s.len;
        if (p % block_size == 0) {
            s.table.push_back(pop());
        } else {
            int32_t last = s.table.back();
            if (ref[last] > 1) {
                int32_t fresh = pop();
                release(last);
                s.table.back() = fresh;
                *src = last;
                *dst = fresh;
            }
        }
        *slot = (int64_t)s.table[p / block_size] * block_size + p % block_size;
        s.len = p + 1;
    }
};

extern "C" {

int pkv_alloc_create(int num_blocks, int block_size, const int32_t* free_order,
                     pkv_allocator** out)
{
    if (!out) return pkv_fail(PKV_ERR_NULL, "pkv_alloc_create: out is NULL");
    *out = nullptr;
    if (num_blocks < 0 || block_size <= 0)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_alloc_create: num_blocks=%d block_size=%d",
                        num_blocks, block_size);
    pkv_allocator* a = new (std::nothrow) pkv_allocator();
    if (!a) return pkv_fail(PKV_ERR_OOM, "pkv_alloc_create: host allocation failed");
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->ref.assign(num_blocks, 0);
    a->registered.assign(num_blocks, 0);
    a->key.assign(num_blocks, 0);
    a->parent_key.assign(num_blocks, 0);
    a->tokens.assign((size_t)num_blocks * block_size, 0);
    a->cached_pos.resize(num_blocks);
    a->dref.assign(num_blocks, 0);
    a->dref_mark.assign(num_blocks, 0);
    a->free_stack.resize(num_blocks);
    std::vector<char> seen(num_blocks, 0);
    for (int i = 0; i < num_blocks; ++i) {
        int32_t b = free_order ? free_order[i] : i;
        if (b < 0 || b >= num_blocks || seen[b]) {
            delete a;
            return pkv_fail(PKV_ERR_SHAPE, "pkv_alloc_create: free_order is not a permutation");
        }
        seen[b] = 1;
        a->free_stack[num_blocks - 1 - i] = b;  // first of free_order on top
    }
    *out = a;
    return PKV_OK;
}

int pkv_alloc_destroy(pkv_allocator* a)
{
    delete a;
    return PKV_OK;
}

int pkv_seq_add(pkv_allocator* a, int64_t seq, int prompt_len)
{
    if (!a) return pkv_fail(PKV_ERR_NULL, "pkv_seq_add: allocator is NULL");
    if (prompt_len < 0) return pkv_fail(PKV_ERR_SHAPE, "pkv_seq_add: negative prompt_len");
    if (a->seqs.count(seq)) return pkv_fail(PKV_ERR_STATE, "pkv_seq_add: sequence exists");
    int64_t n = (prompt_len + (int64_t)a->block_size - 1) / a->block_size;
    if (n > (int64_t)a->available())
        return pkv_fail(PKV_ERR_OOM, "pkv_seq_add: %lld blocks needed, %zu free",
                        (long long)n, a->available());
    pkv_allocator::Seq s;
    s.table.reserve(n);
    for (int64_t i = 0; i < n; ++i) s.table.push_back(a->pop());
    s.len = prompt_len;
    a->seqs.emplace(seq, std::move(s));
    return PKV_OK;
}

int pkv_seq_append(pkv_allocator* a, int64_t seq, int64_t* slot, int64_t* cow_src,
                   int64_t* cow_dst)
{
    if (!a || !slot || !cow_src || !cow_dst)
        return pkv_fail(PKV_ERR_NULL, "pkv_seq_append: NULL argument");
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return pkv_fail(PKV_ERR_STATE, "pkv_seq_append: unknown sequence");
    const pkv_allocator::Seq& s = it->second;
    bool need = s.len % a->block_size == 0 || a->ref[s.table.back()] > 1;
    if (need && a->available() == 0)
        return pkv_fail(PKV_ERR_OOM, "pkv_seq_append: no free block");
    a->append_one(it->second, slot, cow_src, cow_dst);
    return PKV_OK;
}

}  // extern "C"

namespace {

// Blocks one decode step over seqs[0..n) must take (a fresh block for a token
// that starts one, a copy target for a write into a shared partial block),
// found without changing the allocator's state (only its step scratch): the
// walk tracks, per sequence, its length and whether its last block is
// already private, and per shared block the count drops earlier appends of
// the same step make, so that a block shared by two sequences of the step is
// copied once and its last holder writes in place.  Also checks every
// sequence exists and (max_blocks > 0) that no table grows past max_blocks.
// Leaves the step's sequences in a->step_seqs.
int plan_step(pkv_allocator* a, const int64_t* seqs, int n, const char* fn, int max_blocks,
              int64_t* need_out)
{
    const uint64_t stamp = ++a->stamp;
    a->step_seqs.resize(n);
    int64_t need = 0;
    for (int i = 0; i < n; ++i) {
        auto it = a->seqs.find(seqs[i]);
        if (it == a->seqs.end())
            return pkv_fail(PKV_ERR_STATE, "%s: unknown sequence %lld", fn, (long long)seqs[i]);
        pkv_allocator::Seq& s = it->second;
        a->step_seqs[i] = &s;
        if (s.mark == stamp && max_blocks > 0)  // one table row per sequence
            return pkv_fail(PKV_ERR_STATE, "%s: sequence %lld listed twice", fn,
                            (long long)seqs[i]);
        if (s.mark != stamp) {
            s.mark = stamp;
            s.sim_len = s.len;
            s.sim_blocks = (int64_t)s.table.size();
            s.sim_last = s.table.empty() ? -1 : s.table.back();
        }
        if (s.sim_len % a->block_size == 0) {
            s.sim_last = -1;
            s.sim_blocks += 1;
            need += 1;
        } else if (s.sim_last >= 0 && a->ref[s.sim_last] > 1) {
            const int32_t b = s.sim_last;
            if (a->dref_mark[b] != stamp) {
                a->dref_mark[b] = stamp;
                a->dref[b] = 0;
            }
            if (a->ref[b] + a->dref[b] > 1) {
                a->dref[b] -= 1;
                s.sim_last = -1;
                need += 1;
            }
        }
        s.sim_len += 1;
        if (max_blocks > 0 && s.sim_blocks > max_blocks)
            return pkv_fail(PKV_ERR_SHAPE, "%s: sequence %lld would need %lld table entries, %d "
                            "fit", fn, (long long)seqs[i], (long long)s.sim_blocks, max_blocks);
    }
    if (need > (int64_t)a->available())
        return pkv_fail(PKV_ERR_OOM, "%s: %lld blocks needed, %zu free", fn, (long long)need,
                        a->available());
    *need_out = need;
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_step_append(pkv_allocator* a, const int64_t* seqs, int n, int64_t* slots,
                    int64_t* cow_pairs, int* num_pairs)
{
    if (!a || (n > 0 && (!seqs || !slots || !cow_pairs)) || !num_pairs)
        return pkv_fail(PKV_ERR_NULL, "pkv_step_append: NULL argument");
    if (n < 0) return pkv_fail(PKV_ERR_SHAPE, "pkv_step_append: n < 0");
    // plan first (all or nothing), then commit
    int64_t need = 0;
    const int rc = plan_step(a, seqs, n, "pkv_step_append", 0, &need);
    if (rc != PKV_OK) return rc;
    int np = 0;
    for (int i = 0; i < n; ++i) {
        int64_t src, dst;
        a->append_one(*a->step_seqs[i], &slots[i], &src, &dst);
        if (src >= 0) {
            cow_pairs[2 * np] = src;
            cow_pairs[2 * np + 1] = dst;
            ++np;
        }
    }
    *num_pairs = np;
    return PKV_OK;
}

int pkv_step_append_tables(pkv_allocator* a, const int64_t* seqs, int n, int64_t* slots,
                           int64_t* cow_pairs, int* num_pairs, int32_t* tables, int max_blocks,
                           int32_t* lens)
{
    static const char* fn = "pkv_step_append_tables";
    if (!a || (n > 0 && (!seqs || !slots || !cow_pairs || !tables || !lens)) || !num_pairs)
        return pkv_fail(PKV_ERR_NULL, "%s: NULL argument", fn);
    if (n < 0 || max_blocks <= 0) return pkv_fail(PKV_ERR_SHAPE, "%s: n %d, max_blocks %d", fn, n,
                                                  max_blocks);
    int64_t need = 0;
    const int rc = plan_step(a, seqs, n, fn, max_blocks, &need);
    if (rc != PKV_OK) return rc;
    int np = 0;
    for (int i = 0; i < n; ++i) {
        pkv_allocator::Seq& s = *a->step_seqs[i];
        int64_t src, dst;
        a->append_one(s, &slots[i], &src, &dst);
        if (src >= 0) {
            cow_pairs[2 * np] = src;
            cow_pairs[2 * np + 1] = dst;
            ++np;
        }
        // the entries this append can change: the token's block (new, or the
        // copy that replaced a shared one), and the length
        const int64_t e = (s.len - 1) / a->block_size;
        tables[(size_t)i * max_blocks + e] = s.table[e];
        lens[i] = (int32_t)s.len;
    }
    *num_pairs = np;
    return PKV_OK;
}

int pkv_seq_fork(pkv_allocator* a, int64_t parent, int64_t child)
{
    if (!a) return pkv_fail(PKV_ERR_NULL, "pkv_seq_fork: allocator is NULL");
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end()) return pkv_fail(PKV_ERR_STATE, "pkv_seq_fork: unknown parent");
    if (a->seqs.count(child)) return pkv_fail(PKV_ERR_STATE, "pkv_seq_fork: child exists");
    pkv_allocator::Seq s = it->second;
    for (int32_t b : s.table) a->ref[b] += 1;
    a->seqs.emplace(child, std::move(s));
    return PKV_OK;
}

int pkv_seq_free(pkv_allocator* a, int64_t seq)
{
    if (!a) return pkv_fail(PKV_ERR_NULL, "pkv_seq_free: allocator is NULL");
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return pkv_fail(PKV_ERR_STATE, "pkv_seq_free: unknown sequence");
    const std::vector<int32_t>& t = it->second.table;
    for (size_t i = t.size(); i-- > 0;) a->release(t[i]);
    a->seqs.erase(it);
    return PKV_OK;
}

int pkv_seq_swap(pkv_allocator* from, pkv_allocator* to, int64_t seq, int64_t* pairs, int cap,
                 int* num_pairs)
{
    if (!from || !to || !num_pairs) return pkv_fail(PKV_ERR_NULL, "pkv_seq_swap: NULL argument");
    if (from == to) return pkv_fail(PKV_ERR_STATE, "pkv_seq_swap: same allocator");
    if (from->block_size != to->block_size)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_seq_swap: block sizes differ");
    auto it = from->seqs.find(seq);
    if (it == from->seqs.end()) return pkv_fail(PKV_ERR_STATE, "pkv_seq_swap: unknown sequence");
    if (to->seqs.count(seq)) return pkv_fail(PKV_ERR_STATE, "pkv_seq_swap: sequence exists");
    const std::vector<int32_t>& t = it->second.table;
    const int n = (int)t.size();
    if (n > 0 && !pairs) return pkv_fail(PKV_ERR_NULL, "pkv_seq_swap: pairs is NULL");
    if (n > cap) return pkv_fail(PKV_ERR_SHAPE, "pkv_seq_swap: %d pairs, cap %d", n, cap);
    if (n > (int)to->available())
        return pkv_fail(PKV_ERR_OOM, "pkv_seq_swap: %d blocks needed, %zu free", n,
                        to->available());
    pkv_allocator::Seq moved;
    moved.len = it->second.len;
    moved.table.reserve(n);
    for (int i = 0; i < n; ++i) {
        const int32_t b = to->pop();
        moved.table.push_back(b);
        pairs[2 * i] = t[i];
        pairs[2 * i + 1] = b;
    }
    for (int i = n; i-- > 0;) from->release(t[i]);
    from->seqs.erase(it);
    to->seqs.emplace(seq, std::move(moved));
    *num_pairs = n;
    return PKV_OK;
}

int pkv_seq_add_cached(pkv_allocator* a, int64_t seq, const int32_t* tokens, int n,
                       int* reused_tokens)
{
    if (!a || !reused_tokens || (n > 0 && !tokens))
        return pkv_fail(PKV_ERR_NULL, "pkv_seq_add_cached: NULL argument");
    if (n < 0) return pkv_fail(PKV_ERR_SHAPE, "pkv_seq_add_cached: negative length");
    if (a->seqs.count(seq)) return pkv_fail(PKV_ERR_STATE, "pkv_seq_add_cached: sequence exists");
    const int B = a->block_size;
    const int64_t nblocks = (n + (int64_t)B - 1) / B;
    // the longest chain of cached full blocks matching the prompt
    std::vector<int32_t> hits;
    uint64_t parent = 0;
    int64_t revive = 0;
    for (int64_t i = 0; i < n / B; ++i) {
        const uint64_t k = block_key(parent, tokens + i * B, B);
        const int32_t b = a->lookup(k, parent, tokens + i * B);
        if (b < 0) break;
        hits.push_back(b);
        if (a->ref[b] == 0) ++revive;
        parent = k;
    }
    const int64_t fresh = nblocks - (int64_t)hits.size();
    if (fresh > (int64_t)a->available() - revive)
        return pkv_fail(PKV_ERR_OOM, "pkv_seq_add_cached: %lld blocks needed, %zu free",
                        (long long)fresh, a->available() - (size_t)revive);
    pkv_allocator::Seq s;
    s.table.reserve(nblocks);
    for (int32_t b : hits) {
        a->take(b);
        s.table.push_back(b);
    }
    for (int64_t i = 0; i < fresh; ++i) s.table.push_back(a->pop());
    s.len = n;
    a->seqs.emplace(seq, std::move(s));
    a->prefix_hits += (int64_t)hits.size();
    *reused_tokens = (int)hits.size() * B;
    return PKV_OK;
}

int pkv_seq_register_blocks(pkv_allocator* a, int64_t seq, const int32_t* tokens, int n,
                            int* registered)
{
    if (!a || !registered || (n > 0 && !tokens))
        return pkv_fail(PKV_ERR_NULL, "pkv_seq_register_blocks: NULL argument");
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end())
        return pkv_fail(PKV_ERR_STATE, "pkv_seq_register_blocks: unknown sequence");
    if (n < 0 || n > it->second.len)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_seq_register_blocks: %d tokens, sequence holds %lld",
                        n, (long long)it->second.len);
    const int B = a->block_size;
    const std::vector<int32_t>& t = it->second.table;
    uint64_t parent = 0;
    int added = 0;
    for (int i = 0; i < n / B; ++i) {
        const uint64_t k = block_key(parent, tokens + (size_t)i * B, B);
        const int32_t b = t[i];
        if (!a->registered[b] && a->index.find(k) == a->index.end()) {
            a->index.emplace(k, b);
            a->registered[b] = 1;
            a->key[b] = k;
            a->parent_key[b] = parent;
            std::memcpy(&a->tokens[(size_t)b * B], tokens + (size_t)i * B, sizeof(int32_t) * B);
            ++added;
        }
        parent = k;
    }
    *registered = added;
    return PKV_OK;
}

int pkv_prefix_cache_stats(pkv_allocator* a, int64_t* hit_blocks, int64_t* cached_blocks,
                           int64_t* cached_free_blocks)
{
    if (!a || !hit_blocks || !cached_blocks || !cached_free_blocks)
        return pkv_fail(PKV_ERR_NULL, "pkv_prefix_cache_stats: NULL argument");
    *hit_blocks = a->prefix_hits;
    *cached_blocks = (int64_t)a->index.size();
    *cached_free_blocks = (int64_t)a->cached_free.size();
    return PKV_OK;
}

int pkv_seq_len(pkv_allocator* a, int64_t seq, int* len)
{
    if (!a || !len) return pkv_fail(PKV_ERR_NULL, "pkv_seq_len: NULL argument");
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return pkv_fail(PKV_ERR_STATE, "pkv_seq_len: unknown sequence");
    *len = (int)it->second.len;
    return PKV_OK;
}

int pkv_block_table(pkv_allocator* a, int64_t seq, int32_t* out, int cap, int* n)
{
    if (!a || !n || (cap > 0 && !out)) return pkv_fail(PKV_ERR_NULL, "pkv_block_table: NULL");
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return pkv_fail(PKV_ERR_STATE, "pkv_block_table: unknown sequence");
    const std::vector<int32_t>& t = it->second.table;
    *n = (int)t.size();
    int m = cap < (int)t.size() ? cap : (int)t.size();
    if (m > 0) std::memcpy(out, t.data(), sizeof(int32_t) * m);
    if ((int)t.size() > cap)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_block_table: table has %zu entries, cap %d",
                        t.size(), cap);
    return PKV_OK;
}

int pkv_block_tables_dense(pkv_allocator* a, const int64_t* seqs, int n, int max_blocks,
                           int32_t* tables, int32_t* lens)
{
    if (!a || (n > 0 && (!seqs || !tables || !lens)))
        return pkv_fail(PKV_ERR_NULL, "pkv_block_tables_dense: NULL argument");
    if (n < 0 || max_blocks < 0) return pkv_fail(PKV_ERR_SHAPE, "pkv_block_tables_dense: sizes");
    for (int i = 0; i < n; ++i) {
        auto it = a->seqs.find(seqs[i]);
        if (it == a->seqs.end())
            return pkv_fail(PKV_ERR_STATE, "pkv_block_tables_dense: unknown sequence");
        if ((int64_t)it->second.table.size() > max_blocks)
            return pkv_fail(PKV_ERR_SHAPE, "pkv_block_tables_dense: table longer than %d",
                            max_blocks);
    }
    for (int i = 0; i < n; ++i) {
        const pkv_allocator::Seq& s = a->seqs.find(seqs[i])->second;
        int32_t* row = tables + (size_t)i * max_blocks;
        size_t k = s.table.size();
        if (k) std::memcpy(row, s.table.data(), sizeof(int32_t) * k);
        for (size_t j = k; j < (size_t)max_blocks; ++j) row[j] = -1;
        lens[i] = (int32_t)s.len;
    }
    return PKV_OK;
}

int pkv_refcount(pkv_allocator* a, int block, int* count)
{
    if (!a || !count) return pkv_fail(PKV_ERR_NULL, "pkv_refcount: NULL argument");
    if (block < 0 || block >= a->num_blocks)
        return pkv_fail(PKV_ERR_SHAPE, "pkv_refcount: block %d out of range", block);
    *count = a->ref[block];
    return PKV_OK;
}

int pkv_num_free_blocks(pkv_allocator* a, int* n)
{
    if (!a || !n) return pkv_fail(PKV_ERR_NULL, "pkv_num_free_blocks: NULL argument");
    *n = (int)a->available();
    return PKV_OK;
}

int pkv_stats(pkv_allocator* a, int64_t* allocated_positions, int64_t* valid_positions,
              int64_t* blocks_in_use)
{
    if (!a || !allocated_positions || !valid_positions || !blocks_in_use)
        return pkv_fail(PKV_ERR_NULL, "pkv_stats: NULL argument");
    int64_t alloc = 0, valid = 0;
    for (const auto& kv : a->seqs) {
        alloc += (int64_t)kv.second.table.size() * a->block_size;
        valid += kv.second.len;
    }
    *allocated_positions = alloc;
    *valid_positions = valid;
    *blocks_in_use = (int64_t)a->num_blocks - (int64_t)a->available();
    return PKV_OK;
}

}  // extern "C"
