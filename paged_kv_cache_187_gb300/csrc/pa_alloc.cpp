// pa_alloc.cpp -- the host block allocator of the C ABI (include/pa.h, pa_alloc_*).
//
// The v2 block manager of "[core] Multi Step Scheduling #7000" hands out the physical
// blocks of the KV pool and produces the decode metadata (block_tables, slot_mapping,
// seq_lens); "vLLM Project Update" describes the KV cache managed like virtual-memory
// pages, with blocks shared between requests (prefix caching).  The written spec both
// this file and the test oracle follow:
//   1. Physical ids 0..num_blocks-1 are shuffled by Fisher-Yates (i from num_blocks-1
//      down to 1, j = r % (i + 1), r the next splitmix64 output seeded with `seed`).
//   2. The shuffled array is the free list; blocks are popped from its end.
//   3. add_seq(id, n) pops ceil(n / block_size) blocks, in logical order.
//   4. append(id) pops one block first when position len has no block yet, then
//      returns the slot of position len and increments len.
//   5. free_seq(id) drops the sequence's reference to each of its blocks, in logical
//      order; a block whose count reaches 0 is pushed back on the free list.
//   6. A request that needs more blocks than are free fails and changes nothing.
//   7. Every block has a reference count; a popped block starts at 1.
//   8. fork(src, dst, n) makes dst live with length n <= len(src) and the first
//      ceil(n / block_size) blocks of src, each count + 1; nothing is popped.
//   9. Copy-on-write: before append (or reserve with extra > 0) writes position len into
//      a block whose count is > 1, it pops a new block, records (old, new) as a pending
//      copy, puts the new block in the table and decrements the old block's count.
//  10. take_copies returns the pending pairs in order and clears them.
//  11. reserve(id, extra) pops blocks until the sequence owns ceil((len + extra) /
//      block_size) of them (after rule 9); len does not change.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "../../include/pa.h"
#include "pa_internal.h"

struct pa_alloc {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    std::vector<int32_t> free_list;   // popped from the back
    std::vector<int32_t> refcount;    // per physical block
    std::vector<int32_t> copies;      // pending copy-on-write pairs (old, new)
    struct Seq {
        std::vector<int32_t> blocks;
        int32_t len = 0;
    };
    std::unordered_map<int32_t, Seq> seqs;
};

namespace {

pa_status fail(pa_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    return (pa_status)pa::set_last_error(st, buf);
}

pa_status ok() { return (pa_status)pa::set_last_error(PA_OK, ""); }

// splitmix64 (Steele, Lea and Flood, OOPSLA 2014).
uint64_t splitmix64(uint64_t& s) {
    s += 0x9E3779B97F4A7C15ull;
    uint64_t z = s;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

int32_t pop_block(pa_alloc* a) {
    const int32_t b = a->free_list.back();
    a->free_list.pop_back();
    a->refcount[b] = 1;
    return b;
}

// Rule 9: does writing position len of s hit a shared block?
bool needs_cow(const pa_alloc* a, const pa_alloc::Seq& s) {
    const size_t logical = (size_t)(s.len / a->block_size);
    return logical < s.blocks.size() && a->refcount[s.blocks[logical]] > 1;
}

void copy_on_write(pa_alloc* a, pa_alloc::Seq& s) {
    const size_t logical = (size_t)(s.len / a->block_size);
    const int32_t old = s.blocks[logical];
    const int32_t fresh = pop_block(a);
    a->refcount[old] -= 1;
    s.blocks[logical] = fresh;
    a->copies.push_back(old);
    a->copies.push_back(fresh);
}

// Blocks one append to s needs from the free list (a new block, or a private copy).
int32_t append_need(const pa_alloc* a, const pa_alloc::Seq& s) {
    if ((size_t)(s.len / a->block_size) >= s.blocks.size()) return 1;
    return needs_cow(a, s) ? 1 : 0;
}

void append_one(pa_alloc* a, pa_alloc::Seq& s, int32_t* slot_out) {
    if ((size_t)(s.len / a->block_size) >= s.blocks.size()) s.blocks.push_back(pop_block(a));
    else if (needs_cow(a, s)) copy_on_write(a, s);
    *slot_out = s.blocks[s.len / a->block_size] * a->block_size + s.len % a->block_size;
    s.len += 1;
}

}  // namespace

extern "C" {

pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size, uint64_t seed, pa_alloc** out) {
    if (!out) return fail(PA_ERR_INVALID_ARG, "alloc_create: null output");
    *out = nullptr;
    if (num_blocks <= 0 || block_size <= 0)
        return fail(PA_ERR_INVALID_ARG, "alloc_create: num_blocks and block_size must be positive");
    if ((int64_t)num_blocks * block_size > INT32_MAX)
        return fail(PA_ERR_INVALID_ARG, "alloc_create: num_blocks * block_size overflows int32 slots");
    auto* a = new pa_alloc;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->free_list.resize(num_blocks);
    a->refcount.assign(num_blocks, 0);
    for (int32_t i = 0; i < num_blocks; ++i) a->free_list[i] = i;
    uint64_t st = seed;
    for (int32_t i = num_blocks - 1; i >= 1; --i) {
        const int32_t j = (int32_t)(splitmix64(st) % (uint64_t)(i + 1));
        std::swap(a->free_list[i], a->free_list[j]);
    }
    *out = a;
    return ok();
}

void pa_alloc_destroy(pa_alloc* a) { delete a; }

int32_t pa_alloc_num_free(const pa_alloc* a) { return a ? (int32_t)a->free_list.size() : 0; }

pa_status pa_alloc_add_seq(pa_alloc* a, int32_t seq_id, int32_t num_tokens) {
    if (!a || seq_id < 0 || num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "alloc_add_seq: bad args");
    if (a->seqs.count(seq_id)) return fail(PA_ERR_INVALID_ARG, "alloc_add_seq: seq %d is live", seq_id);
    const int64_t need = ((int64_t)num_tokens + a->block_size - 1) / a->block_size;
    if (need > (int64_t)a->free_list.size())
        return fail(PA_ERR_NO_BLOCKS, "alloc_add_seq: need %lld blocks, %zu free", (long long)need,
                    a->free_list.size());
    pa_alloc::Seq s;
    s.len = num_tokens;
    s.blocks.reserve(need);
    for (int64_t i = 0; i < need; ++i) s.blocks.push_back(pop_block(a));
    a->seqs.emplace(seq_id, std::move(s));
    return ok();
}

pa_status pa_alloc_fork(pa_alloc* a, int32_t src_seq, int32_t dst_seq, int32_t num_tokens) {
    if (!a || dst_seq < 0 || num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "alloc_fork: bad args");
    auto it = a->seqs.find(src_seq);
    if (it == a->seqs.end()) return fail(PA_ERR_INVALID_ARG, "alloc_fork: unknown seq %d", src_seq);
    if (a->seqs.count(dst_seq)) return fail(PA_ERR_INVALID_ARG, "alloc_fork: seq %d is live", dst_seq);
    if (num_tokens > it->second.len)
        return fail(PA_ERR_INVALID_ARG, "alloc_fork: %d tokens > length %d of seq %d", num_tokens,
                    it->second.len, src_seq);
    const int32_t nb = (num_tokens + a->block_size - 1) / a->block_size;
    pa_alloc::Seq d;
    d.len = num_tokens;
    d.blocks.assign(it->second.blocks.begin(), it->second.blocks.begin() + nb);
    for (int32_t b : d.blocks) a->refcount[b] += 1;
    a->seqs.emplace(dst_seq, std::move(d));
    return ok();
}

pa_status pa_alloc_append(pa_alloc* a, int32_t seq_id, int32_t* slot_out) {
    if (!a || !slot_out) return fail(PA_ERR_INVALID_ARG, "alloc_append: null argument");
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return fail(PA_ERR_INVALID_ARG, "alloc_append: unknown seq %d", seq_id);
    if (append_need(a, it->second) > (int32_t)a->free_list.size())
        return fail(PA_ERR_NO_BLOCKS, "alloc_append: no free block");
    append_one(a, it->second, slot_out);
    return ok();
}

pa_status pa_alloc_append_batch(pa_alloc* a, const int32_t* seq_ids, int32_t n, int32_t* slots_out) {
    if (!a || n < 0 || (n > 0 && (!seq_ids || !slots_out)))
        return fail(PA_ERR_INVALID_ARG, "alloc_append_batch: bad args");
    int64_t need = 0;
    std::unordered_set<int32_t> seen;
    seen.reserve((size_t)n * 2);
    for (int32_t i = 0; i < n; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end())
            return fail(PA_ERR_INVALID_ARG, "alloc_append_batch: unknown seq %d", seq_ids[i]);
        if (!seen.insert(seq_ids[i]).second)
            return fail(PA_ERR_INVALID_ARG, "alloc_append_batch: seq %d listed twice", seq_ids[i]);
        need += append_need(a, it->second);
    }
    if (need > (int64_t)a->free_list.size())
        return fail(PA_ERR_NO_BLOCKS, "alloc_append_batch: need %lld blocks, %zu free",
                    (long long)need, a->free_list.size());
    for (int32_t i = 0; i < n; ++i) append_one(a, a->seqs[seq_ids[i]], &slots_out[i]);
    return ok();
}

pa_status pa_alloc_reserve_batch(pa_alloc* a, const int32_t* seq_ids, int32_t n,
                                 int32_t extra_tokens) {
    if (!a || n < 0 || extra_tokens < 0 || (n > 0 && !seq_ids))
        return fail(PA_ERR_INVALID_ARG, "alloc_reserve_batch: bad args");
    int64_t need = 0;
    for (int32_t i = 0; i < n; ++i) {
        auto it = a->seqs.find(seq_ids[i]);
        if (it == a->seqs.end())
            return fail(PA_ERR_INVALID_ARG, "alloc_reserve_batch: unknown seq %d", seq_ids[i]);
        const pa_alloc::Seq& s = it->second;
        const int64_t want = ((int64_t)s.len + extra_tokens + a->block_size - 1) / a->block_size;
        need += std::max<int64_t>(0, want - (int64_t)s.blocks.size());
        if (extra_tokens > 0 && needs_cow(a, s)) need += 1;
    }
    if (need > (int64_t)a->free_list.size())
        return fail(PA_ERR_NO_BLOCKS, "alloc_reserve_batch: need %lld blocks, %zu free",
                    (long long)need, a->free_list.size());
    for (int32_t i = 0; i < n; ++i) {
        pa_alloc::Seq& s = a->seqs[seq_ids[i]];
        if (extra_tokens > 0 && needs_cow(a, s)) copy_on_write(a, s);
        const int64_t want = ((int64_t)s.len + extra_tokens + a->block_size - 1) / a->block_size;
        while ((int64_t)s.blocks.size() < want) s.blocks.push_back(pop_block(a));
    }
    return ok();
}

int32_t pa_alloc_num_pending_copies(const pa_alloc* a) {
    return a ? (int32_t)(a->copies.size() / 2) : 0;
}

pa_status pa_alloc_take_copies(pa_alloc* a, int32_t* pairs_out, int32_t max_pairs, int32_t* n_out) {
    if (!a || !n_out || max_pairs < 0) return fail(PA_ERR_INVALID_ARG, "alloc_take_copies: bad args");
    const int32_t n = (int32_t)(a->copies.size() / 2);
    *n_out = n;
    if (n > max_pairs)
        return fail(PA_ERR_INVALID_ARG, "alloc_take_copies: %d pending pairs, room for %d", n,
                    max_pairs);
    if (n > 0 && !pairs_out) return fail(PA_ERR_INVALID_ARG, "alloc_take_copies: null output");
    std::copy(a->copies.begin(), a->copies.end(), pairs_out);
    a->copies.clear();
    return ok();
}

int32_t pa_alloc_refcount(const pa_alloc* a, int32_t block) {
    if (!a || block < 0 || block >= a->num_blocks) return -1;
    return a->refcount[block];
}

pa_status pa_alloc_free_seq(pa_alloc* a, int32_t seq_id) {
    if (!a) return fail(PA_ERR_INVALID_ARG, "alloc_free_seq: null handle");
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return fail(PA_ERR_INVALID_ARG, "alloc_free_seq: unknown seq %d", seq_id);
    for (int32_t b : it->second.blocks)
        if (--a->refcount[b] == 0) a->free_list.push_back(b);
    a->seqs.erase(it);
    return ok();
}

pa_status pa_alloc_slots(const pa_alloc* a, int32_t seq_id, int32_t start, int32_t n, int32_t* out) {
    if (!a || (n > 0 && !out) || start < 0 || n < 0) return fail(PA_ERR_INVALID_ARG, "alloc_slots: bad args");
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return fail(PA_ERR_INVALID_ARG, "alloc_slots: unknown seq %d", seq_id);
    const pa_alloc::Seq& s = it->second;
    if ((int64_t)start + n > s.len) return fail(PA_ERR_INVALID_ARG, "alloc_slots: past the sequence end");
    for (int32_t i = 0; i < n; ++i) {
        const int32_t t = start + i;
        out[i] = s.blocks[t / a->block_size] * a->block_size + t % a->block_size;
    }
    return ok();
}

pa_status pa_alloc_block_tables(const pa_alloc* a, const int32_t* seq_ids, int32_t n,
                                int32_t max_blocks_per_seq, int32_t* out) {
    if (!a || n < 0 || max_blocks_per_seq <= 0 || (n > 0 && (!seq_ids || !out)))
        return fail(PA_ERR_INVALID_ARG, "alloc_block_tables: bad args");
    for (int32_t r = 0; r < n; ++r) {
        auto it = a->seqs.find(seq_ids[r]);
        if (it == a->seqs.end())
            return fail(PA_ERR_INVALID_ARG, "alloc_block_tables: unknown seq %d", seq_ids[r]);
        const std::vector<int32_t>& b = it->second.blocks;
        if ((int64_t)b.size() > max_blocks_per_seq)
            return fail(PA_ERR_INVALID_ARG, "alloc_block_tables: seq %d has %zu blocks > %d",
                        seq_ids[r], b.size(), max_blocks_per_seq);
        int32_t* row = out + (size_t)r * max_blocks_per_seq;
        std::copy(b.begin(), b.end(), row);
        std::fill(row + b.size(), row + max_blocks_per_seq, -1);
    }
    return ok();
}

pa_status pa_alloc_context_lens(const pa_alloc* a, const int32_t* seq_ids, int32_t n, int32_t* out) {
    if (!a || n < 0 || (n > 0 && (!seq_ids || !out)))
        return fail(PA_ERR_INVALID_ARG, "alloc_context_lens: bad args");
    for (int32_t r = 0; r < n; ++r) {
        auto it = a->seqs.find(seq_ids[r]);
        if (it == a->seqs.end())
            return fail(PA_ERR_INVALID_ARG, "alloc_context_lens: unknown seq %d", seq_ids[r]);
        out[r] = it->second.len;
    }
    return ok();
}

}  // extern "C"
