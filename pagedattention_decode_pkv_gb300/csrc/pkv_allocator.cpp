// Host block allocator: who owns which physical block of the paged KV pool.
//
// "Paged KV Cache - AI infra interview lesson":
//   - Walk the Shapes First: the slot of position p is
//     block_table[p // bs] * bs + p % bs, and a sequence needs a new block
//     exactly at the step where its length becomes 1 mod bs.
//   - Append slots during decode; Separate allocation, sharing and release: a
//     physical block goes from free to allocated to shared and returns to the
//     free pool only after its final reference is released.
// "Chapter 2 -- KV cache, memory hierarchy, continuous batching, and
// PagedAttention", Deterministic evals for this layer (Accounting, Lifecycle):
// free + allocated = pool; allocated >= blocks referenced by live block
// tables; no two writable logical blocks alias.
//
// Policy: the lowest-numbered free block is handed out first, so traces are
// deterministic.  Sharing (fork) covers whole blocks only, so the block a
// sequence appends into is always its own.
#include <climits>
#include <cstdint>
#include <map>
#include <mutex>
#include <new>
#include <set>
#include <vector>

#include "pkv_internal.h"

struct pkv_block_allocator {
    int32_t num_blocks = 0, block_size = 0;
    std::vector<int32_t> refcount;  // table entries that reference each block
    std::set<int32_t> free_blocks;  // refcount 0, ordered: lowest first
    struct Seq {
        std::vector<int32_t> blocks;
        int64_t len = 0;
    };
    std::map<int64_t, Seq> seqs;
    std::mutex mu;
};

using namespace pkv;

namespace {

int64_t blocks_for(int64_t tokens, int32_t bs) { return (tokens + bs - 1) / bs; }

// Takes n free blocks (lowest first) or none.
bool take(pkv_block_allocator *a, int64_t n, std::vector<int32_t> &out) {
    if (n > static_cast<int64_t>(a->free_blocks.size())) return false;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = *a->free_blocks.begin();
        a->free_blocks.erase(a->free_blocks.begin());
        a->refcount[b] = 1;
        out.push_back(b);
    }
    return true;
}

void drop(pkv_block_allocator *a, int32_t b) {
    if (--a->refcount[b] == 0) a->free_blocks.insert(b);
}

}  // namespace

extern "C" pkv_status pkv_allocator_create(int32_t num_blocks, int32_t block_size, pkv_block_allocator **out) {
    if (!out || num_blocks < 0 || block_size <= 0 || static_cast<int64_t>(num_blocks) * block_size > INT32_MAX)
        return set_error(PKV_ERR_INVALID_ARG, "allocator: bad sizes (num_blocks=%d block_size=%d)", num_blocks,
                         block_size);
    auto *a = new (std::nothrow) pkv_block_allocator;
    if (!a) return set_error(PKV_ERR_INVALID_ARG, "allocator: out of host memory");
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->refcount.assign(num_blocks, 0);
    for (int32_t b = 0; b < num_blocks; ++b) a->free_blocks.insert(a->free_blocks.end(), b);
    *out = a;
    return ok();
}

extern "C" void pkv_allocator_destroy(pkv_block_allocator *a) { delete a; }

extern "C" pkv_status pkv_allocator_add_sequence(pkv_block_allocator *a, int64_t seq, int64_t num_tokens,
                                                 const int32_t *blocks) {
    if (!a || num_tokens < 0) return set_error(PKV_ERR_INVALID_ARG, "allocator: bad arguments");
    std::lock_guard<std::mutex> lock(a->mu);
    if (a->seqs.count(seq)) return set_error(PKV_ERR_INVALID_ARG, "allocator: sequence %lld exists", (long long)seq);
    const int64_t n = blocks_for(num_tokens, a->block_size);
    pkv_block_allocator::Seq s;
    s.len = num_tokens;
    if (blocks) {  // adopt the caller's blocks: each must be free and listed once
        std::set<int32_t> seen;
        for (int64_t i = 0; i < n; ++i) {
            const int32_t b = blocks[i];
            if (b < 0 || b >= a->num_blocks || a->refcount[b] != 0 || !seen.insert(b).second)
                return set_error(PKV_ERR_INVALID_ARG, "allocator: block %d is not free", b);
        }
        for (int64_t i = 0; i < n; ++i) {
            a->free_blocks.erase(blocks[i]);
            a->refcount[blocks[i]] = 1;
            s.blocks.push_back(blocks[i]);
        }
    } else if (!take(a, n, s.blocks)) {
        return set_error(PKV_ERR_OUT_OF_RANGE, "allocator: %lld blocks needed, %zu free", (long long)n,
                         a->free_blocks.size());
    }
    a->seqs.emplace(seq, std::move(s));
    return ok();
}

extern "C" pkv_status pkv_allocator_fork(pkv_block_allocator *a, int64_t parent, int64_t child,
                                         int64_t num_tokens) {
    if (!a) return set_error(PKV_ERR_INVALID_ARG, "allocator: NULL handle");
    std::lock_guard<std::mutex> lock(a->mu);
    auto it = a->seqs.find(parent);
    if (it == a->seqs.end()) return set_error(PKV_ERR_INVALID_ARG, "allocator: no sequence %lld", (long long)parent);
    if (a->seqs.count(child)) return set_error(PKV_ERR_INVALID_ARG, "allocator: sequence %lld exists", (long long)child);
    if (num_tokens < 0 || num_tokens > it->second.len || num_tokens % a->block_size)
        return set_error(PKV_ERR_INVALID_ARG, "allocator: a shared prefix is whole blocks of the parent (%lld tokens)",
                         (long long)num_tokens);
    pkv_block_allocator::Seq s;
    s.len = num_tokens;
    for (int64_t i = 0; i < num_tokens / a->block_size; ++i) {
        const int32_t b = it->second.blocks[i];
        ++a->refcount[b];
        s.blocks.push_back(b);
    }
    a->seqs.emplace(child, std::move(s));
    return ok();
}

extern "C" pkv_status pkv_allocator_append(pkv_block_allocator *a, int64_t seq, int64_t num_tokens, int32_t *slots) {
    if (!a || num_tokens < 0) return set_error(PKV_ERR_INVALID_ARG, "allocator: bad arguments");
    std::lock_guard<std::mutex> lock(a->mu);
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return set_error(PKV_ERR_INVALID_ARG, "allocator: no sequence %lld", (long long)seq);
    auto &s = it->second;
    const int32_t bs = a->block_size;
    const int64_t need = blocks_for(s.len + num_tokens, bs) - static_cast<int64_t>(s.blocks.size());
    std::vector<int32_t> fresh;
    if (need > 0 && !take(a, need, fresh))
        return set_error(PKV_ERR_OUT_OF_RANGE, "allocator: %lld blocks needed, %zu free", (long long)need,
                         a->free_blocks.size());
    s.blocks.insert(s.blocks.end(), fresh.begin(), fresh.end());
    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t p = s.len + i;
        if (slots) slots[i] = static_cast<int32_t>(static_cast<int64_t>(s.blocks[p / bs]) * bs + p % bs);
    }
    s.len += num_tokens;
    return ok();
}

extern "C" pkv_status pkv_allocator_release(pkv_block_allocator *a, int64_t seq) {
    if (!a) return set_error(PKV_ERR_INVALID_ARG, "allocator: NULL handle");
    std::lock_guard<std::mutex> lock(a->mu);
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return set_error(PKV_ERR_INVALID_ARG, "allocator: no sequence %lld", (long long)seq);
    for (int32_t b : it->second.blocks) drop(a, b);
    a->seqs.erase(it);
    return ok();
}

extern "C" pkv_status pkv_allocator_block_table(pkv_block_allocator *a, int64_t seq, int32_t *row,
                                                int32_t max_blocks, int64_t *num_tokens, int32_t *num_used) {
    if (!a || max_blocks < 0 || (max_blocks > 0 && !row))
        return set_error(PKV_ERR_INVALID_ARG, "allocator: bad arguments");
    std::lock_guard<std::mutex> lock(a->mu);
    auto it = a->seqs.find(seq);
    if (it == a->seqs.end()) return set_error(PKV_ERR_INVALID_ARG, "allocator: no sequence %lld", (long long)seq);
    const auto &s = it->second;
    if (static_cast<int64_t>(s.blocks.size()) > max_blocks)
        return set_error(PKV_ERR_OUT_OF_RANGE, "allocator: sequence %lld holds %zu blocks, row has %d",
                         (long long)seq, s.blocks.size(), max_blocks);
    for (int32_t i = 0; i < max_blocks; ++i) row[i] = i < static_cast<int32_t>(s.blocks.size()) ? s.blocks[i] : -1;
    if (num_tokens) *num_tokens = s.len;
    if (num_used) *num_used = static_cast<int32_t>(s.blocks.size());
    return ok();
}

extern "C" pkv_status pkv_allocator_stats(pkv_block_allocator *a, int64_t *free_blocks, int64_t *allocated_blocks,
                                          int64_t *referenced_blocks, int64_t *num_seqs) {
    if (!a) return set_error(PKV_ERR_INVALID_ARG, "allocator: NULL handle");
    std::lock_guard<std::mutex> lock(a->mu);
    std::set<int32_t> referenced;
    for (const auto &kv : a->seqs) referenced.insert(kv.second.blocks.begin(), kv.second.blocks.end());
    int64_t allocated = 0;
    for (int32_t r : a->refcount) allocated += r > 0;
    if (free_blocks) *free_blocks = static_cast<int64_t>(a->free_blocks.size());
    if (allocated_blocks) *allocated_blocks = allocated;
    if (referenced_blocks) *referenced_blocks = static_cast<int64_t>(referenced.size());
    if (num_seqs) *num_seqs = static_cast<int64_t>(a->seqs.size());
    return ok();
}

extern "C" int32_t pkv_allocator_check(pkv_block_allocator *a) {
    if (!a) return -1;
    std::lock_guard<std::mutex> lock(a->mu);
    const int32_t bs = a->block_size;
    std::vector<int32_t> refs(a->num_blocks, 0);
    for (const auto &kv : a->seqs) {
        const auto &s = kv.second;
        if (static_cast<int64_t>(s.blocks.size()) != blocks_for(s.len, bs)) return 5;  // table covers the length
        for (int32_t b : s.blocks) {
            if (b < 0 || b >= a->num_blocks) return 5;
            ++refs[b];
        }
    }
    int64_t allocated = 0;
    for (int32_t b = 0; b < a->num_blocks; ++b) {
        const bool is_free = a->free_blocks.count(b) != 0;
        if (a->refcount[b] != refs[b]) return 2;  // reference counts = live table entries
        if (is_free == (refs[b] > 0)) return 3;   // a block is free exactly when nothing references it
        allocated += refs[b] > 0;
    }
    if (static_cast<int64_t>(a->free_blocks.size()) + allocated != a->num_blocks) return 1;  // free + allocated = pool
    for (const auto &kv : a->seqs) {  // the block a sequence writes next is its own
        const auto &s = kv.second;
        if (s.len % bs != 0 && refs[s.blocks.back()] != 1) return 4;
    }
    return 0;
}
