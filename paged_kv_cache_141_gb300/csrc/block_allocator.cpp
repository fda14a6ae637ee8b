// block_allocator.cpp -- the host-side block allocator of the paged KV cache:
// a free list of physical block ids with reference counts.
//
//  * Blocks are handed out from the end of the free list, ceil(tokens / B) at
//    a time, all or nothing ("TGI PagedAttention deep-dive" (lpnh.cn)
//    sec. 4.3: SimpleAllocator takes div_ceil(tokens, block_size) blocks from
//    the end of free_blocks; block 0 is reserved for health checks; "Lecture
//    3: PagedAttention and vLLM", "Core data structure: Block Table": raise
//    when there are too few free blocks).
//  * fork adds a reference to blocks another sequence already holds, so that
//    sequences share them by reference; free drops one reference and returns a
//    block to the free list at zero ("Continuous Batching and PagedAttention"
//    sec. 3.2, PagedKVCache.fork / free with ref_counts).
//  * append_slot gives the slot of a sequence's next token: a new block when
//    the token starts one, and copy-on-write when the token would land in a
//    block someone else still references -- a fresh block replaces it in the
//    sequence's table and the caller copies the old block's contents before
//    writing ("vLLM Page Attention Continuous Batching" (lbrq.cn), "Sharing KV
//    Cache-COW": a branch appending to a block with ref_count > 1 gets a new
//    block with the old contents copied, the old block stays with the other
//    branch).
// All operations validate first and change nothing when they fail. A mutex
// makes each call atomic with respect to the others.
#include <climits>
#include <mutex>
#include <new>
#include <vector>

#include "pagedkv.h"

struct pa_block_allocator {
    int64_t num_blocks = 0;
    int block_size = 0;
    int64_t first = 0;                 // 1 when block 0 is reserved
    std::vector<int32_t> free_list;    // taken from the back
    std::vector<int32_t> refs;         // references per block; 0 = free
    std::mutex mu;
};

extern "C" {

pa_block_allocator* pa_allocator_create(int64_t num_blocks, int block_size, int reserve_block0) {
    if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
    pa_block_allocator* a = new (std::nothrow) pa_block_allocator();
    if (!a) return nullptr;
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->first = reserve_block0 ? 1 : 0;
    a->refs.assign((size_t)num_blocks, 0);
    // the back of the list is handed out first: lowest ids first
    for (int64_t b = num_blocks - 1; b >= a->first; --b) a->free_list.push_back((int32_t)b);
    return a;
}

void pa_allocator_destroy(pa_block_allocator* a) { delete a; }

int64_t pa_allocator_num_free(pa_block_allocator* a) {
    if (!a) return -1;
    std::lock_guard<std::mutex> g(a->mu);
    return (int64_t)a->free_list.size();
}

int32_t pa_allocator_refcount(pa_block_allocator* a, int32_t block) {
    if (!a || block < 0 || block >= a->num_blocks) return -1;
    std::lock_guard<std::mutex> g(a->mu);
    return a->refs[(size_t)block];
}

pa_status pa_allocator_allocate(pa_block_allocator* a, int64_t num_tokens, int32_t* blocks,
                                int64_t capacity, int64_t* num_allocated) {
    if (!a || num_tokens < 0 || (num_tokens > 0 && !blocks) || !num_allocated)
        return PA_ERR_INVALID_ARG;
    const int64_t n = (num_tokens + a->block_size - 1) / a->block_size;
    if (n > capacity) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(a->mu);
    if ((int64_t)a->free_list.size() < n) return PA_ERR_NO_BLOCKS;
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = a->free_list.back();
        a->free_list.pop_back();
        a->refs[(size_t)b] = 1;
        blocks[i] = b;
    }
    *num_allocated = n;
    return PA_OK;
}

static bool held_all(const pa_block_allocator* a, const int32_t* blocks, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = blocks[i];
        if (b < a->first || b >= a->num_blocks || a->refs[(size_t)b] <= 0) return false;
    }
    return true;
}

pa_status pa_allocator_fork(pa_block_allocator* a, const int32_t* blocks, int64_t n) {
    if (!a || n < 0 || (n > 0 && !blocks)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(a->mu);
    if (!held_all(a, blocks, n)) return PA_ERR_INVALID_ARG;
    for (int64_t i = 0; i < n; ++i) a->refs[(size_t)blocks[i]] += 1;
    return PA_OK;
}

pa_status pa_allocator_free(pa_block_allocator* a, const int32_t* blocks, int64_t n) {
    if (!a || n < 0 || (n > 0 && !blocks)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(a->mu);
    // a block listed k times must hold at least k references
    std::vector<int32_t> drop;
    drop.reserve((size_t)n);
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = blocks[i];
        if (b < a->first || b >= a->num_blocks) return PA_ERR_INVALID_ARG;
        drop.push_back(b);
    }
    std::vector<int32_t> count;
    for (int32_t b : drop) {
        if ((size_t)b >= count.size()) count.resize((size_t)b + 1, 0);
        if (++count[(size_t)b] > a->refs[(size_t)b]) return PA_ERR_INVALID_ARG;
    }
    for (int32_t b : drop) {
        if (--a->refs[(size_t)b] == 0) a->free_list.push_back(b);
    }
    return PA_OK;
}

pa_status pa_allocator_append_slot(pa_block_allocator* a, int32_t* table, int64_t* table_len,
                                   int64_t capacity, int64_t position, int64_t* slot,
                                   int32_t* copy_src, int32_t* copy_dst) {
    if (!a || !table || !table_len || !slot || !copy_src || !copy_dst || position < 0)
        return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(a->mu);
    const int64_t B = a->block_size;
    const int64_t len = *table_len;
    const int64_t j = position / B;
    if (len < 0 || len > capacity || j > len || (j == len && position % B != 0))
        return PA_ERR_INVALID_ARG;             // positions are appended in order
    if (!held_all(a, table, len)) return PA_ERR_INVALID_ARG;
    *copy_src = -1;
    *copy_dst = -1;
    if (j == len) {                            // the token starts a new block
        if (len == capacity) return PA_ERR_INVALID_ARG;
        if (a->free_list.empty()) return PA_ERR_NO_BLOCKS;
        const int32_t b = a->free_list.back();
        a->free_list.pop_back();
        a->refs[(size_t)b] = 1;
        table[len] = b;
        *table_len = len + 1;
    } else if (a->refs[(size_t)table[j]] > 1) {  // shared: copy on write
        if (a->free_list.empty()) return PA_ERR_NO_BLOCKS;
        const int32_t old = table[j];
        const int32_t b = a->free_list.back();
        a->free_list.pop_back();
        a->refs[(size_t)b] = 1;
        a->refs[(size_t)old] -= 1;
        table[j] = b;
        *copy_src = old;
        *copy_dst = b;
    }
    *slot = (int64_t)table[j] * B + position % B;
    return PA_OK;
}

}  // extern "C"
