// radix_allocator.cpp -- the prefix-caching block allocator: a radix trie from
// token sequences to the physical blocks that hold their K/V, so that a new
// request reuses the blocks of any cached prefix ("TGI PagedAttention
// deep-dive" (lpnh.cn) sec. 5.2-5.3, RadixAllocator).
//
//  * Keys and values have the same length at block granularity: a node holds
//    k * block_size tokens and the k blocks that hold them, so a cached
//    "abc" also answers "a" and "ab" (sec. 5.2). Only whole blocks are
//    shared: with block_size 2 a 5-token prompt caches 2 blocks (sec. 5.4).
//  * Every node counts the live allocations that use it (ref_count) and
//    remembers when it was last used; a node in use is never evicted.
//  * allocate: the longest cached block-aligned prefix of the prompt is found
//    (its nodes are touched and referenced before anything is evicted, so the
//    prefix cannot be evicted under the request), the rest of the request's
//    blocks come from the free list, evicting least-recently-used leaves with
//    no references when the list is short; prefix_len tokens need no
//    recomputation (sec. 5.3).
//  * free: the references are dropped and the request's token -> block
//    mapping is inserted into the trie; a node that only partly matches is
//    split at the block where the sequences part (split_node, sec. 5.2).
//    Blocks the trie does not take (a partial last block, a range another
//    request cached first) return to the free list.
// Every call validates first and changes nothing when it fails; a mutex
// serialises calls.
#include <algorithm>
#include <climits>
#include <map>
#include <mutex>
#include <new>
#include <set>
#include <unordered_map>
#include <vector>

#include "pagedkv.h"

namespace {

struct Node {
    std::vector<int32_t> key;                          // tokens, a multiple of block_size
    std::vector<int32_t> blocks;                       // key.size() / block_size
    Node* parent = nullptr;
    std::map<std::vector<int32_t>, Node*> children;    // by the child's first block of tokens
    int64_t refs = 0;
    uint64_t last = 0;                                 // logical time of the last use
    uint64_t id = 0;
    bool evictable = false;                            // listed in the LRU set
};

// A request holds one reference on every node of its prefix, i.e. on the
// deepest prefix node and all its ancestors. Only that node is stored: a
// later split inserts the new head between it and its parent, so walking up
// the parents still visits exactly the nodes that hold the reference.
struct Allocation {
    Node* last = nullptr;                              // deepest prefix node (null: no prefix)
    int64_t prefix_blocks = 0;
    std::vector<int32_t> prefix_tokens;                // the cached prefix it was given
    std::vector<int32_t> blocks;                       // prefix blocks, then owned ones
};

}  // namespace

struct pa_radix_allocator {
    int64_t num_blocks = 0;
    int B = 0;
    std::vector<int32_t> free_list;                    // taken from the back
    Node root;
    uint64_t clock = 0;
    uint64_t next_node = 1;
    int64_t next_alloc = 1;
    int64_t cached_blocks = 0;                         // blocks held by trie nodes
    std::set<std::pair<uint64_t, uint64_t>> lru;       // (last use, node id) of evictable leaves
    std::unordered_map<uint64_t, Node*> by_id;
    std::unordered_map<int64_t, Allocation> live;
    std::mutex mu;

    ~pa_radix_allocator() { destroy(&root); }

    void destroy(Node* n) {
        for (auto& kv : n->children) {
            destroy(kv.second);
            delete kv.second;
        }
        n->children.clear();
    }

    std::vector<int32_t> chunk(const int32_t* t) const { return std::vector<int32_t>(t, t + B); }

    // keep the LRU set in step with a node's state
    void refresh(Node* n) {
        if (n == &root) return;
        if (n->evictable) {
            lru.erase({n->last, n->id});
            n->evictable = false;
        }
        if (n->refs == 0 && n->children.empty()) {
            lru.insert({n->last, n->id});
            n->evictable = true;
        }
    }

    void touch(Node* n, uint64_t t) {
        if (n->evictable) lru.erase({n->last, n->id});
        n->last = t;
        if (n->evictable) lru.insert({n->last, n->id});
    }

    Node* new_node(Node* parent, std::vector<int32_t> key, std::vector<int32_t> blocks, uint64_t t) {
        Node* n = new Node();
        n->key = std::move(key);
        n->blocks = std::move(blocks);
        n->parent = parent;
        n->last = t;
        n->id = next_node++;
        by_id[n->id] = n;
        parent->children[chunk(n->key.data())] = n;
        cached_blocks += (int64_t)n->blocks.size();
        refresh(n);
        refresh(parent);
        return n;
    }

    // Split n after its first m blocks (0 < m < blocks): the head becomes a
    // new parent that inherits n's references and time.
    Node* split(Node* n, size_t m) {
        Node* parent = n->parent;
        Node* head = new Node();
        head->key.assign(n->key.begin(), n->key.begin() + (ptrdiff_t)(m * B));
        head->blocks.assign(n->blocks.begin(), n->blocks.begin() + (ptrdiff_t)m);
        head->parent = parent;
        head->refs = n->refs;
        head->last = n->last;
        head->id = next_node++;
        by_id[head->id] = head;
        parent->children[chunk(head->key.data())] = head;   // same first block as n had
        n->key.erase(n->key.begin(), n->key.begin() + (ptrdiff_t)(m * B));
        n->blocks.erase(n->blocks.begin(), n->blocks.begin() + (ptrdiff_t)m);
        n->parent = head;
        head->children[chunk(n->key.data())] = n;
        refresh(head);
        refresh(n);
        return head;
    }

    // Walk the longest cached block-aligned prefix of tokens[0, n_blocks*B):
    // full nodes are appended to path; a last node matched only in part is
    // split so that the path ends on a node boundary.
    void match(const int32_t* tokens, int64_t n_blocks, std::vector<Node*>& path) {
        Node* node = &root;
        int64_t i = 0;
        while (i < n_blocks) {
            auto it = node->children.find(chunk(tokens + i * B));
            if (it == node->children.end()) break;
            Node* child = it->second;
            size_t m = 1;
            const size_t nb = child->blocks.size();
            while (m < nb && i + (int64_t)m < n_blocks &&
                   std::equal(tokens + (i + (int64_t)m) * B, tokens + (i + (int64_t)m + 1) * B,
                              child->key.begin() + (ptrdiff_t)(m * B)))
                ++m;
            if (m < nb) child = split(child, m);
            path.push_back(child);
            i += (int64_t)m;
            node = child;
        }
    }

    // drop one reference from n and each of its ancestors
    void release(Node* n) {
        for (; n && n != &root; n = n->parent) {
            n->refs -= 1;
            refresh(n);
        }
    }

    void evict_one() {
        auto it = lru.begin();
        Node* n = by_id[it->second];
        lru.erase(it);
        n->evictable = false;
        for (int32_t b : n->blocks) free_list.push_back(b);
        cached_blocks -= (int64_t)n->blocks.size();
        Node* parent = n->parent;
        parent->children.erase(chunk(n->key.data()));
        by_id.erase(n->id);
        delete n;
        refresh(parent);
    }
};

extern "C" {

pa_radix_allocator* pa_radix_create(int64_t num_blocks, int block_size, int reserve_block0) {
    if (num_blocks <= 0 || num_blocks > INT32_MAX || block_size <= 0) return nullptr;
    pa_radix_allocator* a = new (std::nothrow) pa_radix_allocator();
    if (!a) return nullptr;
    a->num_blocks = num_blocks;
    a->B = block_size;
    const int64_t first = reserve_block0 ? 1 : 0;
    for (int64_t b = num_blocks - 1; b >= first; --b) a->free_list.push_back((int32_t)b);
    return a;
}

void pa_radix_destroy(pa_radix_allocator* a) { delete a; }

pa_status pa_radix_allocate(pa_radix_allocator* a, const int32_t* tokens, int64_t num_tokens,
                            int64_t total_tokens, int32_t* blocks, int64_t capacity,
                            int64_t* num_allocated, int64_t* prefix_len, int64_t* allocation_id) {
    if (!a || num_tokens < 0 || (num_tokens > 0 && !tokens) || total_tokens < num_tokens ||
        !num_allocated || !prefix_len || !allocation_id)
        return PA_ERR_INVALID_ARG;
    const int64_t B = a->B;
    const int64_t n_total = (total_tokens + B - 1) / B;
    if (n_total > capacity || (n_total > 0 && !blocks)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(a->mu);
    const uint64_t t = ++a->clock;
    Allocation al;
    std::vector<Node*> path;
    a->match(tokens, num_tokens / B, path);
    // reference and touch the prefix before any eviction can see it
    for (Node* n : path) {
        n->refs += 1;
        a->touch(n, t);
        a->refresh(n);
        al.prefix_blocks += (int64_t)n->blocks.size();
    }
    al.last = path.empty() ? nullptr : path.back();
    const int64_t need = n_total - al.prefix_blocks;
    while ((int64_t)a->free_list.size() < need && !a->lru.empty()) a->evict_one();
    if ((int64_t)a->free_list.size() < need) {
        a->release(al.last);
        return PA_ERR_NO_BLOCKS;
    }
    for (Node* n : path) al.blocks.insert(al.blocks.end(), n->blocks.begin(), n->blocks.end());
    al.prefix_tokens.assign(tokens, tokens + al.prefix_blocks * B);
    for (int64_t k = 0; k < need; ++k) {
        al.blocks.push_back(a->free_list.back());
        a->free_list.pop_back();
    }
    std::copy(al.blocks.begin(), al.blocks.end(), blocks);
    *num_allocated = (int64_t)al.blocks.size();
    *prefix_len = al.prefix_blocks * B;
    const int64_t id = a->next_alloc++;
    *allocation_id = id;
    a->live.emplace(id, std::move(al));
    return PA_OK;
}

pa_status pa_radix_free(pa_radix_allocator* a, int64_t allocation_id, const int32_t* tokens,
                        int64_t num_tokens) {
    if (!a || num_tokens < 0 || (num_tokens > 0 && !tokens)) return PA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> g(a->mu);
    auto it = a->live.find(allocation_id);
    if (it == a->live.end()) return PA_ERR_INVALID_ARG;
    const int64_t B = a->B;
    Allocation& al = it->second;
    // the sequence must still start with the prefix it was given
    if (num_tokens < al.prefix_blocks * B ||
        !std::equal(al.prefix_tokens.begin(), al.prefix_tokens.end(), tokens))
        return PA_ERR_INVALID_ARG;
    const uint64_t t = ++a->clock;
    a->release(al.last);
    // insert tokens -> blocks for the whole blocks the request holds
    const int64_t n_full = std::min<int64_t>(num_tokens / B, (int64_t)al.blocks.size());
    std::vector<char> kept(al.blocks.size(), 0);
    for (int64_t k = 0; k < al.prefix_blocks; ++k) kept[(size_t)k] = 1;   // the trie's own
    Node* node = &a->root;
    int64_t i = 0;
    while (i < n_full) {
        auto c = node->children.find(a->chunk(tokens + i * B));
        if (c == node->children.end()) {
            std::vector<int32_t> key(tokens + i * B, tokens + n_full * B);
            std::vector<int32_t> blk(al.blocks.begin() + i, al.blocks.begin() + n_full);
            for (int64_t k = i; k < n_full; ++k) kept[(size_t)k] = 1;
            a->new_node(node, std::move(key), std::move(blk), t);
            break;
        }
        Node* child = c->second;
        size_t m = 1;
        const size_t nb = child->blocks.size();
        while (m < nb && i + (int64_t)m < n_full &&
               std::equal(tokens + (i + (int64_t)m) * B, tokens + (i + (int64_t)m + 1) * B,
                          child->key.begin() + (ptrdiff_t)(m * B)))
            ++m;
        // positions already cached keep the trie's blocks; ours there are spare.
        // Split where the sequences part, if there is more to insert.
        a->touch(child, t);
        if (m < nb && i + (int64_t)m < n_full) child = a->split(child, m);
        node = child;
        i += (int64_t)m;
    }
    for (size_t k = 0; k < al.blocks.size(); ++k)
        if (!kept[k]) a->free_list.push_back(al.blocks[k]);
    a->live.erase(it);
    return PA_OK;
}

int64_t pa_radix_num_free(pa_radix_allocator* a) {
    if (!a) return -1;
    std::lock_guard<std::mutex> g(a->mu);
    return (int64_t)a->free_list.size();
}

int64_t pa_radix_num_cached(pa_radix_allocator* a) {
    if (!a) return -1;
    std::lock_guard<std::mutex> g(a->mu);
    return a->cached_blocks;
}

int64_t pa_radix_num_evictable(pa_radix_allocator* a) {
    if (!a) return -1;
    std::lock_guard<std::mutex> g(a->mu);
    int64_t n = 0;
    for (const auto& e : a->lru) n += (int64_t)a->by_id.at(e.second)->blocks.size();
    return n;
}

}  // extern "C"
