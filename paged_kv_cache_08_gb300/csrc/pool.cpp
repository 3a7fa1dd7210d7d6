// Host block pool: the untimed bookkeeping that produces block tables and slot mappings.
//
// Free set: a binary min-heap of the free block ids, so that an allocation takes the lowest
// free id (the order the free-bitmap allocator of "端侧 SLM 显存保活术：在 4GB 内存板卡上实现
// 轻量 PagedAttention 与 KV 缓存分块", section "嵌入式轻量 Block 分配器设计", hands blocks out in,
// kept here as a requirement: the worked examples number their blocks that way) in O(log n),
// and a release pushes the id back.  A block is free exactly when its reference count is 0.
// Reference counts: shared prefix blocks ("共享前缀块（Prefix Caching）" on the same page)
// and copy-on-write on append ("显存虚拟化革命：PagedAttention 内存池管理与显存碎片终结", §四).
// Token append and release follow the lifecycle diagram of that page's §三.
// Slotted blocks (pa_slots_*): short nodes packed into shared blocks and addressed by
// (block_id, slot_offset, length), the radix-tree fragmentation page's "Slotted Block 分槽与
// 微块共享架构".
#include <cstdint>
#include <cstdlib>
#include <new>
#include <algorithm>
#include <functional>
#include <vector>

#include "../../include/pa.h"

struct pa_pool {
    int num_blocks;
    std::vector<int32_t> free_heap;   // free ids, a min-heap under std::greater (front = lowest)
    std::vector<int32_t> refs;        // 0 = free
};

namespace {

inline bool valid_id(const pa_pool* p, int id) { return p && id >= 0 && id < p->num_blocks; }

// The lowest free id, taken out of the free set; -1 when the set is empty.
inline int take_lowest_free(pa_pool* p) {
    if (p->free_heap.empty()) return -1;
    std::pop_heap(p->free_heap.begin(), p->free_heap.end(), std::greater<int32_t>());
    const int id = p->free_heap.back();
    p->free_heap.pop_back();
    return id;
}

inline void give_back(pa_pool* p, int id) {
    p->free_heap.push_back(id);
    std::push_heap(p->free_heap.begin(), p->free_heap.end(), std::greater<int32_t>());
}

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

pa_pool* pa_pool_create(int num_blocks) {
    if (num_blocks <= 0) return nullptr;
    pa_pool* p = new (std::nothrow) pa_pool;
    if (!p) return nullptr;
    try {
        p->num_blocks = num_blocks;
        // 0, 1, ..., n-1 in increasing order is already a min-heap
        p->free_heap.resize((size_t)num_blocks);
        for (int i = 0; i < num_blocks; ++i) p->free_heap[(size_t)i] = i;
        p->refs.assign((size_t)num_blocks, 0);
    } catch (...) {
        delete p;
        return nullptr;
    }
    return p;
}

void pa_pool_destroy(pa_pool* pool) { delete pool; }

int pa_pool_alloc(pa_pool* pool) {
    if (!pool) return PA_ERR_INVALID_ARG;
    const int id = take_lowest_free(pool);
    if (id < 0) return PA_ERR_POOL_EXHAUSTED;
    pool->refs[id] = 1;
    return id;
}

int pa_pool_incref(pa_pool* pool, int block_id) {
    if (!valid_id(pool, block_id) || pool->refs[block_id] <= 0) return PA_ERR_BOUNDS;
    return ++pool->refs[block_id];
}

int pa_pool_decref(pa_pool* pool, int block_id) {
    if (!valid_id(pool, block_id) || pool->refs[block_id] <= 0) return PA_ERR_BOUNDS;
    int r = --pool->refs[block_id];
    if (r == 0) give_back(pool, block_id);
    return r;
}

int pa_pool_refcount(const pa_pool* pool, int block_id) {
    if (!valid_id(pool, block_id)) return PA_ERR_BOUNDS;
    return pool->refs[block_id];
}

int pa_pool_num_free(const pa_pool* pool) { return pool ? (int)pool->free_heap.size() : PA_ERR_INVALID_ARG; }

int pa_pool_num_blocks(const pa_pool* pool) { return pool ? pool->num_blocks : PA_ERR_INVALID_ARG; }

int pa_pool_assign(pa_pool* pool, int32_t* table_row, int max_blocks, int context_len,
                   int block_size, const int32_t* shared_row, int shared_blocks) {
    if (!pool || !table_row || max_blocks < 0 || context_len < 0 || block_size <= 0 ||
        shared_blocks < 0 || (shared_blocks > 0 && !shared_row))
        return PA_ERR_INVALID_ARG;
    const int need = ceil_div(context_len, block_size);
    if (need > max_blocks || shared_blocks > need) return PA_ERR_BOUNDS;
    for (int i = 0; i < shared_blocks; ++i)
        if (!valid_id(pool, shared_row[i]) || pool->refs[shared_row[i]] <= 0) return PA_ERR_BOUNDS;
    if (need - shared_blocks > (int)pool->free_heap.size()) return PA_ERR_POOL_EXHAUSTED;
    for (int i = 0; i < shared_blocks; ++i) {
        table_row[i] = shared_row[i];
        ++pool->refs[shared_row[i]];
    }
    for (int i = shared_blocks; i < need; ++i) table_row[i] = pa_pool_alloc(pool);
    for (int i = need; i < max_blocks; ++i) table_row[i] = -1;
    return PA_OK;
}

int pa_pool_append_token(pa_pool* pool, int32_t* table_row, int max_blocks, int context_len,
                         int block_size, int64_t* slot, int32_t* cow_src, int32_t* cow_dst) {
    if (!pool || !table_row || !slot || max_blocks < 0 || context_len < 0 || block_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (cow_src) *cow_src = -1;
    if (cow_dst) *cow_dst = -1;
    const int logical = context_len / block_size;  // block of the new token
    const int offset = context_len % block_size;
    if (logical >= max_blocks) return PA_ERR_BOUNDS;
    if (offset == 0) {
        // the last block is full (or the sequence is empty): take a fresh block
        int id = pa_pool_alloc(pool);
        if (id < 0) return id;
        table_row[logical] = id;
    } else {
        int cur = table_row[logical];
        if (!valid_id(pool, cur) || pool->refs[cur] <= 0) return PA_ERR_BOUNDS;
        if (pool->refs[cur] > 1) {
            // shared and not full: copy-on-write before the write lands in it
            int id = pa_pool_alloc(pool);
            if (id < 0) return id;
            --pool->refs[cur];
            table_row[logical] = id;
            if (cow_src) *cow_src = cur;
            if (cow_dst) *cow_dst = id;
        }
    }
    *slot = (int64_t)table_row[logical] * block_size + offset;
    return PA_OK;
}

int pa_pool_release(pa_pool* pool, int32_t* table_row, int max_blocks, int context_len,
                    int block_size) {
    if (!pool || !table_row || context_len < 0 || block_size <= 0) return PA_ERR_INVALID_ARG;
    const int n = ceil_div(context_len, block_size);
    if (n > max_blocks) return PA_ERR_BOUNDS;
    for (int i = 0; i < n; ++i) {
        if (pa_pool_decref(pool, table_row[i]) < 0) return PA_ERR_BOUNDS;
        table_row[i] = -1;
    }
    return PA_OK;
}

int pa_pool_move_blocks(pa_pool* from, pa_pool* to, int32_t* table_row, int n, int32_t* src_ids,
                        int32_t* dst_ids) {
    if (!from || !to || n < 0 || (n > 0 && (!table_row || !src_ids || !dst_ids))) return PA_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (!valid_id(from, table_row[i]) || from->refs[table_row[i]] <= 0) return PA_ERR_BOUNDS;
    if (n > (int)to->free_heap.size()) return PA_ERR_POOL_EXHAUSTED;
    for (int i = 0; i < n; ++i) {
        const int id = pa_pool_alloc(to);   // cannot fail: n blocks are free
        src_ids[i] = table_row[i];
        dst_ids[i] = id;
        pa_pool_decref(from, table_row[i]);
        table_row[i] = id;
    }
    return n;
}

// ---- slotted blocks ----
// A node of n <= B tokens goes to the earliest-opened block whose free tail still holds n
// (slots are appended at the tail: offset = tokens already placed), else to a fresh block, the
// lowest free id.  A block counts its live slots; a released slot's space is reused only once
// the block has emptied and gone back to the free set, so live slots never overlap.
struct pa_slots {
    int num_blocks, block_size;
    std::vector<int> tail;     // tokens placed in the block (next slot offset)
    std::vector<int> live;     // live slots in the block
    std::vector<int> open;     // blocks with room left, in the order they were opened
    int num_free;
};

pa_slots* pa_slots_create(int num_blocks, int block_size) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pa_slots* p = new (std::nothrow) pa_slots;
    if (!p) return nullptr;
    try {
        p->num_blocks = num_blocks;
        p->block_size = block_size;
        p->tail.assign((size_t)num_blocks, 0);
        p->live.assign((size_t)num_blocks, 0);
        p->num_free = num_blocks;
    } catch (...) {
        delete p;
        return nullptr;
    }
    return p;
}

void pa_slots_destroy(pa_slots* p) { delete p; }

int pa_slots_alloc(pa_slots* p, int n, int32_t* block, int32_t* offset) {
    if (!p || !block || !offset || n <= 0 || n > p->block_size) return PA_ERR_INVALID_ARG;
    for (size_t i = 0; i < p->open.size(); ++i) {
        const int b = p->open[i];
        if (p->block_size - p->tail[b] >= n) {
            *block = b;
            *offset = p->tail[b];
            p->tail[b] += n;
            ++p->live[b];
            if (p->tail[b] == p->block_size) p->open.erase(p->open.begin() + (long)i);
            return PA_OK;
        }
    }
    for (int b = 0; b < p->num_blocks; ++b) {
        if (p->live[b] == 0 && p->tail[b] == 0) {   // free
            *block = b;
            *offset = 0;
            p->tail[b] = n;
            p->live[b] = 1;
            --p->num_free;
            if (n < p->block_size) p->open.push_back(b);
            return PA_OK;
        }
    }
    return PA_ERR_POOL_EXHAUSTED;
}

int pa_slots_release(pa_slots* p, int32_t block, int32_t offset, int n) {
    if (!p || block < 0 || block >= p->num_blocks || p->live[block] <= 0 || offset < 0 || n <= 0 ||
        offset + n > p->tail[block])
        return PA_ERR_BOUNDS;
    if (--p->live[block] == 0) {
        p->tail[block] = 0;
        ++p->num_free;
        p->open.erase(std::remove(p->open.begin(), p->open.end(), (int)block), p->open.end());
    }
    return p->live[block];
}

int pa_slots_tail(const pa_slots* p, int32_t block) {
    if (!p || block < 0 || block >= p->num_blocks) return PA_ERR_BOUNDS;
    return p->tail[block];
}

int pa_slots_live(const pa_slots* p, int32_t block) {
    if (!p || block < 0 || block >= p->num_blocks) return PA_ERR_BOUNDS;
    return p->live[block];
}

int pa_slots_num_free(const pa_slots* p) { return p ? p->num_free : PA_ERR_INVALID_ARG; }

int pa_build_slot_mapping(const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                          int num_seqs, int block_size, int64_t* slots) {
    if (num_seqs < 0 || block_size <= 0 || max_blocks < 0) return PA_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!block_tables || !context_lens || !slots)) return PA_ERR_INVALID_ARG;
    for (int s = 0; s < num_seqs; ++s) {
        const int L = context_lens[s];
        if (L < 0 || (int64_t)L > (int64_t)max_blocks * block_size) return PA_ERR_BOUNDS;
        if (L == 0) {
            slots[s] = -1;
            continue;
        }
        const int t = L - 1;
        const int32_t phys = block_tables[(int64_t)s * max_blocks + t / block_size];
        if (phys < 0) return PA_ERR_BOUNDS;
        slots[s] = (int64_t)phys * block_size + t % block_size;
    }
    return PA_OK;
}

}  // extern "C"
