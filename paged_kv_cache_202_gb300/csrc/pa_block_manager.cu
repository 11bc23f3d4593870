// Host block manager: the free list and reference counts of a paged KV pool.
//
// "PagedAttention: The Cache Was Storing Nothing" §2.2-§2.3: the cache is cut
// into fixed-size blocks, any free block will do for any request, tables of
// several sequences may point at the same physical blocks (shared prefixes,
// beam candidates), and a shared block is copied only when a sequence diverges
// and writes into it. The "Paged Attention Meets FlexAttention" review
// describes allocation as constant time from a free list. Here the free list
// is a stack of block ids (allocate and release are O(1) per block) and every
// block carries a reference count = the number of tables naming it. One
// mutex makes every call thread-safe.
#include <mutex>
#include <unordered_map>
#include <vector>

#include "pa.h"

struct pa_block_manager {
    std::mutex mu;
    std::vector<int32_t> free_stack;  // top = back
    std::vector<int32_t> refcount;
};

namespace {

bool valid_id(const pa_block_manager* bm, int32_t id) {
    return id >= 0 && id < static_cast<int32_t>(bm->refcount.size());
}

}  // namespace

extern "C" {

pa_status pa_bm_create(int num_blocks, pa_block_manager** out) {
    if (!out) return PA_ERR_NULL;
    if (num_blocks < 1) return PA_ERR_SHAPE;
    pa_block_manager* bm = new pa_block_manager();
    bm->refcount.assign(static_cast<size_t>(num_blocks), 0);
    bm->free_stack.reserve(static_cast<size_t>(num_blocks));
    for (int32_t id = num_blocks - 1; id >= 0; --id) bm->free_stack.push_back(id);  // 0 on top
    *out = bm;
    return PA_OK;
}

pa_status pa_bm_destroy(pa_block_manager* bm) {
    delete bm;
    return PA_OK;
}

pa_status pa_bm_alloc(pa_block_manager* bm, int n, int32_t* ids) {
    if (!bm || (n > 0 && !ids)) return PA_ERR_NULL;
    if (n < 0) return PA_ERR_SHAPE;
    std::lock_guard<std::mutex> lk(bm->mu);
    if (static_cast<size_t>(n) > bm->free_stack.size()) return PA_ERR_NO_BLOCKS;
    for (int i = 0; i < n; ++i) {
        const int32_t id = bm->free_stack.back();
        bm->free_stack.pop_back();
        bm->refcount[static_cast<size_t>(id)] = 1;
        ids[i] = id;
    }
    return PA_OK;
}

pa_status pa_bm_fork(pa_block_manager* bm, const int32_t* ids, int n) {
    if (!bm || (n > 0 && !ids)) return PA_ERR_NULL;
    if (n < 0) return PA_ERR_SHAPE;
    std::lock_guard<std::mutex> lk(bm->mu);
    for (int i = 0; i < n; ++i)
        if (!valid_id(bm, ids[i]) || bm->refcount[static_cast<size_t>(ids[i])] < 1)
            return PA_ERR_BOUNDS;
    for (int i = 0; i < n; ++i) ++bm->refcount[static_cast<size_t>(ids[i])];
    return PA_OK;
}

pa_status pa_bm_release(pa_block_manager* bm, const int32_t* ids, int n) {
    if (!bm || (n > 0 && !ids)) return PA_ERR_NULL;
    if (n < 0) return PA_ERR_SHAPE;
    std::lock_guard<std::mutex> lk(bm->mu);
    // Validate against the counts this call would leave (an id may repeat).
    std::unordered_map<int32_t, int32_t> drops;
    for (int i = 0; i < n; ++i) {
        if (!valid_id(bm, ids[i])) return PA_ERR_BOUNDS;
        if (++drops[ids[i]] > bm->refcount[static_cast<size_t>(ids[i])]) return PA_ERR_BOUNDS;
    }
    for (int i = 0; i < n; ++i) {
        int32_t& c = bm->refcount[static_cast<size_t>(ids[i])];
        if (--c == 0) bm->free_stack.push_back(ids[i]);
    }
    return PA_OK;
}

pa_status pa_bm_refcount(const pa_block_manager* bm, int32_t id, int* count) {
    if (!bm || !count) return PA_ERR_NULL;
    pa_block_manager* m = const_cast<pa_block_manager*>(bm);
    std::lock_guard<std::mutex> lk(m->mu);
    if (!valid_id(bm, id)) return PA_ERR_BOUNDS;
    *count = bm->refcount[static_cast<size_t>(id)];
    return PA_OK;
}

pa_status pa_bm_num_free(const pa_block_manager* bm, int* n) {
    if (!bm || !n) return PA_ERR_NULL;
    pa_block_manager* m = const_cast<pa_block_manager*>(bm);
    std::lock_guard<std::mutex> lk(m->mu);
    *n = static_cast<int>(bm->free_stack.size());
    return PA_OK;
}

pa_status pa_bm_prepare_append(pa_block_manager* bm, int32_t* tables, int B, int max_blocks,
                               const int32_t* cache_lens, int block_size, int32_t* copy_src,
                               int32_t* copy_dst, int* n_copies) {
    if (!bm || !n_copies || (B > 0 && (!tables || !cache_lens || !copy_src || !copy_dst)))
        return PA_ERR_NULL;
    if (B < 0 || max_blocks < 1) return PA_ERR_SHAPE;
    if (block_size != 16 && block_size != 32) return PA_ERR_BLOCK_SIZE;
    std::lock_guard<std::mutex> lk(bm->mu);
    // Check everything first so that a failing call changes nothing: count the
    // fresh blocks the batch needs, replaying the count changes it would make
    // (two sequences writing one shared block: the first copies, the last keeps it).
    size_t need = 0;
    std::unordered_map<int32_t, int32_t> counts;
    for (int b = 0; b < B; ++b) {
        const int64_t pos = cache_lens[b];
        if (pos < 0 || pos >= static_cast<int64_t>(max_blocks) * block_size) return PA_ERR_BOUNDS;
        const int32_t id = tables[static_cast<int64_t>(b) * max_blocks + pos / block_size];
        if (id >= 0 && (!valid_id(bm, id) || bm->refcount[static_cast<size_t>(id)] < 1))
            return PA_ERR_BOUNDS;
        if (id < 0) {
            ++need;
            continue;
        }
        auto it = counts.emplace(id, bm->refcount[static_cast<size_t>(id)]).first;
        if (it->second > 1) {
            ++need;
            --it->second;
        }
    }
    if (need > bm->free_stack.size()) return PA_ERR_NO_BLOCKS;
    int nc = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t pos = cache_lens[b];
        int32_t& slot = tables[static_cast<int64_t>(b) * max_blocks + pos / block_size];
        if (slot >= 0 && bm->refcount[static_cast<size_t>(slot)] == 1) continue;  // private block
        const int32_t fresh = bm->free_stack.back();
        bm->free_stack.pop_back();
        bm->refcount[static_cast<size_t>(fresh)] = 1;
        if (slot >= 0) {  // shared: copy on write
            copy_src[nc] = slot;
            copy_dst[nc] = fresh;
            ++nc;
            --bm->refcount[static_cast<size_t>(slot)];  // stays >= 1: others still share it
        }
        slot = fresh;
    }
    *n_copies = nc;
    return PA_OK;
}

}  // extern "C"
