// Host-side free-block pool and block-table builder.
//
// The pool is the free-block queue of "连续批处理与KV缓存" §4.2 (all free
// blocks in one queue, taken from the front, returned at the back, O(1)
// per block), stored as a fixed ring of num_blocks int32 so that no
// operation moves the whole list. Requests hold ordered lists of blocks and
// may reference pinned shared blocks in front of them (a shared prompt
// prefix: "vLLM核心概念" §3.2; "轻量级推理引擎实战" §2.1). A held block carries
// a reference count -- the live requests holding it -- so that a request can
// be forked (the child holds every block of the parent) and a block is
// replaced by a private copy only when one holder writes into it
// (copy-on-write, "vLLM核心概念" §3.2); free returns a block to the pool when
// its last holder lets go.
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/pkv.h"

struct pkv_allocator {
    int32_t num_blocks = 0;
    int32_t block_size = 0;
    std::vector<int32_t> ring;  // capacity num_blocks; free ids live in [head, head + count)
    int64_t head = 0;
    int64_t count = 0;
    std::vector<int32_t> refs;  // per block: live requests holding it (0 = free or pinned-only)
    struct Request {
        std::vector<int32_t> shared;  // pinned blocks, read-only, not counted
        std::vector<int32_t> owned;   // held blocks, counted in refs
    };
    std::unordered_map<int64_t, Request> live;

    int32_t pop_front() {
        int32_t id = ring[static_cast<size_t>(head)];
        head = (head + 1 == num_blocks) ? 0 : head + 1;
        --count;
        refs[static_cast<size_t>(id)] = 1;
        return id;
    }
    void push_back(int32_t id) {
        int64_t tail = head + count;
        if (tail >= num_blocks) tail -= num_blocks;
        ring[static_cast<size_t>(tail)] = id;
        ++count;
    }
};

extern "C" {

pkv_allocator* pkv_allocator_create(int32_t num_blocks, int32_t block_size,
                                    const int32_t* initial_order) {
    if (num_blocks <= 0 || block_size <= 0) return nullptr;
    pkv_allocator* a = new (std::nothrow) pkv_allocator();
    if (!a) return nullptr;
    try {
        a->ring.resize(static_cast<size_t>(num_blocks));
        a->refs.assign(static_cast<size_t>(num_blocks), 0);
        if (initial_order) {
            std::vector<uint8_t> seen(static_cast<size_t>(num_blocks), 0);
            for (int32_t i = 0; i < num_blocks; ++i) {
                int32_t id = initial_order[i];
                if (id < 0 || id >= num_blocks || seen[static_cast<size_t>(id)]) {
                    delete a;
                    return nullptr;
                }
                seen[static_cast<size_t>(id)] = 1;
                a->ring[static_cast<size_t>(i)] = id;
            }
        } else {
            for (int32_t i = 0; i < num_blocks; ++i) a->ring[static_cast<size_t>(i)] = i;
        }
    } catch (...) {
        delete a;
        return nullptr;
    }
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    a->head = 0;
    a->count = num_blocks;
    return a;
}

void pkv_allocator_destroy(pkv_allocator* a) { delete a; }

int pkv_alloc(pkv_allocator* a, int64_t req_id, int32_t n_blocks, int32_t* out_ids) {
    if (!a || n_blocks < 0 || (n_blocks > 0 && !out_ids)) return PKV_ERR_INVALID;
    if (a->live.count(req_id)) return PKV_ERR_EXISTS;
    if (a->count < n_blocks) return PKV_ERR_OOM;
    try {
        pkv_allocator::Request r;
        r.owned.reserve(static_cast<size_t>(n_blocks) + 8);
        auto it = a->live.emplace(req_id, std::move(r)).first;
        for (int32_t i = 0; i < n_blocks; ++i) {
            int32_t id = a->pop_front();
            it->second.owned.push_back(id);
            out_ids[i] = id;
        }
    } catch (...) {
        return PKV_ERR_OOM;
    }
    return PKV_OK;
}

int pkv_append_block(pkv_allocator* a, int64_t req_id, int32_t* out_id) {
    if (!a || !out_id) return PKV_ERR_INVALID;
    auto it = a->live.find(req_id);
    if (it == a->live.end()) return PKV_ERR_NOT_FOUND;
    if (a->count == 0) return PKV_ERR_OOM;
    try {
        it->second.owned.reserve(it->second.owned.size() + 1);
    } catch (...) {
        return PKV_ERR_OOM;
    }
    int32_t id = a->pop_front();
    it->second.owned.push_back(id);
    *out_id = id;
    return PKV_OK;
}

int pkv_free(pkv_allocator* a, int64_t req_id) {
    if (!a) return PKV_ERR_INVALID;
    auto it = a->live.find(req_id);
    if (it == a->live.end()) return PKV_ERR_NOT_FOUND;
    for (int32_t id : it->second.owned)
        if (--a->refs[static_cast<size_t>(id)] == 0) a->push_back(id);
    a->live.erase(it);
    return PKV_OK;
}

int pkv_attach_shared(pkv_allocator* a, int64_t req_id, const int32_t* ids, int32_t n) {
    if (!a || n < 0 || (n > 0 && !ids)) return PKV_ERR_INVALID;
    auto it = a->live.find(req_id);
    if (it == a->live.end()) return PKV_ERR_NOT_FOUND;
    for (int32_t i = 0; i < n; ++i)
        if (ids[i] < 0 || ids[i] >= a->num_blocks) return PKV_ERR_INVALID;
    try {
        auto& sh = it->second.shared;
        sh.insert(sh.begin(), ids, ids + n);
    } catch (...) {
        return PKV_ERR_OOM;
    }
    return PKV_OK;
}

int pkv_fork(pkv_allocator* a, int64_t parent, int64_t child) {
    if (!a) return PKV_ERR_INVALID;
    auto it = a->live.find(parent);
    if (it == a->live.end()) return PKV_ERR_NOT_FOUND;
    if (a->live.count(child)) return PKV_ERR_EXISTS;
    try {
        pkv_allocator::Request r = it->second;  // copies both lists
        a->live.emplace(child, std::move(r));
    } catch (...) {
        return PKV_ERR_OOM;
    }
    for (int32_t id : a->live.find(child)->second.owned) ++a->refs[static_cast<size_t>(id)];
    return PKV_OK;
}

int pkv_cow_block(pkv_allocator* a, int64_t req_id, int32_t index, int32_t* out_src, int32_t* out_dst) {
    if (!a || !out_src || !out_dst || index < 0) return PKV_ERR_INVALID;
    auto it = a->live.find(req_id);
    if (it == a->live.end()) return PKV_ERR_NOT_FOUND;
    auto& r = it->second;
    const size_t ns = r.shared.size();
    if (static_cast<size_t>(index) < ns) return PKV_ERR_INVALID;  // pinned blocks are read-only
    const size_t k = static_cast<size_t>(index) - ns;
    if (k >= r.owned.size()) return PKV_ERR_INVALID;
    const int32_t old = r.owned[k];
    *out_src = *out_dst = -1;
    if (a->refs[static_cast<size_t>(old)] <= 1) return PKV_OK;  // held by this request alone
    if (a->count == 0) return PKV_ERR_OOM;
    const int32_t fresh = a->pop_front();
    --a->refs[static_cast<size_t>(old)];
    r.owned[k] = fresh;
    *out_src = old;
    *out_dst = fresh;
    return PKV_OK;
}

int pkv_block_refs(const pkv_allocator* a, int32_t block) {
    if (!a || block < 0 || block >= a->num_blocks) return PKV_ERR_INVALID;
    return a->refs[static_cast<size_t>(block)];
}

int pkv_num_free(const pkv_allocator* a) { return a ? static_cast<int>(a->count) : -1; }

int pkv_request_table(const pkv_allocator* a, int64_t req_id, int32_t* out, int32_t cap) {
    if (!a || cap < 0 || (cap > 0 && !out)) return PKV_ERR_INVALID;
    auto it = a->live.find(req_id);
    if (it == a->live.end()) return PKV_ERR_NOT_FOUND;
    const auto& r = it->second;
    int32_t n = 0;
    for (int32_t id : r.shared) { if (n < cap) out[n] = id; ++n; }
    for (int32_t id : r.owned)  { if (n < cap) out[n] = id; ++n; }
    return n;
}

int pkv_free_list(const pkv_allocator* a, int32_t* out, int32_t cap) {
    if (!a || cap < 0 || (cap > 0 && !out)) return PKV_ERR_INVALID;
    int64_t pos = a->head;
    for (int64_t i = 0; i < a->count && i < cap; ++i) {
        out[i] = a->ring[static_cast<size_t>(pos)];
        pos = (pos + 1 == a->num_blocks) ? 0 : pos + 1;
    }
    return static_cast<int>(a->count);
}

int pkv_build_block_tables(const pkv_allocator* a, const int64_t* req_ids, int32_t B,
                           int32_t max_blocks, int32_t* out_table) {
    if (!a || B < 0 || max_blocks < 0 || (B > 0 && (!req_ids || (max_blocks > 0 && !out_table))))
        return PKV_ERR_INVALID;
    for (int32_t b = 0; b < B; ++b) {
        int32_t* row = out_table + static_cast<size_t>(b) * static_cast<size_t>(max_blocks);
        auto it = a->live.find(req_ids[b]);
        if (it == a->live.end()) return PKV_ERR_NOT_FOUND;
        const auto& r = it->second;
        size_t n = r.shared.size() + r.owned.size();
        if (n > static_cast<size_t>(max_blocks)) return PKV_ERR_INVALID;
        if (!r.shared.empty()) std::memcpy(row, r.shared.data(), r.shared.size() * sizeof(int32_t));
        if (!r.owned.empty())
            std::memcpy(row + r.shared.size(), r.owned.data(), r.owned.size() * sizeof(int32_t));
        for (size_t i = n; i < static_cast<size_t>(max_blocks); ++i) row[i] = -1;
    }
    return PKV_OK;
}

}  // extern "C"
