// runtime.cu -- host-side admission runtime: the shared-affix registry and the private-slot
// page allocator of one KV pool layout.
//
// Page: "Affix Cache for Diffusion Large Language Models", Sec. 4.1-4.2: the cache is split
// into a shared region that holds each common affix once and per-request private regions
// (anchors and the request's own positions); admission resolves a request's shared affix,
// gives its anchors and own positions private slots, and records the maps before the online
// loop.  This file keeps that bookkeeping: which slots hold which registered affix (reference
// counted, so later compatible requests reuse it) and which private pages belong to which
// request.  It touches no device memory; the maps themselves are built on the device by
// acache_build_slot_maps from the slot lists handed out here.
//
// Layout of a pool of num_slots slots (the same for every layer):
//   [0, private_begin)          shared region, carved into contiguous runs, one per affix
//   [private_begin, num_slots)  private region, fixed-size pages of page_slots slots
#include <stdint.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "acache.h"

struct acache_pool {
    int64_t num_slots = 0, private_begin = 0;
    int32_t page_slots = 0;
    std::mutex mu;
    // shared region: free runs keyed by start (coalesced on release), affixes by key
    std::map<int64_t, int64_t> free_runs;           // start -> length
    struct Affix {
        int64_t base;
        int32_t len;
        int64_t refs;
    };
    std::unordered_map<uint64_t, Affix> affixes;
    // private region: a stack of free page indices and the pages each request holds
    std::vector<int64_t> free_pages;
    std::unordered_map<int64_t, std::vector<int64_t>> requests;
    int64_t next_request = 1;
};

namespace {

int64_t take_run(acache_pool* p, int64_t len) {   // first fit; -1 if no run is long enough
    for (auto it = p->free_runs.begin(); it != p->free_runs.end(); ++it) {
        if (it->second < len) continue;
        const int64_t base = it->first, rest = it->second - len;
        p->free_runs.erase(it);
        if (rest > 0) p->free_runs.emplace(base + len, rest);
        return base;
    }
    return -1;
}

void give_run(acache_pool* p, int64_t base, int64_t len) {   // insert and merge with neighbours
    auto next = p->free_runs.lower_bound(base);
    if (next != p->free_runs.end() && next->first == base + len) {
        len += next->second;
        next = p->free_runs.erase(next);
    }
    if (next != p->free_runs.begin()) {
        auto prev = std::prev(next);
        if (prev->first + prev->second == base) {
            prev->second += len;
            return;
        }
    }
    p->free_runs.emplace(base, len);
}

}  // namespace

extern "C" {

int acache_pool_create(int64_t num_slots, int64_t private_begin, int32_t page_slots, acache_pool** out) {
    if (!out) return ACACHE_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_slots < 0 || private_begin < 0 || private_begin > num_slots || page_slots <= 0 ||
        num_slots > INT32_MAX)   // slot indices are int32 in every map
        return ACACHE_ERR_INVALID_ARG;
    acache_pool* p = new (std::nothrow) acache_pool();
    if (!p) return ACACHE_ERR_WORKSPACE;
    p->num_slots = num_slots;
    p->private_begin = private_begin;
    p->page_slots = page_slots;
    if (private_begin > 0) p->free_runs.emplace(0, private_begin);
    const int64_t pages = (num_slots - private_begin) / page_slots;   // a partial tail page is unused
    p->free_pages.reserve((size_t)pages);
    for (int64_t i = pages - 1; i >= 0; --i) p->free_pages.push_back(i);   // page 0 handed out first
    *out = p;
    return ACACHE_OK;
}

void acache_pool_destroy(acache_pool* p) { delete p; }

int acache_pool_register_affix(acache_pool* p, uint64_t key, int32_t affix_len, int32_t* shared_base,
                               int32_t* created) {
    if (!p || !shared_base || !created || affix_len <= 0) return ACACHE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(p->mu);
    auto it = p->affixes.find(key);
    if (it != p->affixes.end()) {
        if (it->second.len != affix_len) return ACACHE_ERR_INVALID_ARG;   // same key, other affix
        ++it->second.refs;
        *shared_base = (int32_t)it->second.base;
        *created = 0;
        return ACACHE_OK;
    }
    const int64_t base = take_run(p, affix_len);
    if (base < 0) return ACACHE_ERR_WORKSPACE;
    p->affixes.emplace(key, acache_pool::Affix{base, affix_len, 1});
    *shared_base = (int32_t)base;
    *created = 1;
    return ACACHE_OK;
}

int acache_pool_release_affix(acache_pool* p, uint64_t key) {
    if (!p) return ACACHE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(p->mu);
    auto it = p->affixes.find(key);
    if (it == p->affixes.end()) return ACACHE_ERR_INVALID_ARG;
    if (--it->second.refs == 0) {
        give_run(p, it->second.base, it->second.len);
        p->affixes.erase(it);
    }
    return ACACHE_OK;
}

int acache_pool_alloc_private(acache_pool* p, int32_t rows, int32_t* slots, int64_t* request_id) {
    if (!p || !request_id || rows < 0 || (rows > 0 && !slots)) return ACACHE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(p->mu);
    const int64_t need = ((int64_t)rows + p->page_slots - 1) / p->page_slots;
    if (need > (int64_t)p->free_pages.size()) return ACACHE_ERR_WORKSPACE;
    std::vector<int64_t> pages;
    try {
        pages.reserve((size_t)need);
        for (int64_t i = 0; i < need; ++i) {
            pages.push_back(p->free_pages.back());
            p->free_pages.pop_back();
        }
        p->requests.emplace(p->next_request, pages);
    } catch (...) {
        for (int64_t pg : pages) p->free_pages.push_back(pg);
        return ACACHE_ERR_WORKSPACE;
    }
    for (int32_t i = 0; i < rows; ++i)
        slots[i] = (int32_t)(p->private_begin + pages[i / p->page_slots] * p->page_slots + i % p->page_slots);
    *request_id = p->next_request++;
    return ACACHE_OK;
}

int acache_pool_free_private(acache_pool* p, int64_t request_id) {
    if (!p) return ACACHE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(p->mu);
    auto it = p->requests.find(request_id);
    if (it == p->requests.end()) return ACACHE_ERR_INVALID_ARG;
    for (auto pg = it->second.rbegin(); pg != it->second.rend(); ++pg) p->free_pages.push_back(*pg);
    p->requests.erase(it);
    return ACACHE_OK;
}

int acache_pool_stats(acache_pool* p, int64_t* free_shared_slots, int64_t* free_private_slots,
                      int32_t* n_affixes, int32_t* n_requests) {
    if (!p) return ACACHE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(p->mu);
    int64_t fs = 0;
    for (const auto& r : p->free_runs) fs += r.second;
    if (free_shared_slots) *free_shared_slots = fs;
    if (free_private_slots) *free_private_slots = (int64_t)p->free_pages.size() * p->page_slots;
    if (n_affixes) *n_affixes = (int32_t)p->affixes.size();
    if (n_requests) *n_requests = (int32_t)p->requests.size();
    return ACACHE_OK;
}

}  // extern "C"
