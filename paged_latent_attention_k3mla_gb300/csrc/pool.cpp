// pool.cpp -- host free-list page allocator for the paged latent cache.
//
// pegainfer PR #869, "K3: paged latent MLA KV + absorbed decode", M1 commit: a
// per-slot block table with a host mirror backed by a plain free-list allocator
// that claims a page when a slot crosses a 64-token boundary and releases all
// of a slot's pages on reset; a pool size of 0 derives full coverage so every
// slot can reach max_ctx.  The review on that PR asks for the pool's total and
// allocated page counts to be exposed (k3mla_pool_stats).
//
// Page sharing (the PR's follow-up list: block-pool reuse of cached prefixes):
// pages carry a reference count.  A slot can map another slot's first pages
// (k3mla_pool_share_prefix); a write into a page mapped by more than one slot
// first takes a private copy (k3mla_pool_cow names the copy; the device moves
// the bytes with k3mla_copy_pages); a page returns to the free list when its
// last slot releases it.
#include <cstdint>
#include <cstdlib>
#include <new>
#include <vector>

#include "../../include/k3mla.h"

struct k3mla_pool {
    int n_pages;
    int n_slots;
    int max_ctx;
    int max_pages;                // table columns = ceil(max_ctx / 64)
    std::vector<int32_t> free;    // stack: back() is claimed next
    std::vector<int32_t> table;   // [n_slots][max_pages], -1 = unmapped
    std::vector<int32_t> mapped;  // pages mapped per slot
    std::vector<int32_t> refs;    // [n_pages] slots mapping the page (0 = free)
};

static uint64_t splitmix64(uint64_t* s)
{
    uint64_t z = (*s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

extern "C" int k3mla_pool_create(int n_pages, int n_slots, int max_ctx, uint64_t shuffle_seed,
                                 k3mla_pool** out)
{
    if (!out || n_slots <= 0 || max_ctx <= 0 || n_pages < 0) return K3MLA_E_INVALID;
    *out = nullptr;
    const int max_pages = (max_ctx + K3MLA_PAGE - 1) / K3MLA_PAGE;
    const long long full = (long long)n_slots * max_pages;
    if (n_pages == 0) {
        if (full > 0x7FFFFFFFll) return K3MLA_E_INVALID;
        n_pages = (int)full;
    }
    k3mla_pool* p = new (std::nothrow) k3mla_pool();
    if (!p) return K3MLA_E_INVALID;
    p->n_pages = n_pages;
    p->n_slots = n_slots;
    p->max_ctx = max_ctx;
    p->max_pages = max_pages;
    p->table.assign((size_t)n_slots * max_pages, -1);
    p->mapped.assign(n_slots, 0);
    p->refs.assign(n_pages, 0);
    // Free list as a stack whose top is page 0 (ids claimed in ascending order)
    // unless shuffled.
    p->free.resize(n_pages);
    for (int i = 0; i < n_pages; ++i) p->free[i] = n_pages - 1 - i;
    if (shuffle_seed != 0) {
        uint64_t s = shuffle_seed;
        for (int i = n_pages - 1; i > 0; --i) {
            int j = (int)(splitmix64(&s) % (uint64_t)(i + 1));
            int32_t t = p->free[i];
            p->free[i] = p->free[j];
            p->free[j] = t;
        }
    }
    *out = p;
    return K3MLA_OK;
}

extern "C" int k3mla_pool_ensure(k3mla_pool* p, int slot, int new_len)
{
    if (!p || new_len < 0) return K3MLA_E_INVALID;
    if (slot < 0 || slot >= p->n_slots) return K3MLA_E_SLOT;
    if (new_len > p->max_ctx) return K3MLA_E_CTX;
    const int need = (new_len + K3MLA_PAGE - 1) / K3MLA_PAGE;
    const int have = p->mapped[slot];
    if (need <= have) return K3MLA_OK;
    if ((size_t)(need - have) > p->free.size()) return K3MLA_E_NO_PAGES;  // all-or-nothing
    int32_t* row = p->table.data() + (size_t)slot * p->max_pages;
    for (int lp = have; lp < need; ++lp) {
        row[lp] = p->free.back();
        p->free.pop_back();
        p->refs[row[lp]] = 1;
    }
    p->mapped[slot] = need;
    return K3MLA_OK;
}

extern "C" int k3mla_pool_ensure_all(k3mla_pool* p, const int32_t* new_len, int n)
{
    if (!p || !new_len || n < 0 || n > p->n_slots) return K3MLA_E_INVALID;
    for (int b = 0; b < n; ++b) {
        const int rc = k3mla_pool_ensure(p, b, new_len[b]);
        if (rc) return rc;
    }
    return K3MLA_OK;
}

extern "C" int k3mla_pool_release_slot(k3mla_pool* p, int slot)
{
    if (!p) return K3MLA_E_INVALID;
    if (slot < 0 || slot >= p->n_slots) return K3MLA_E_SLOT;
    int32_t* row = p->table.data() + (size_t)slot * p->max_pages;
    // Push back in reverse so that a re-claim of the same count takes the same ids; a page another
    // slot still maps stays out of the free list.
    for (int lp = p->mapped[slot] - 1; lp >= 0; --lp) {
        if (--p->refs[row[lp]] == 0) p->free.push_back(row[lp]);
        row[lp] = -1;
    }
    p->mapped[slot] = 0;
    return K3MLA_OK;
}

extern "C" int k3mla_pool_share_prefix(k3mla_pool* p, int dst_slot, int src_slot, int n_tokens)
{
    if (!p || n_tokens < 0) return K3MLA_E_INVALID;
    if (dst_slot < 0 || dst_slot >= p->n_slots || src_slot < 0 || src_slot >= p->n_slots) return K3MLA_E_SLOT;
    if (n_tokens > p->max_ctx) return K3MLA_E_CTX;
    const int need = (n_tokens + K3MLA_PAGE - 1) / K3MLA_PAGE;
    if (dst_slot == src_slot || p->mapped[dst_slot] != 0 || need > p->mapped[src_slot]) return K3MLA_E_INVALID;
    const int32_t* src = p->table.data() + (size_t)src_slot * p->max_pages;
    int32_t* dst = p->table.data() + (size_t)dst_slot * p->max_pages;
    for (int lp = 0; lp < need; ++lp) {
        dst[lp] = src[lp];
        ++p->refs[src[lp]];
    }
    p->mapped[dst_slot] = need;
    return K3MLA_OK;
}

extern "C" int k3mla_pool_cow(k3mla_pool* p, int slot, int pos, int32_t* src_page, int32_t* dst_page)
{
    if (!p || pos < 0 || !src_page || !dst_page) return K3MLA_E_INVALID;
    if (slot < 0 || slot >= p->n_slots) return K3MLA_E_SLOT;
    const int lp = pos / K3MLA_PAGE;
    if (lp >= p->mapped[slot]) return K3MLA_E_CTX;  // map the position first (k3mla_pool_ensure)
    int32_t* row = p->table.data() + (size_t)slot * p->max_pages;
    const int32_t old = row[lp];
    if (p->refs[old] == 1) return 0;  // the slot owns the page alone: write in place
    if (p->free.empty()) return K3MLA_E_NO_PAGES;
    const int32_t fresh = p->free.back();
    p->free.pop_back();
    p->refs[fresh] = 1;
    --p->refs[old];
    row[lp] = fresh;
    *src_page = old;
    *dst_page = fresh;
    return 1;
}

extern "C" int k3mla_pool_page_refs(const k3mla_pool* p, int page)
{
    if (!p || page < 0 || page >= p->n_pages) return K3MLA_E_INVALID;
    return p->refs[page];
}

extern "C" const int32_t* k3mla_pool_host_table(const k3mla_pool* p) { return p ? p->table.data() : nullptr; }
extern "C" int k3mla_pool_max_pages(const k3mla_pool* p) { return p ? p->max_pages : 0; }
extern "C" int k3mla_pool_n_pages(const k3mla_pool* p) { return p ? p->n_pages : 0; }

extern "C" int k3mla_pool_stats(const k3mla_pool* p, int* total, int* used)
{
    if (!p) return K3MLA_E_INVALID;
    if (total) *total = p->n_pages;
    if (used) *used = p->n_pages - (int)p->free.size();
    return K3MLA_OK;
}

extern "C" void k3mla_pool_destroy(k3mla_pool* p) { delete p; }
