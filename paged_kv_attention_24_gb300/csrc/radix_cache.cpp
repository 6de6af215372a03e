// Radix prefix cache and page allocator for the unified KV pool (host side).
//
// "Mini-SGLang 实战指南", §6.5 "Radix Cache": requests reuse the KV of shared
// prefixes through a radix tree; §6.2: the page is the pool's allocation
// unit.  The public contract is in include/msgl_radix.h.
//
// Every page of the pool is in exactly one state: free, held by a running
// request, or cached as one node of the tree.  A node is one full page.  Its
// key is the page's token ids, and its children are the pages that can follow
// it.  Pins (reference counts) keep the matched path of a running request
// out of eviction; leaves with no pins are evicted least recently used first.
// The evictable leaves are kept in an ordered set keyed by (stamp, page id),
// updated on every pin, unpin, stamp change, insert and eviction, so an
// eviction costs O(log n) per page freed instead of a walk of the whole tree.
#include <stdint.h>
#include <string.h>

#include <map>
#include <memory>
#include <set>
#include <unordered_map>
#include <utility>
#include <vector>

#include "../../include/msgl_radix.h"

namespace {

enum PageState : uint8_t { kFree = 0, kHeld = 1, kCached = 2 };

struct Node {
    std::vector<int32_t> key;                       // the page's token ids (empty for the root)
    int32_t page = -1;                              // pool page id (-1 for the root)
    int32_t pins = 0;
    uint64_t stamp = 0;                             // last match / insert
    Node *parent = nullptr;
    std::map<std::vector<int32_t>, std::unique_ptr<Node>> children;
};

}  // namespace

struct msgl_radix_cache {
    int32_t page_size = 0;
    int32_t num_pages = 0;
    std::vector<uint8_t> state;                     // PageState per page
    std::vector<int32_t> free_list;                 // stack of free page ids
    std::unordered_map<int32_t, Node *> node_of;    // cached page -> its node
    Node root;
    uint64_t clock = 0;
    int64_t next_lease = 1;
    std::unordered_map<int64_t, std::vector<Node *>> leases;
    int32_t pinned_pages = 0;
    std::set<std::pair<uint64_t, int32_t>> evictable;   // (stamp, page) of every unpinned leaf

    bool is_evictable(const Node *n) const { return n != &root && n->children.empty() && n->pins == 0; }
    // Call untrack before changing a node's stamp, pins or children, track after.
    void untrack(const Node *n) {
        if (is_evictable(n)) evictable.erase({n->stamp, n->page});
    }
    void track(const Node *n) {
        if (is_evictable(n)) evictable.insert({n->stamp, n->page});
    }
    void touch(Node *n, uint64_t now) {
        untrack(n);
        n->stamp = now;
        track(n);
    }
    void pin(Node *n) {
        untrack(n);
        if (n->pins++ == 0) ++pinned_pages;
    }
    void unpin(Node *n) {
        if (--n->pins == 0) --pinned_pages;
        track(n);
    }
    void free_page(int32_t p) {
        state[p] = kFree;
        free_list.push_back(p);
    }

    // Evict unpinned leaves, oldest first (ties: lower page id first), until `need`
    // pages are free or none is left.  A parent whose last child goes becomes a leaf
    // and joins the candidates.
    void evict(int32_t need) {
        while ((int32_t)free_list.size() < need && !evictable.empty()) {
            const int32_t page = evictable.begin()->second;
            evictable.erase(evictable.begin());
            Node *n = node_of[page];
            Node *parent = n->parent;
            node_of.erase(page);
            free_page(page);
            parent->children.erase(n->key);   // destroys n
            track(parent);
        }
    }
};

extern "C" {

msgl_radix_cache *msgl_radix_create(int32_t page_size, int32_t num_pages) {
    if (page_size <= 0 || num_pages < 0) return nullptr;
    msgl_radix_cache *c = new msgl_radix_cache();
    c->page_size = page_size;
    c->num_pages = num_pages;
    c->state.assign((size_t)num_pages, kFree);
    c->free_list.reserve((size_t)num_pages);
    for (int32_t p = num_pages - 1; p >= 0; --p) c->free_list.push_back(p);   // page 0 handed out first
    return c;
}

void msgl_radix_destroy(msgl_radix_cache *c) { delete c; }

int32_t msgl_radix_match(msgl_radix_cache *c, const int32_t *tokens, int32_t n, int32_t *out_pages,
                         int32_t cap, int64_t *lease) {
    if (!c || n < 0 || (n > 0 && !tokens) || cap < 0 || (cap > 0 && !out_pages) || !lease)
        return MSGL_RADIX_ERR_ARG;
    const int32_t ps = c->page_size;
    std::vector<Node *> path;
    Node *cur = &c->root;
    const uint64_t now = ++c->clock;
    std::vector<int32_t> key((size_t)ps);
    for (int32_t i = 0; (i + 1) * ps <= n && i < cap; ++i) {
        memcpy(key.data(), tokens + (size_t)i * ps, sizeof(int32_t) * (size_t)ps);
        auto it = cur->children.find(key);
        if (it == cur->children.end()) break;
        cur = it->second.get();
        c->touch(cur, now);
        c->pin(cur);
        out_pages[i] = cur->page;
        path.push_back(cur);
    }
    const int64_t id = c->next_lease++;
    c->leases.emplace(id, std::move(path));
    *lease = id;
    return (int32_t)(c->leases[id].size()) * ps;
}

int32_t msgl_radix_alloc(msgl_radix_cache *c, int32_t n, int32_t *out_pages) {
    if (!c || n < 0 || (n > 0 && !out_pages)) return MSGL_RADIX_ERR_ARG;
    if ((int32_t)c->free_list.size() < n) c->evict(n);
    if ((int32_t)c->free_list.size() < n) return MSGL_RADIX_ERR_NO_PAGES;
    for (int32_t i = 0; i < n; ++i) {
        const int32_t p = c->free_list.back();
        c->free_list.pop_back();
        c->state[p] = kHeld;
        out_pages[i] = p;
    }
    return n;
}

static int32_t end_lease(msgl_radix_cache *c, int64_t lease) {
    auto it = c->leases.find(lease);
    if (it == c->leases.end()) return MSGL_RADIX_ERR_LEASE;
    for (Node *p : it->second) c->unpin(p);
    c->leases.erase(it);
    return 0;
}

int32_t msgl_radix_insert(msgl_radix_cache *c, const int32_t *tokens, int32_t n, const int32_t *pages,
                          int64_t lease) {
    if (!c || n < 0 || (n > 0 && (!tokens || !pages))) return MSGL_RADIX_ERR_ARG;
    const int32_t ps = c->page_size;
    const int32_t n_pages = (n + ps - 1) / ps;
    for (int32_t i = 0; i < n_pages; ++i)
        if (pages[i] < 0 || pages[i] >= c->num_pages) return MSGL_RADIX_ERR_PAGE;
    if (c->leases.find(lease) == c->leases.end()) return MSGL_RADIX_ERR_LEASE;
    const uint64_t now = ++c->clock;
    int32_t added = 0;
    Node *cur = &c->root;
    std::vector<int32_t> key((size_t)ps);
    for (int32_t i = 0; i < n_pages; ++i) {
        const int32_t p = pages[i];
        if ((i + 1) * ps > n) {                       // trailing partial page: not cacheable
            if (c->state[p] == kHeld) c->free_page(p);
            continue;
        }
        memcpy(key.data(), tokens + (size_t)i * ps, sizeof(int32_t) * (size_t)ps);
        auto it = cur->children.find(key);
        if (it != cur->children.end()) {
            Node *nd = it->second.get();
            if (nd->page != p && c->state[p] == kHeld) c->free_page(p);   // duplicate of a cached page
            c->touch(nd, now);
            cur = nd;
            continue;
        }
        if (c->state[p] != kHeld) {
            // a page that is free or cached elsewhere cannot back this chunk: stop caching here,
            // but still return the request's remaining held pages
            for (int32_t k = i; k < n_pages; ++k)
                if (c->state[pages[k]] == kHeld) c->free_page(pages[k]);
            break;
        }
        std::unique_ptr<Node> nd(new Node());
        nd->key = key;
        nd->page = p;
        nd->stamp = now;
        nd->parent = cur;
        Node *raw = nd.get();
        c->untrack(cur);                              // cur gains a child: no longer a leaf
        cur->children.emplace(key, std::move(nd));
        c->track(raw);
        c->state[p] = kCached;
        c->node_of[p] = raw;
        cur = raw;
        ++added;
    }
    end_lease(c, lease);
    return added;
}

int32_t msgl_radix_release(msgl_radix_cache *c, int64_t lease, const int32_t *pages, int32_t n_pages) {
    if (!c || n_pages < 0 || (n_pages > 0 && !pages)) return MSGL_RADIX_ERR_ARG;
    for (int32_t i = 0; i < n_pages; ++i)
        if (pages[i] < 0 || pages[i] >= c->num_pages) return MSGL_RADIX_ERR_PAGE;
    const int32_t rc = end_lease(c, lease);
    if (rc) return rc;
    for (int32_t i = 0; i < n_pages; ++i)
        if (c->state[pages[i]] == kHeld) c->free_page(pages[i]);
    return 0;
}

int32_t msgl_radix_stats(const msgl_radix_cache *c, int32_t *free_pages, int32_t *cached_pages,
                         int32_t *pinned_pages) {
    if (!c) return MSGL_RADIX_ERR_ARG;
    if (free_pages) *free_pages = (int32_t)c->free_list.size();
    if (cached_pages) *cached_pages = (int32_t)c->node_of.size();
    if (pinned_pages) *pinned_pages = c->pinned_pages;
    return 0;
}

}  // extern "C"
