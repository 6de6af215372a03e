/*
 * Radix prefix cache and page allocator for the unified KV pool (host side).
 *
 * The engine keeps every request's KV in one pool allocated page by page,
 * and reuses the KV of prefixes that requests share through a radix tree
 * over token ids ("Mini-SGLang 实战指南", §6.2 "Page Size", §6.5 "Radix
 * Cache"; "不懂SGLang？从miniSGLang开始", §1.2 "调度引擎", item 3: a pool
 * and a manager).  This component produces the inputs of the attention
 * calls in include/msgl_attn.h: each request's page table and its cached
 * prefix length (prefix_lens of msgl_attn_extend).
 *
 * Model
 *   - The pool has num_pages pages of page_size tokens.  A page is free,
 *     cached (a node of the tree: the KV of one page-aligned chunk of some
 *     token prefix), or held by a running request.
 *   - A tree node is one full page.  Its key is the page's page_size token
 *     ids, and its path from the root spells the prefix.  Only whole pages
 *     are cached, so a match is always a multiple of page_size tokens.
 *   - msgl_radix_match pins the matched path, so those pages cannot be
 *     evicted while the request runs.  msgl_radix_insert (or
 *     msgl_radix_release) ends that lease.
 *   - msgl_radix_alloc takes free pages first, then evicts unpinned leaves,
 *     least recently matched or inserted first.
 *
 * The object is not thread-safe: one scheduler thread owns it.  Functions
 * return a negative value on error (see the codes below) and never abort.
 */
#ifndef MSGL_RADIX_H
#define MSGL_RADIX_H

#include <stdint.h>

#include "msgl_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

#define MSGL_RADIX_ERR_ARG (-1)       /* bad pointer or size */
#define MSGL_RADIX_ERR_NO_PAGES (-2)  /* not enough free or evictable pages */
#define MSGL_RADIX_ERR_LEASE (-3)     /* unknown or already ended lease */
#define MSGL_RADIX_ERR_PAGE (-4)      /* page id outside the pool */

typedef struct msgl_radix_cache msgl_radix_cache;

/* A cache over num_pages pages of page_size tokens, all free.  NULL on bad arguments. */
MSGL_API msgl_radix_cache *msgl_radix_create(int32_t page_size, int32_t num_pages);
MSGL_API void msgl_radix_destroy(msgl_radix_cache *c);

/*
 * Longest cached prefix of tokens[0..n) in whole pages.  Writes its page ids
 * (in sequence order) to out_pages (capacity cap) and returns the matched
 * token count (a multiple of page_size, at most n).  The matched pages are
 * pinned until the lease written to *lease ends; a match of length 0 still
 * opens a lease.
 */
MSGL_API int32_t msgl_radix_match(msgl_radix_cache *c, const int32_t *tokens, int32_t n,
                                  int32_t *out_pages, int32_t cap, int64_t *lease);

/* Take n pages for a running request (evicting cached leaves if needed). Returns n or an error. */
MSGL_API int32_t msgl_radix_alloc(msgl_radix_cache *c, int32_t n, int32_t *out_pages);

/*
 * A request finished (or a chunk completed): cache the full pages of
 * tokens[0..n), whose KV sits in pages[0..ceil(n/page_size)), and end the
 * lease.  A page whose prefix is already cached under another page id is
 * returned to the free list.  So is a trailing partial page.  Returns the
 * number of pages newly added to the tree.
 */
MSGL_API int32_t msgl_radix_insert(msgl_radix_cache *c, const int32_t *tokens, int32_t n,
                                   const int32_t *pages, int64_t lease);

/* End a lease without caching anything; pages[0..n_pages) (those the request held) become free. */
MSGL_API int32_t msgl_radix_release(msgl_radix_cache *c, int64_t lease, const int32_t *pages,
                                    int32_t n_pages);

/* Page counts: free, cached in the tree, cached and pinned by an open lease. */
MSGL_API int32_t msgl_radix_stats(const msgl_radix_cache *c, int32_t *free_pages, int32_t *cached_pages,
                                  int32_t *pinned_pages);

#ifdef __cplusplus
}
#endif

#endif /* MSGL_RADIX_H */
