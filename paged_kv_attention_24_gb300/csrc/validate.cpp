// Host-side metadata checks (msgl_check_*_meta): the conditions the kernels
// check on the device, evaluated on host copies of the arrays so that a test
// or a debugging session learns which entry is wrong.  Nothing here touches
// the GPU.  What the metadata means: "不懂SGLang？从miniSGLang开始", §1.3
// item 3 (page table and positions locate each request's KV in the pool);
// "Mini-SGLang 实战指南", §6.1 (a chunk sits after its cached prefix) and
// §6.2 (the page is the pool's allocation unit).
#include <stdarg.h>
#include <stdio.h>

#include <unordered_set>

#include "../../include/msgl_attn.h"

namespace msgl {
void set_last_error(const char *msg);
}

namespace {

msgl_status bad(msgl_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
msgl_status bad(msgl_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    msgl::set_last_error(buf);
    return s;
}

bool pow2(int32_t x) { return x > 0 && (x & (x - 1)) == 0; }

// Pages of keys 0..n_keys-1 of request b: index below width, id inside the pool.
msgl_status check_pages(int64_t num_pages, int32_t page_size, const int32_t *page_ids, int32_t stride,
                        int32_t width, int32_t b, int64_t n_keys) {
    const int64_t n_pages = (n_keys + page_size - 1) / page_size;
    if (n_pages > width)
        return bad(MSGL_ERR_OUT_OF_RANGE, "request %d: %lld keys need %lld pages but the table width is %d", b,
                   (long long)n_keys, (long long)n_pages, width);
    for (int64_t p = 0; p < n_pages; ++p) {
        const int32_t id = page_ids[(int64_t)b * stride + p];
        if (id < 0 || id >= num_pages)
            return bad(MSGL_ERR_OUT_OF_RANGE, "request %d: page_ids[%lld] = %d is outside [0, %lld)", b,
                       (long long)p, id, (long long)num_pages);
    }
    return MSGL_OK;
}

msgl_status check_pool_scalars(int64_t num_slots, int32_t page_size, const int32_t *page_ids, int32_t stride,
                               int32_t width) {
    if (num_slots < 0) return bad(MSGL_ERR_INVALID_ARG, "num_slots must be >= 0");
    if (!pow2(page_size) || page_size > 256)
        return bad(MSGL_ERR_INVALID_ARG, "page_size %d is not a power of two in [1, 256]", page_size);
    if (num_slots % page_size) return bad(MSGL_ERR_INVALID_ARG, "num_slots is not a multiple of page_size");
    if (width < 0 || stride < width) return bad(MSGL_ERR_INVALID_ARG, "page table needs 0 <= width <= stride");
    if (!page_ids && width > 0) return bad(MSGL_ERR_INVALID_ARG, "page_ids is NULL");
    return MSGL_OK;
}

}  // namespace

extern "C" {

msgl_status msgl_check_store_meta(int64_t num_slots, const int32_t *out_loc, int32_t n_tokens) {
    msgl::set_last_error("");
    if (n_tokens < 0 || num_slots < 0) return bad(MSGL_ERR_INVALID_ARG, "n_tokens and num_slots must be >= 0");
    if (n_tokens > 0 && !out_loc) return bad(MSGL_ERR_INVALID_ARG, "out_loc is NULL");
    std::unordered_set<int32_t> seen;
    seen.reserve((size_t)n_tokens);
    for (int32_t t = 0; t < n_tokens; ++t) {
        const int32_t s = out_loc[t];
        if (s < 0 || s >= num_slots)
            return bad(MSGL_ERR_OUT_OF_RANGE, "out_loc[%d] = %d is outside [0, %lld)", t, s, (long long)num_slots);
        if (!seen.insert(s).second)
            return bad(MSGL_ERR_INVALID_ARG, "out_loc[%d] = %d names a slot an earlier row already writes", t, s);
    }
    return MSGL_OK;
}

msgl_status msgl_check_extend_meta(int64_t num_slots, int32_t page_size, const int32_t *page_ids, int32_t stride,
                                   int32_t width, const int32_t *prefix_lens, const int32_t *ext_lens,
                                   const int32_t *cu_ext, const int32_t *positions, int32_t num_reqs,
                                   int32_t total_tokens, int32_t max_ext_len, int32_t max_seq_len) {
    msgl::set_last_error("");
    msgl_status rc = check_pool_scalars(num_slots, page_size, page_ids, stride, width);
    if (rc) return rc;
    if (num_reqs < 0 || total_tokens < 0) return bad(MSGL_ERR_INVALID_ARG, "num_reqs and total_tokens must be >= 0");
    if (num_reqs > 0 && (!prefix_lens || !ext_lens || !cu_ext))
        return bad(MSGL_ERR_INVALID_ARG, "prefix_lens, ext_lens and cu_ext must be non-NULL");
    if (num_reqs == 0) {
        if (total_tokens != 0) return bad(MSGL_ERR_INVALID_ARG, "no requests but total_tokens = %d", total_tokens);
        return MSGL_OK;
    }
    if (cu_ext[0] != 0) return bad(MSGL_ERR_INVALID_ARG, "cu_ext[0] = %d, expected 0", cu_ext[0]);
    const int64_t num_pages = num_slots / page_size;
    for (int32_t b = 0; b < num_reqs; ++b) {
        const int32_t pre = prefix_lens[b], ext = ext_lens[b];
        if (pre < 0 || ext < 0)
            return bad(MSGL_ERR_INVALID_ARG, "request %d: prefix_len %d and ext_len %d must be >= 0", b, pre, ext);
        if ((int64_t)cu_ext[b + 1] - cu_ext[b] != ext)
            return bad(MSGL_ERR_INVALID_ARG, "request %d: cu_ext[%d] - cu_ext[%d] = %lld but ext_len = %d", b, b + 1,
                       b, (long long)cu_ext[b + 1] - cu_ext[b], ext);
        if (cu_ext[b + 1] > total_tokens)
            return bad(MSGL_ERR_INVALID_ARG, "cu_ext[%d] = %d exceeds total_tokens %d", b + 1, cu_ext[b + 1],
                       total_tokens);
        if (ext > max_ext_len)
            return bad(MSGL_ERR_INVALID_ARG, "request %d: ext_len %d exceeds max_ext_len %d", b, ext, max_ext_len);
        if ((int64_t)pre + ext > max_seq_len)
            return bad(MSGL_ERR_INVALID_ARG, "request %d: prefix_len + ext_len = %lld exceeds max_seq_len %d", b,
                       (long long)pre + ext, max_seq_len);
        if (positions)
            for (int32_t i = 0; i < ext; ++i)
                if (positions[cu_ext[b] + i] != pre + i)
                    return bad(MSGL_ERR_INVALID_ARG, "request %d row %d: positions[%d] = %d, expected %d", b, i,
                               cu_ext[b] + i, positions[cu_ext[b] + i], pre + i);
        if ((rc = check_pages(num_pages, page_size, page_ids, stride, width, b, (int64_t)pre + ext))) return rc;
    }
    if (cu_ext[num_reqs] != total_tokens)
        return bad(MSGL_ERR_INVALID_ARG, "cu_ext[%d] = %d but total_tokens = %d", num_reqs, cu_ext[num_reqs],
                   total_tokens);
    return MSGL_OK;
}

msgl_status msgl_check_decode_meta(int64_t num_slots, int32_t page_size, const int32_t *page_ids, int32_t stride,
                                   int32_t width, const int32_t *seq_lens, int32_t num_reqs, int32_t max_seq_len) {
    msgl::set_last_error("");
    msgl_status rc = check_pool_scalars(num_slots, page_size, page_ids, stride, width);
    if (rc) return rc;
    if (num_reqs < 0) return bad(MSGL_ERR_INVALID_ARG, "num_reqs must be >= 0");
    if (num_reqs > 0 && !seq_lens) return bad(MSGL_ERR_INVALID_ARG, "seq_lens is NULL");
    const int64_t num_pages = num_slots / page_size;
    for (int32_t b = 0; b < num_reqs; ++b) {
        const int32_t n = seq_lens[b];
        if (n < 1 || n > max_seq_len)
            return bad(MSGL_ERR_INVALID_ARG, "request %d: seq_len %d is outside [1, max_seq_len = %d]", b, n,
                       max_seq_len);
        if ((rc = check_pages(num_pages, page_size, page_ids, stride, width, b, n))) return rc;
    }
    return MSGL_OK;
}

}  // extern "C"
