// The C ABI of libmsgl_attn: argument checks, launch planning and status
// reporting.  Every compute step runs in the kernels of the other files.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "kernels.h"

namespace {

thread_local char g_last_error[512];

msgl_status fail(msgl_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
msgl_status fail(msgl_status s, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return s;
}

msgl_status cuda_fail(cudaError_t e, const char *what) {
    return fail(MSGL_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int log2_exact(int32_t x) {
    if (x <= 0 || (x & (x - 1)) != 0) return -1;
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

// Checks shared by every call on the pool; fills the kernels' view of it.
msgl_status check_pool(const msgl_kv_pool *pool, msgl::PoolView &view) {
    if (!pool) return fail(MSGL_ERR_INVALID_ARG, "pool is NULL");
    if (!pool->k_pool || !pool->v_pool) return fail(MSGL_ERR_INVALID_ARG, "pool buffers are NULL");
    if (!aligned16(pool->k_pool) || !aligned16(pool->v_pool))
        return fail(MSGL_ERR_INVALID_ARG, "pool buffers must be 16-byte aligned");
    if (pool->head_dim != msgl::kHeadDim)
        return fail(MSGL_ERR_UNSUPPORTED, "head_dim %d is not supported (only 128)", pool->head_dim);
    if (pool->num_kv_heads <= 0) return fail(MSGL_ERR_INVALID_ARG, "num_kv_heads must be > 0");
    if (pool->num_kv_heads > 64) return fail(MSGL_ERR_UNSUPPORTED, "num_kv_heads > 64");
    const int l2 = log2_exact(pool->page_size);
    if (l2 < 0 || pool->page_size > 256)
        return fail(MSGL_ERR_UNSUPPORTED, "page_size %d is not a power of two in [1, 256]", pool->page_size);
    if (pool->num_slots < 0 || pool->num_slots % pool->page_size != 0)
        return fail(MSGL_ERR_INVALID_ARG, "num_slots must be a non-negative multiple of page_size");
    if (pool->num_slots / pool->page_size > INT32_MAX)
        return fail(MSGL_ERR_UNSUPPORTED, "more than 2^31-1 pages");
    view.k = static_cast<const __nv_bfloat16 *>(pool->k_pool);
    view.v = static_cast<const __nv_bfloat16 *>(pool->v_pool);
    view.num_slots = pool->num_slots;
    view.num_pages = (int32_t)(pool->num_slots / pool->page_size);
    view.log2_ps = l2;
    view.hkv = pool->num_kv_heads;
    return MSGL_OK;
}

msgl_status check_pages(const msgl_page_table *pages, int32_t num_reqs, msgl::PageView &view) {
    if (!pages) return fail(MSGL_ERR_INVALID_ARG, "page table is NULL");
    if (num_reqs > 0 && !pages->page_ids) return fail(MSGL_ERR_INVALID_ARG, "page_ids is NULL");
    if (pages->width < 0 || pages->stride < pages->width)
        return fail(MSGL_ERR_INVALID_ARG, "page table needs 0 <= width <= stride");
    view.ids = pages->page_ids;
    view.stride = pages->stride;
    view.width = pages->width;
    return MSGL_OK;
}

msgl_status check_heads(int32_t hq, int32_t hkv) {
    if (hq <= 0 || hq % hkv != 0)
        return fail(MSGL_ERR_INVALID_ARG, "num_q_heads %d is not a positive multiple of num_kv_heads %d", hq, hkv);
    if (hq / hkv > msgl::kMaxGroup)
        return fail(MSGL_ERR_UNSUPPORTED, "more than %d q heads per kv head", msgl::kMaxGroup);
    return MSGL_OK;
}

msgl_status check_scale(float scale) {
    if (!(scale > 0.f) || !isfinite(scale)) return fail(MSGL_ERR_INVALID_ARG, "scale must be finite and > 0");
    return MSGL_OK;
}

}  // namespace

namespace msgl {
// Lets other translation units of the library set this thread's error text.
void set_last_error(const char *msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

int sm_count() {
    static int cached[64];   // per device; racing first calls store the same value
    int dev = 0;
    cudaGetDevice(&dev);
    int sms = (dev >= 0 && dev < 64) ? cached[dev] : 0;
    if (sms == 0) {
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
        if (dev >= 0 && dev < 64) cached[dev] = sms;
    }
    return sms;
}
}  // namespace msgl

// Validates a decode call and fills its kernel arguments (a.num_reqs = 0: nothing to launch).
static msgl_status prepare_decode(const msgl_kv_pool *pool, const msgl_page_table *pages, const void *q,
                                  int32_t num_q_heads, const void *k_new, const void *v_new,
                                  const int32_t *new_loc, const int32_t *seq_lens, int32_t num_reqs,
                                  int32_t max_seq_len, float scale, void *o, float *lse, void *workspace,
                                  size_t workspace_bytes, uint32_t *status, msgl::DecodeArgs &a,
                                  msgl::DecodePlan &plan) {
    msgl::PoolView pv;
    msgl::PageView pg;
    msgl_status s = check_pool(pool, pv);
    if (s) return s;
    if ((s = check_heads(num_q_heads, pool->num_kv_heads))) return s;
    if ((s = check_scale(scale))) return s;
    if (num_reqs < 0) return fail(MSGL_ERR_INVALID_ARG, "num_reqs < 0");
    a = msgl::DecodeArgs{};
    a.num_reqs = num_reqs;
    if (num_reqs == 0) return MSGL_OK;
    if ((s = check_pages(pages, num_reqs, pg))) return s;
    if (max_seq_len <= 0) return fail(MSGL_ERR_INVALID_ARG, "max_seq_len must be > 0");
    if (!q || !seq_lens || !o || !lse) return fail(MSGL_ERR_INVALID_ARG, "q, seq_lens, o and lse must be non-NULL");
    if (!aligned16(q) || !aligned16(o)) return fail(MSGL_ERR_INVALID_ARG, "q and o must be 16-byte aligned");
    plan = msgl::plan_decode(num_reqs, num_q_heads, pool->num_kv_heads, max_seq_len);
    if (!workspace || workspace_bytes < plan.workspace)
        return fail(MSGL_ERR_WORKSPACE, "decode needs %zu workspace bytes, got %zu", plan.workspace,
                    workspace ? workspace_bytes : (size_t)0);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(MSGL_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    a.pool = pv;
    a.pages = pg;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.seq_lens = seq_lens;
    a.hq = num_q_heads;
    a.max_seq_len = max_seq_len;
    a.scale = scale;
    a.o = static_cast<__nv_bfloat16 *>(o);
    a.lse = lse;
    a.part_o = static_cast<float *>(workspace);
    a.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) + plan.o_bytes);
    a.status = status;
    a.k_new = static_cast<const __nv_bfloat16 *>(k_new);
    a.v_new = static_cast<const __nv_bfloat16 *>(v_new);
    a.new_loc = new_loc;
    return MSGL_OK;
}

static msgl_status decode_impl(const msgl_kv_pool *pool, const msgl_page_table *pages, const void *q,
                               int32_t num_q_heads, const void *k_new, const void *v_new,
                               const int32_t *new_loc, const int32_t *seq_lens, int32_t num_reqs,
                               int32_t max_seq_len, float scale, void *o, float *lse, void *workspace,
                               size_t workspace_bytes, uint32_t *status, msgl_stream_t stream) {
    g_last_error[0] = 0;
    msgl::DecodeArgs a;
    msgl::DecodePlan plan{};
    msgl_status s = prepare_decode(pool, pages, q, num_q_heads, k_new, v_new, new_loc, seq_lens, num_reqs,
                                   max_seq_len, scale, o, lse, workspace, workspace_bytes, status, a, plan);
    if (s || num_reqs == 0) return s;
    cudaError_t e = msgl::launch_decode(a, plan, (cudaStream_t)stream);
    return e == cudaSuccess ? MSGL_OK : cuda_fail(e, "decode launch");
}

// Validates an extend call and fills its kernel arguments (a.num_reqs = 0: nothing to launch).
static msgl_status prepare_extend(const msgl_kv_pool *pool, const msgl_page_table *pages, const void *q,
                                  int32_t num_q_heads, const int32_t *prefix_lens, const int32_t *ext_lens,
                                  const int32_t *cu_ext, const int32_t *positions, int32_t num_reqs,
                                  int32_t total_tokens, int32_t max_ext_len, int32_t max_seq_len, float scale,
                                  void *o, float *lse, void *workspace, size_t workspace_bytes,
                                  uint32_t *status, msgl::ExtendArgs &a) {
    msgl::PoolView pv;
    msgl::PageView pg;
    msgl_status s = check_pool(pool, pv);
    if (s) return s;
    if ((s = check_heads(num_q_heads, pool->num_kv_heads))) return s;
    if ((s = check_scale(scale))) return s;
    if (num_reqs < 0 || total_tokens < 0 || max_ext_len < 0 || max_seq_len < 0)
        return fail(MSGL_ERR_INVALID_ARG, "negative size");
    a = msgl::ExtendArgs{};
    if (num_reqs == 0 || total_tokens == 0) return MSGL_OK;
    if ((s = check_pages(pages, num_reqs, pg))) return s;
    if (max_ext_len == 0 || max_seq_len < max_ext_len)
        return fail(MSGL_ERR_INVALID_ARG, "need 0 < max_ext_len <= max_seq_len");
    if (!q || !prefix_lens || !ext_lens || !cu_ext || !o || !lse)
        return fail(MSGL_ERR_INVALID_ARG, "q, prefix_lens, ext_lens, cu_ext, o and lse must be non-NULL");
    if (!aligned16(q) || !aligned16(o)) return fail(MSGL_ERR_INVALID_ARG, "q and o must be 16-byte aligned");
    const size_t need = msgl::extend_workspace_bytes(num_reqs, total_tokens, num_q_heads,
                                                     pool->num_kv_heads, max_seq_len);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(MSGL_ERR_WORKSPACE, "extend needs %zu workspace bytes", need);
    a.pool = pv;
    a.pages = pg;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.prefix_lens = prefix_lens;
    a.ext_lens = ext_lens;
    a.cu_ext = cu_ext;
    a.positions = positions;
    a.num_reqs = num_reqs;
    a.total_tokens = total_tokens;
    a.hq = num_q_heads;
    a.max_ext_len = max_ext_len;
    a.max_seq_len = max_seq_len;
    a.scale = scale;
    a.o = static_cast<__nv_bfloat16 *>(o);
    a.lse = lse;
    a.workspace = workspace;
    a.status = status;
    return MSGL_OK;
}

extern "C" {

int32_t msgl_abi_version(void) { return MSGL_ABI_VERSION; }

const char *msgl_last_error(void) { return g_last_error; }

const char *msgl_status_string(msgl_status s) {
    switch (s) {
        case MSGL_OK: return "ok";
        case MSGL_ERR_INVALID_ARG: return "invalid argument";
        case MSGL_ERR_UNSUPPORTED: return "unsupported argument";
        case MSGL_ERR_CUDA: return "CUDA error";
        case MSGL_ERR_OUT_OF_RANGE: return "device index out of range";
        case MSGL_ERR_TIMEOUT: return "in-kernel wait timed out";
        case MSGL_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

msgl_status msgl_store_kv(const msgl_kv_pool *pool, const void *k, const void *v,
                          const int32_t *out_loc, int32_t n_tokens, uint32_t *status,
                          msgl_stream_t stream) {
    g_last_error[0] = 0;
    msgl::PoolView pv;
    msgl_status s = check_pool(pool, pv);
    if (s) return s;
    if (n_tokens < 0) return fail(MSGL_ERR_INVALID_ARG, "n_tokens < 0");
    if (n_tokens == 0) return MSGL_OK;
    if (!k || !v || !out_loc) return fail(MSGL_ERR_INVALID_ARG, "k, v and out_loc must be non-NULL");
    if (!aligned16(k) || !aligned16(v)) return fail(MSGL_ERR_INVALID_ARG, "k and v must be 16-byte aligned");
    cudaError_t e = msgl::launch_store_kv(pv, static_cast<__nv_bfloat16 *>(pool->k_pool),
                                          static_cast<__nv_bfloat16 *>(pool->v_pool),
                                          static_cast<const __nv_bfloat16 *>(k),
                                          static_cast<const __nv_bfloat16 *>(v), out_loc, n_tokens,
                                          status, (cudaStream_t)stream);
    return e == cudaSuccess ? MSGL_OK : cuda_fail(e, "store_kv launch");
}

size_t msgl_decode_workspace_size(int32_t num_reqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_seq_len) {
    if (num_reqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim != msgl::kHeadDim ||
        max_seq_len <= 0)
        return 0;
    return msgl::plan_decode(num_reqs, num_q_heads, num_kv_heads, max_seq_len).workspace;
}

msgl_status msgl_attn_decode(const msgl_kv_pool *pool, const msgl_page_table *pages,
                             const void *q, int32_t num_q_heads, const int32_t *seq_lens,
                             int32_t num_reqs, int32_t max_seq_len, float scale, void *o,
                             float *lse, void *workspace, size_t workspace_bytes,
                             uint32_t *status, msgl_stream_t stream) {
    return decode_impl(pool, pages, q, num_q_heads, nullptr, nullptr, nullptr, seq_lens, num_reqs,
                       max_seq_len, scale, o, lse, workspace, workspace_bytes, status, stream);
}

msgl_status msgl_attn_decode_append(const msgl_kv_pool *pool, const msgl_page_table *pages,
                                    const void *q, int32_t num_q_heads, const void *k_new,
                                    const void *v_new, const int32_t *new_loc,
                                    const int32_t *seq_lens, int32_t num_reqs, int32_t max_seq_len,
                                    float scale, void *o, float *lse, void *workspace,
                                    size_t workspace_bytes, uint32_t *status, msgl_stream_t stream) {
    g_last_error[0] = 0;
    if (num_reqs > 0) {
        if (!k_new || !v_new || !new_loc)
            return fail(MSGL_ERR_INVALID_ARG, "k_new, v_new and new_loc must be non-NULL");
        if (!aligned16(k_new) || !aligned16(v_new))
            return fail(MSGL_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    }
    return decode_impl(pool, pages, q, num_q_heads, k_new, v_new, new_loc, seq_lens, num_reqs,
                       max_seq_len, scale, o, lse, workspace, workspace_bytes, status, stream);
}

size_t msgl_extend_workspace_size(int32_t num_reqs, int32_t total_tokens, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t max_seq_len) {
    if (num_reqs <= 0 || total_tokens <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        head_dim != msgl::kHeadDim)
        return 0;
    return msgl::extend_workspace_bytes(num_reqs, total_tokens, num_q_heads, num_kv_heads, max_seq_len);
}

msgl_status msgl_attn_extend(const msgl_kv_pool *pool, const msgl_page_table *pages,
                             const void *q, int32_t num_q_heads, const int32_t *prefix_lens,
                             const int32_t *ext_lens, const int32_t *cu_ext,
                             const int32_t *positions, int32_t num_reqs, int32_t total_tokens,
                             int32_t max_ext_len, int32_t max_seq_len, float scale, void *o,
                             float *lse, void *workspace, size_t workspace_bytes,
                             uint32_t *status, msgl_stream_t stream) {
    g_last_error[0] = 0;
    msgl::ExtendArgs a;
    msgl_status s = prepare_extend(pool, pages, q, num_q_heads, prefix_lens, ext_lens, cu_ext, positions,
                                   num_reqs, total_tokens, max_ext_len, max_seq_len, scale, o, lse, workspace,
                                   workspace_bytes, status, a);
    if (s || a.num_reqs == 0) return s;
    cudaError_t e = msgl::launch_extend(a, (cudaStream_t)stream);
    return e == cudaSuccess ? MSGL_OK : cuda_fail(e, "extend launch");
}

msgl_status msgl_attn_mixed(const msgl_kv_pool *pool, const msgl_extend_batch *ext, const msgl_decode_batch *dec,
                            int32_t num_q_heads, float scale, void *workspace, size_t workspace_bytes,
                            uint32_t *status, msgl_stream_t stream) {
    g_last_error[0] = 0;
    if (!ext || !dec) return fail(MSGL_ERR_INVALID_ARG, "ext and dec must be non-NULL");
    // the decode partials take the front of the workspace, the extend's share follows
    msgl::DecodeArgs da;
    msgl::DecodePlan plan{};
    msgl_status s = prepare_decode(pool, &dec->pages, dec->q, num_q_heads, nullptr, nullptr, nullptr,
                                   dec->seq_lens, dec->num_reqs, dec->max_seq_len, scale, dec->o, dec->lse,
                                   workspace, workspace_bytes, status, da, plan);
    if (s) return s;
    const size_t dec_bytes = dec->num_reqs > 0 ? (plan.workspace + 255) / 256 * 256 : 0;
    msgl::ExtendArgs ea;
    void *ext_ws = workspace && workspace_bytes > dec_bytes ? static_cast<char *>(workspace) + dec_bytes : nullptr;
    s = prepare_extend(pool, &ext->pages, ext->q, num_q_heads, ext->prefix_lens, ext->ext_lens, ext->cu_ext,
                       ext->positions, ext->num_reqs, ext->total_tokens, ext->max_ext_len, ext->max_seq_len,
                       scale, ext->o, ext->lse, ext_ws, ext_ws ? workspace_bytes - dec_bytes : 0, status, ea);
    if (s) return s;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    if (da.num_reqs > 0 && ea.num_reqs > 0) {
        // split first; the extend's CTAs fill SMs as the split's ranges finish; merge last
        e = msgl::launch_decode(da, plan, st, msgl::DecodePhase::kSplit);
        if (e == cudaSuccess) {
            ea.pdl = true;
            e = msgl::launch_extend(ea, st);
        }
        if (e == cudaSuccess) e = msgl::launch_decode(da, plan, st, msgl::DecodePhase::kMerge);
    } else if (da.num_reqs > 0) {
        e = msgl::launch_decode(da, plan, st);
    } else if (ea.num_reqs > 0) {
        e = msgl::launch_extend(ea, st);
    }
    return e == cudaSuccess ? MSGL_OK : cuda_fail(e, "mixed step launch");
}

msgl_status msgl_read_status(const uint32_t *status, uint32_t *flags, msgl_stream_t stream) {
    g_last_error[0] = 0;
    if (!status) return fail(MSGL_ERR_INVALID_ARG, "status is NULL");
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    uint32_t h = 0;
    e = cudaMemcpy(&h, status, sizeof h, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status copy");
    if (flags) *flags = h;
    if (h == 0) return MSGL_OK;
    if (h & MSGL_DEVERR_TIMEOUT) return MSGL_ERR_TIMEOUT;
    return MSGL_ERR_OUT_OF_RANGE;
}

}  // extern "C"
