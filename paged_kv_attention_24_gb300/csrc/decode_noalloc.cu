// Decode without caller-provided workspace, for callers that cannot allocate
// device memory.
//
// msgl_attn_decode needs scratch for its key-chunk partials, which the
// caller normally allocates (msgl_decode_workspace_size bytes).  Some
// callers cannot do that: an engine whose device memory is all handed out
// by a host-side pool planned at start-up (a stray cudaMalloc would break
// its budget or fragment it), a plugin interface that only passes in the
// input and output pointers, or a latency-critical loop where cudaMalloc's
// implicit device synchronisation would stall every other stream.  For
// them, msgl_attn_decode_noalloc takes its scratch from a fixed array that
// lives in this library's device image instead.
//
// The array is MSGL_DECODE_NOALLOC_SCRATCH_BYTES (32 MiB) of device memory
// reserved on every GPU that loads the library, held until the process
// exits.  Host code cannot use the array's name as a device address (on the
// host it names a stand-in object), so the first call on each device looks
// up the real address with cudaGetSymbolAddress while that device is
// current, and caches it.  Under lazy module loading that lookup is also
// what loads the module and places the array on the device, so callers make
// their first call at start-up.  The cache is keyed by device ordinal: it
// assumes one context per device for the life of the process (a device
// reset or another driver-API context needs a fresh process).
//
// All calls on a device share the one array and it keeps whatever the last
// call left in it.  Nothing has to start at zero: every partial the merge
// reads is written earlier in the same call.  Two calls whose kernels
// overlap on the GPU (different streams, no ordering between them) write
// the same scratch and race; order them on one stream or with events.
#include <mutex>
#include <stdio.h>

#include "kernels.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[MSGL_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once per device).
msgl_status scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
        msgl::set_last_error(msg);
        return MSGL_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        msgl::set_last_error("device ordinal beyond the scratch table (64 devices)");
        return MSGL_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess || !p) {
            char msg[256];
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
            msgl::set_last_error(msg);
            return MSGL_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MSGL_OK;
}

}  // namespace

extern "C" msgl_status msgl_attn_decode_noalloc(const msgl_kv_pool *pool, const msgl_page_table *pages,
                                                const void *q, int32_t num_q_heads,
                                                const int32_t *seq_lens, int32_t num_reqs,
                                                int32_t max_seq_len, float scale, void *o, float *lse,
                                                uint32_t *status, msgl_stream_t stream) {
    if (pool && num_reqs > 0) {
        const size_t need = msgl_decode_workspace_size(num_reqs, num_q_heads, pool->num_kv_heads,
                                                       pool->head_dim, max_seq_len);
        if (need > (size_t)MSGL_DECODE_NOALLOC_SCRATCH_BYTES) {
            char msg[256];
            snprintf(msg, sizeof msg,
                     "this decode needs %zu scratch bytes but the built-in scratch holds %zu; "
                     "use msgl_attn_decode with a caller workspace or a smaller batch",
                     need, (size_t)MSGL_DECODE_NOALLOC_SCRATCH_BYTES);
            msgl::set_last_error(msg);
            return MSGL_ERR_WORKSPACE;
        }
    }
    void *scratch = nullptr;
    msgl_status s = scratch_address(&scratch);
    if (s != MSGL_OK) return s;
    return msgl_attn_decode(pool, pages, q, num_q_heads, seq_lens, num_reqs, max_seq_len, scale, o,
                            lse, scratch, (size_t)MSGL_DECODE_NOALLOC_SCRATCH_BYTES, status, stream);
}
