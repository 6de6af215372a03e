// Extend (chunked prefill) step: chunk row i of request b attends keys
// 0..prefix_b + i of the request's pages ("Mini-SGLang 实战指南", §6.1
// "Chunked Prefill" and §6.5 "Radix Cache": a chunk runs over the cached
// prefix plus its own causal part).
#include "kernels.h"
#include "rows_kernel.cuh"

namespace msgl {

size_t extend_workspace_bytes(int32_t, int32_t, int32_t, int32_t, int32_t) { return 0; }

template <int G>
static void launch_rows_extend(const RowsArgs &r, dim3 grid, cudaStream_t stream) {
    attn_rows_kernel<G, true><<<grid, kRowsWarps * 32, 0, stream>>>(r);
}

cudaError_t launch_extend(const ExtendArgs &a, cudaStream_t stream) {
    if (a.num_reqs == 0 || a.total_tokens == 0 || a.max_ext_len == 0) return cudaSuccess;
    RowsArgs r{};
    r.pool = a.pool;
    r.pages = a.pages;
    r.q = a.q;
    r.hq = a.hq;
    r.total_tokens = a.total_tokens;
    r.scale_log2 = a.scale * kLog2e;
    r.max_seq_len = a.max_seq_len;
    r.prefix_lens = a.prefix_lens;
    r.ext_lens = a.ext_lens;
    r.cu_ext = a.cu_ext;
    r.positions = a.positions;
    r.chunk = a.max_seq_len;
    r.num_splits = 1;
    r.o = a.o;
    r.lse = a.lse;
    r.status = a.status;
    const int G = a.hq / a.pool.hkv;
    dim3 grid(a.max_ext_len, a.pool.hkv, a.num_reqs);
    switch (G) {
        case 1: launch_rows_extend<1>(r, grid, stream); break;
        case 2: launch_rows_extend<2>(r, grid, stream); break;
        case 3: launch_rows_extend<3>(r, grid, stream); break;
        case 4: launch_rows_extend<4>(r, grid, stream); break;
        case 5: launch_rows_extend<5>(r, grid, stream); break;
        case 6: launch_rows_extend<6>(r, grid, stream); break;
        case 7: launch_rows_extend<7>(r, grid, stream); break;
        case 8: launch_rows_extend<8>(r, grid, stream); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace msgl
