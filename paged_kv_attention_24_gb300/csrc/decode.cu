// Decode step: one query row per request over all of its pages, with the
// keys split into chunks that run in parallel and a log-sum-exp merge.
//
// "Mini-SGLang 实战指南", §6.3: decode has its own attention kernel, apart
// from prefill; §6.4: decode is replayed under CUDA graphs, so the launch
// shape depends only on host scalars (num_reqs, max_seq_len); chunks past a
// request's length exit at once.
#include <math.h>

#include "kernels.h"
#include "rows_kernel.cuh"

namespace msgl {

DecodePlan plan_decode(int32_t num_reqs, int32_t hq, int32_t hkv, int32_t max_seq_len) {
    DecodePlan p;
    const int64_t per_split = (int64_t)num_reqs * hkv;
    const int64_t target = 152 * 8;   // resident 128-thread CTAs on a full GPU
    int64_t splits = per_split > 0 ? (target + per_split - 1) / per_split : 1;
    const int64_t max_useful = ((int64_t)max_seq_len + 255) / 256;
    if (splits > max_useful) splits = max_useful;
    if (splits < 1) splits = 1;
    int64_t chunk = ((int64_t)max_seq_len + splits - 1) / splits;
    chunk = (chunk + 63) / 64 * 64;
    if (chunk < 64) chunk = 64;
    splits = ((int64_t)max_seq_len + chunk - 1) / chunk;
    if (splits < 1) splits = 1;
    p.num_splits = (int32_t)splits;
    p.chunk = (int32_t)chunk;
    const size_t n_part = (size_t)num_reqs * hq * (size_t)splits;
    const size_t o_bytes = (n_part * kHeadDim * sizeof(float) + 255) / 256 * 256;
    const size_t l_bytes = (n_part * sizeof(float) + 255) / 256 * 256;
    p.workspace = splits > 1 ? o_bytes + l_bytes : 0;   // one chunk writes o/lse directly
    return p;
}

// Merge the chunk partials of one (request, q head): weights exp(lse_s - max),
// o = sum w_s o_s / sum w_s, lse = max + ln(sum w_s).  A NaN partial lse marks
// a chunk that hit a bad index: the whole row is written as o = 0, lse = -inf.
__global__ void __launch_bounds__(kHeadDim) decode_merge_kernel(
    const float *__restrict__ part_o, const float *__restrict__ part_lse, int32_t num_splits,
    int32_t hq, __nv_bfloat16 *__restrict__ o, float *__restrict__ lse) {
    const int64_t bh = blockIdx.x;
    const int d = threadIdx.x;
    const float *pl = part_lse + bh * num_splits;
    float M = -INFINITY;
    bool failed = false;
    for (int s = 0; s < num_splits; ++s) {
        const float x = pl[s];
        if (isnan(x)) failed = true;
        else M = fmaxf(M, x);
    }
    float L = 0.f, O = 0.f;
    if (!failed && M != -INFINITY) {
        for (int s = 0; s < num_splits; ++s) {
            const float x = pl[s];
            if (x == -INFINITY) continue;
            const float w = __expf(x - M);
            L += w;
            O += w * part_o[(bh * num_splits + s) * kHeadDim + d];
        }
    }
    const bool zero = failed || L == 0.f;
    o[bh * kHeadDim + d] = __float2bfloat16_rn(zero ? 0.f : O / L);
    if (d == 0) lse[bh] = zero ? -INFINITY : M + logf(L);
}

template <int G>
static void launch_rows_decode(const RowsArgs &r, dim3 grid, cudaStream_t stream) {
    attn_rows_kernel<G, false><<<grid, kRowsWarps * 32, 0, stream>>>(r);
}

cudaError_t launch_decode(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream) {
    if (a.num_reqs == 0) return cudaSuccess;
    RowsArgs r{};
    r.pool = a.pool;
    r.pages = a.pages;
    r.q = a.q;
    r.hq = a.hq;
    r.scale_log2 = a.scale * kLog2e;
    r.seq_lens = a.seq_lens;
    r.max_seq_len = a.max_seq_len;
    r.chunk = plan.chunk;
    r.num_splits = plan.num_splits;
    r.o = a.o;
    r.lse = a.lse;
    r.part_o = a.part_o;
    r.part_lse = a.part_lse;
    r.status = a.status;
    const int G = a.hq / a.pool.hkv;
    dim3 grid(plan.num_splits, a.pool.hkv, a.num_reqs);
    switch (G) {
        case 1: launch_rows_decode<1>(r, grid, stream); break;
        case 2: launch_rows_decode<2>(r, grid, stream); break;
        case 3: launch_rows_decode<3>(r, grid, stream); break;
        case 4: launch_rows_decode<4>(r, grid, stream); break;
        case 5: launch_rows_decode<5>(r, grid, stream); break;
        case 6: launch_rows_decode<6>(r, grid, stream); break;
        case 7: launch_rows_decode<7>(r, grid, stream); break;
        case 8: launch_rows_decode<8>(r, grid, stream); break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || plan.num_splits == 1) return e;
    decode_merge_kernel<<<(unsigned)((int64_t)a.num_reqs * a.hq), kHeadDim, 0, stream>>>(
        a.part_o, a.part_lse, plan.num_splits, a.hq, a.o, a.lse);
    return cudaGetLastError();
}

}  // namespace msgl
