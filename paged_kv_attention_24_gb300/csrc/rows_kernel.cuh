// Row-at-a-time paged GQA attention on CUDA cores.
//
// One CTA = one query row x one kv head x one key chunk; its 4 warps stride
// over the chunk's keys, each lane owning 4 of the 128 dims, and keep a
// running (max, sum, weighted V) per q head of the group (online softmax in
// base 2 with the scale folded into log2 e).  The warps' states are merged
// in shared memory at the end.  Every key is located through the page table
// (slot = page_id * page_size + offset) with a range check; a bad index
// marks the row as failed instead of being read.
#pragma once

#include "common.cuh"

namespace msgl {

struct RowsArgs {
    PoolView pool;
    PageView pages;
    const __nv_bfloat16 *q;
    int32_t hq;
    int32_t total_tokens; // extend: rows in q / o
    float scale_log2;   // scale * log2(e)
    // decode: row b = request b, keys 0..seq_lens[b]-1
    const int32_t *seq_lens;
    int32_t max_seq_len;
    // extend: blockIdx.x = chunk row i of request b
    const int32_t *prefix_lens, *ext_lens, *cu_ext, *positions;
    int32_t chunk, num_splits;
    __nv_bfloat16 *o;     // final output (num_splits == 1)
    float *lse;
    float *part_o;        // split partials (num_splits > 1)
    float *part_lse;
    uint32_t *status;
};

constexpr int kRowsWarps = 4;

template <int G, bool EXTEND>
__global__ void __launch_bounds__(kRowsWarps * 32) attn_rows_kernel(const RowsArgs a) {
    const int b = blockIdx.z;
    const int g = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    __shared__ float q_s[G][kHeadDim];
    __shared__ float red_m[kRowsWarps][G], red_l[kRowsWarps][G];
    __shared__ float red_o[kRowsWarps][G][kHeadDim];
    __shared__ int bad_s;

    int split = 0, n_keys = 0, qrow = 0;
    bool row_bad = false;
    if (EXTEND) {
        const int i = blockIdx.x;
        const int ext = __ldg(a.ext_lens + b);
        if (i >= ext) return;
        const int pre = __ldg(a.prefix_lens + b);
        qrow = __ldg(a.cu_ext + b) + i;
        if (qrow < 0 || qrow >= a.total_tokens) {   // cu_ext inconsistent with total_tokens
            if (threadIdx.x == 0) report(a.status, MSGL_DEVERR_LENGTH);
            return;
        }
        n_keys = pre + i + 1;
        if (threadIdx.x == 0) {
            if (a.positions && __ldg(a.positions + qrow) != pre + i) report(a.status, MSGL_DEVERR_POSITION);
            if (__ldg(a.cu_ext + b + 1) - __ldg(a.cu_ext + b) != ext || pre < 0 || n_keys > a.max_seq_len ||
                (i == 0 && ext > (int)gridDim.x))
                report(a.status, MSGL_DEVERR_LENGTH);
        }
        if (pre < 0 || n_keys > a.max_seq_len) row_bad = true;
    } else {
        split = blockIdx.x;
        qrow = b;
        n_keys = __ldg(a.seq_lens + b);
        if (n_keys < 1 || n_keys > a.max_seq_len) {
            if (threadIdx.x == 0 && split == 0) report(a.status, MSGL_DEVERR_LENGTH);
            row_bad = true;
        }
    }
    const int k0 = split * a.chunk;
    const int k1 = row_bad ? k0 : min(n_keys, k0 + a.chunk);

    if (threadIdx.x == 0) bad_s = row_bad ? 1 : 0;
    for (int x = threadIdx.x; x < G * kHeadDim; x += blockDim.x) {
        const int h = x / kHeadDim, d = x % kHeadDim;
        q_s[h][d] = __bfloat162float(a.q[((int64_t)qrow * a.hq + g * G + h) * kHeadDim + d]);
    }
    __syncthreads();

    float qr[G][4], acc[G][4], m[G], l[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
        for (int e = 0; e < 4; ++e) { qr[h][e] = q_s[h][lane * 4 + e]; acc[h][e] = 0.f; }
        m[h] = -INFINITY;
        l[h] = 0.f;
    }
    const int64_t head_off = (int64_t)g * kHeadDim + lane * 4;
    const int64_t slot_stride = (int64_t)a.pool.hkv * kHeadDim;
    for (int j = k0 + warp; j < k1; j += kRowsWarps) {
        bool bad = false;
        const int64_t slot = slot_of(a.pool, a.pages, b, j, bad);
        if (bad) { bad_s = 1; continue; }
        const uint2 kk = *reinterpret_cast<const uint2 *>(a.pool.k + slot * slot_stride + head_off);
        const uint2 vv = *reinterpret_cast<const uint2 *>(a.pool.v + slot * slot_stride + head_off);
        const float kf[4] = {bf16_lo(kk.x), bf16_hi(kk.x), bf16_lo(kk.y), bf16_hi(kk.y)};
        const float vf[4] = {bf16_lo(vv.x), bf16_hi(vv.x), bf16_lo(vv.y), bf16_hi(vv.y)};
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float s = qr[h][0] * kf[0] + qr[h][1] * kf[1] + qr[h][2] * kf[2] + qr[h][3] * kf[3];
            s = warp_sum(s) * a.scale_log2;
            const float mn = fmaxf(m[h], s);
            const float alpha = exp2f(m[h] - mn);
            const float p = exp2f(s - mn);
            l[h] = l[h] * alpha + p;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[h][e] = acc[h][e] * alpha + p * vf[e];
            m[h] = mn;
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
        if (lane == 0) { red_m[warp][h] = m[h]; red_l[warp][h] = l[h]; }
#pragma unroll
        for (int e = 0; e < 4; ++e) red_o[warp][h][lane * 4 + e] = acc[h][e];
    }
    __syncthreads();
    const bool failed = bad_s != 0;
    if (threadIdx.x == 0 && failed && !row_bad) report(a.status, MSGL_DEVERR_PAGE_RANGE);
    for (int x = threadIdx.x; x < G * kHeadDim; x += blockDim.x) {
        const int h = x / kHeadDim, d = x % kHeadDim;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kRowsWarps; ++w) M = fmaxf(M, red_m[w][h]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kRowsWarps; ++w) {
                if (red_m[w][h] == -INFINITY) continue;
                const float f = exp2f(red_m[w][h] - M);
                L += red_l[w][h] * f;
                O += red_o[w][h][d] * f;
            }
        }
        const int hh = g * G + h;
        const bool empty = (L == 0.f);
        const float out = (failed || empty) ? 0.f : O / L;
        const float lse_v = (failed || empty) ? -INFINITY : (M + log2f(L)) * kLn2;
        if (a.num_splits == 1) {
            a.o[((int64_t)qrow * a.hq + hh) * kHeadDim + d] = __float2bfloat16_rn(out);
            if (d == 0) a.lse[(int64_t)qrow * a.hq + hh] = lse_v;
        } else {
            const int64_t pi = ((int64_t)b * a.hq + hh) * a.num_splits + split;
            a.part_o[pi * kHeadDim + d] = out;
            // a failed chunk is marked with NaN so that the merge zeroes the whole row
            if (d == 0) a.part_lse[pi] = failed ? __int_as_float(0x7fc00000) : lse_v;
        }
    }
}

}  // namespace msgl
