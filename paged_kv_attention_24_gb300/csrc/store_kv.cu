// Store step: scatter the new K/V rows of a forward into their pool slots.
//
// "不懂SGLang？从miniSGLang开始", §1.3 "前向运算" item 1: the K/V that
// attention reads is the pool's history plus the newly computed K/V; all
// requests allocate from one unified pool (§1.2 item 3).  This kernel is the
// step that makes the new rows part of the pool.
//
// A pool row (one slot, all kv heads) is Hkv*128 bf16 = 2 KiB for Hkv = 8,
// i.e. 128 16-byte vectors.  One warp moves one row: each lane loads its
// vectors of the row's K and V (four each at Hkv = 8, all loads issued before
// the first store) and writes them to the slot, so every warp instruction
// touches 512 contiguous bytes.  The grid holds one warp per token up to the
// GPU's resident capacity (4 blocks of 8 warps per SM at <= 64 registers a
// thread), so all of a step's rows are issued in the first pass or two;
// larger batches stride.
#include "kernels.h"

namespace msgl {

namespace {

constexpr int kStoreThreads = 256;
constexpr int kStoreBlocksPerSm = 4;
constexpr int kStoreUnroll = 4;   // vectors of K (and of V) per lane per pass

__global__ void __launch_bounds__(kStoreThreads, kStoreBlocksPerSm) store_kv_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, uint4 *__restrict__ k_pool,
    uint4 *__restrict__ v_pool, const int32_t *__restrict__ out_loc, int32_t n_tokens,
    int32_t row_vec, int64_t num_slots, uint32_t *status) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * kStoreThreads) >> 5;
    for (int64_t t = ((int64_t)blockIdx.x * kStoreThreads + threadIdx.x) >> 5; t < n_tokens; t += nwarps) {
        const int64_t slot = __ldg(out_loc + t);
        if (slot < 0 || slot >= num_slots) {
            if (lane == 0) report(status, MSGL_DEVERR_SLOT_RANGE);
            continue;
        }
        const uint4 *ks = k + t * row_vec, *vs = v + t * row_vec;
        uint4 *kd = k_pool + slot * row_vec, *vd = v_pool + slot * row_vec;
        for (int c0 = 0; c0 < row_vec; c0 += 32 * kStoreUnroll) {
            uint4 kv[kStoreUnroll], vv[kStoreUnroll];
#pragma unroll
            for (int u = 0; u < kStoreUnroll; ++u) {
                const int c = c0 + u * 32 + lane;
                if (c < row_vec) {
                    kv[u] = ld_stream_16(ks + c);
                    vv[u] = ld_stream_16(vs + c);
                }
            }
#pragma unroll
            for (int u = 0; u < kStoreUnroll; ++u) {
                const int c = c0 + u * 32 + lane;
                if (c < row_vec) {
                    st_stream_16(kd + c, kv[u]);
                    st_stream_16(vd + c, vv[u]);
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_store_kv(const PoolView &pool, __nv_bfloat16 *k_pool, __nv_bfloat16 *v_pool,
                            const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                            const int32_t *out_loc, int32_t n_tokens, uint32_t *status,
                            cudaStream_t stream) {
    if (n_tokens == 0) return cudaSuccess;
    const int32_t row_vec = pool.hkv * kHeadDim * 2 / 16;
    const int64_t want = ((int64_t)n_tokens + kStoreThreads / 32 - 1) / (kStoreThreads / 32);
    const int64_t cap = (int64_t)sm_count() * kStoreBlocksPerSm;
    const int grid = (int)(want < cap ? want : cap);
    store_kv_kernel<<<grid, kStoreThreads, 0, stream>>>(
        reinterpret_cast<const uint4 *>(k), reinterpret_cast<const uint4 *>(v),
        reinterpret_cast<uint4 *>(k_pool), reinterpret_cast<uint4 *>(v_pool), out_loc, n_tokens,
        row_vec, pool.num_slots, status);
    return cudaGetLastError();
}

}  // namespace msgl
