// Store step: scatter the new K/V rows of a forward into their pool slots.
//
// "不懂SGLang？从miniSGLang开始", §1.3 "前向运算" item 1: the K/V that
// attention reads is the pool's history plus the newly computed K/V; all
// requests allocate from one unified pool (§1.2 item 3).  This kernel is the
// step that makes the new rows part of the pool.
//
// A pool row (one slot, all kv heads) is Hkv*128 bf16 = 2 KiB for Hkv = 8,
// i.e. 128 16-byte vectors.  Consecutive threads copy consecutive vectors of
// a row, so every warp reads and writes 512 contiguous bytes; each token's
// slot index is read once per vector (it stays in L1).  The grid is a
// multiple of the SM count and strides over the whole copy.
#include "kernels.h"

namespace msgl {

__global__ void __launch_bounds__(256) store_kv_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, uint4 *__restrict__ k_pool,
    uint4 *__restrict__ v_pool, const int32_t *__restrict__ out_loc, int64_t n_vec,
    int32_t row_vec, int64_t num_slots, uint32_t *status) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec; i += stride) {
        const int64_t t = i / row_vec;
        const int32_t c = (int32_t)(i - t * row_vec);
        const int64_t slot = __ldg(out_loc + t);
        if (slot < 0 || slot >= num_slots) {
            if (c == 0) report(status, MSGL_DEVERR_SLOT_RANGE);
            continue;
        }
        const uint4 kv = ld_stream_16(k + i);
        const uint4 vv = ld_stream_16(v + i);
        st_stream_16(k_pool + slot * row_vec + c, kv);
        st_stream_16(v_pool + slot * row_vec + c, vv);
    }
}

cudaError_t launch_store_kv(const PoolView &pool, __nv_bfloat16 *k_pool, __nv_bfloat16 *v_pool,
                            const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                            const int32_t *out_loc, int32_t n_tokens, uint32_t *status,
                            cudaStream_t stream) {
    if (n_tokens == 0) return cudaSuccess;
    const int32_t row_vec = pool.hkv * kHeadDim * 2 / 16;
    const int64_t n_vec = (int64_t)n_tokens * row_vec;
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = (n_vec + 255) / 256;
    const int64_t cap = (int64_t)sms * 8;
    const int grid = (int)(want < cap ? want : cap);
    store_kv_kernel<<<grid, 256, 0, stream>>>(
        reinterpret_cast<const uint4 *>(k), reinterpret_cast<const uint4 *>(v),
        reinterpret_cast<uint4 *>(k_pool), reinterpret_cast<uint4 *>(v_pool), out_loc, n_vec,
        row_vec, pool.num_slots, status);
    return cudaGetLastError();
}

}  // namespace msgl
