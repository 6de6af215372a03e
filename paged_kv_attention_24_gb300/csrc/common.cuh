// Shared device helpers for libmsgl_attn (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/msgl_attn.h"

namespace msgl {

constexpr int kHeadDim = 128;          // the only head_dim the kernels are built for
constexpr int kMaxGroup = 64;          // largest q-heads-per-kv-head ratio supported
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// View of the pool as the kernels use it.
struct PoolView {
    const __nv_bfloat16 *k;
    const __nv_bfloat16 *v;
    int64_t num_slots;
    int32_t num_pages;   // num_slots / page_size
    int32_t log2_ps;     // page_size = 1 << log2_ps
    int32_t hkv;
};

struct PageView {
    const int32_t *ids;
    int32_t stride;
    int32_t width;
};

// Slot of key j of request b, or -1 (and *bad set) when the page index or id is out of range.
__device__ __forceinline__ int64_t slot_of(const PoolView &pool, const PageView &pt, int b, int j,
                                           bool &bad) {
    const int pidx = j >> pool.log2_ps;
    if (pidx >= pt.width) { bad = true; return -1; }
    const int pid = __ldg(pt.ids + (int64_t)b * pt.stride + pidx);
    if (pid < 0 || pid >= pool.num_pages) { bad = true; return -1; }
    return ((int64_t)pid << pool.log2_ps) + (j & ((1 << pool.log2_ps) - 1));
}

__device__ __forceinline__ void report(uint32_t *status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ uint4 ld_stream_16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_stream_16(void *p, uint4 r) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(r.x), "r"(r.y),
                 "r"(r.z), "r"(r.w)
                 : "memory");
}

}  // namespace msgl
