// Launchers shared between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace msgl {

// ---------------------------------------------------------------- store
cudaError_t launch_store_kv(const PoolView &pool, __nv_bfloat16 *k_pool, __nv_bfloat16 *v_pool,
                            const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                            const int32_t *out_loc, int32_t n_tokens, uint32_t *status,
                            cudaStream_t stream);

// --------------------------------------------------------------- decode
struct DecodePlan {
    size_t o_bytes;       // bytes of the fp32 partial outputs (start of the workspace)
    size_t workspace;     // total bytes: partial outputs, then partial LSEs
};
DecodePlan plan_decode(int32_t num_reqs, int32_t hq, int32_t hkv, int32_t max_seq_len);

struct DecodeArgs {
    PoolView pool;
    PageView pages;
    const __nv_bfloat16 *q;
    const int32_t *seq_lens;
    int32_t num_reqs, hq, max_seq_len;
    float scale;
    __nv_bfloat16 *o;
    float *lse;
    float *part_o;      // [num_reqs + max CTAs, hq, 128] segment partials
    float *part_lse;    // [num_reqs + max CTAs, hq]
    uint32_t *status;
    const __nv_bfloat16 *k_new = nullptr, *v_new = nullptr;   // append mode (see msgl_attn_decode_append)
    const int32_t *new_loc = nullptr;
};
// Which kernels of a decode call to launch: the split (partials per key range), the
// merge (LSE fold of the partials, launched with programmatic dependent launch), or both.
enum class DecodePhase { kSplit, kMerge, kBoth };
cudaError_t launch_decode(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream,
                          DecodePhase phase = DecodePhase::kBoth);

// --------------------------------------------------------------- extend
size_t extend_workspace_bytes(int32_t num_reqs, int32_t total_tokens, int32_t hq, int32_t hkv,
                              int32_t max_seq_len);

struct ExtendArgs {
    PoolView pool;
    PageView pages;
    const __nv_bfloat16 *q;
    const int32_t *prefix_lens, *ext_lens, *cu_ext, *positions;
    int32_t num_reqs, total_tokens, hq, max_ext_len, max_seq_len;
    float scale;
    __nv_bfloat16 *o;
    float *lse;
    void *workspace;
    uint32_t *status;
    // launch with programmatic dependent launch: CTAs may start while the previous
    // kernel on the stream still runs (the grid's last CTA waits for that kernel, so the
    // grid does not complete before it)
    bool pdl = false;
};
cudaError_t launch_extend(const ExtendArgs &a, cudaStream_t stream);

// cuTensorMapEncodeTiled from the driver (NULL if unavailable); looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// SM count of the current device, queried once per device and cached (0..63;
// other ordinals are queried on every call).
int sm_count();

// Sets the text msgl_last_error() returns on this thread.
void set_last_error(const char *msg);

}  // namespace msgl
