/*
 * libmsgl_attn — paged-KV grouped-query attention for GB300 (sm_103a).
 *
 * The attention step a Mini-SGLang-style serving engine runs every forward:
 * new K/V rows are scattered into a unified, paged KV pool, then prefill
 * chunks ("extend") and single-token decode rows attend over each request's
 * pages.  The pages describing the engine define the pieces this ABI takes:
 *
 *   - one unified KV pool, allocated in pages of a configurable size
 *     ("Mini-SGLang 实战指南", §6.2 "Page Size"; §6.5 "Radix Cache";
 *     "不懂SGLang？从miniSGLang开始", §1.2 "调度引擎", item 3);
 *   - attention reads the pool's history plus the newly computed K/V, and
 *     locates each request's data through the page table and positions
 *     ("不懂SGLang？从miniSGLang开始", §1.3 "前向运算", items 1 and 3);
 *   - prefill runs in chunks over a cached (radix-shared) prefix
 *     ("Mini-SGLang 实战指南", §6.1 "Chunked Prefill", §6.5);
 *   - prefill and decode are separate attention calls
 *     ("Mini-SGLang 实战指南", §6.3).
 *
 * Definitions used by every call (the pages fix no formula; this is the
 * plain reading of causal softmax attention with grouped heads):
 *   G        = num_q_heads / num_kv_heads (1..64); q head h reads kv head h / G
 *   slot(j)  = page_table[b][j / page_size] * page_size + j % page_size
 *   a query row at absolute position p attends keys j = 0..p:
 *   s_j = scale * <q, K[slot(j)][h/G]>,  o = sum_j softmax(s)_j V[slot(j)][h/G],
 *   lse = ln(sum_j exp(s_j))   (natural log, fp32)
 *
 * Conventions
 *   - Every pointer named "device" is CUDA device memory owned by the
 *     caller; the library allocates nothing, keeps no state between calls
 *     and never frees caller memory.  All calls are asynchronous on
 *     `stream` (NULL = the legacy default stream) except msgl_read_status.
 *   - bf16 tensors are row-major, contiguous, 16-byte aligned.
 *   - Host-side validation failures return before anything is launched.
 *   - Device-side index errors never trap: the kernel ORs a bit into the
 *     caller's status word (when `status` is non-NULL), skips the bad
 *     access and writes that output row as o = 0, lse = -inf.
 *   - Waits inside kernels are bounded; a wait that gives up sets
 *     MSGL_DEVERR_TIMEOUT and the kernel returns.
 */
#ifndef MSGL_ATTN_H
#define MSGL_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSGL_ABI_VERSION 1

#if defined(__GNUC__)
#define MSGL_API __attribute__((visibility("default")))
#else
#define MSGL_API
#endif

/* A cudaStream_t (the runtime and driver stream handle types are the same pointer). */
typedef struct CUstream_st *msgl_stream_t;

typedef enum msgl_status {
    MSGL_OK = 0,
    MSGL_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or scalar */
    MSGL_ERR_UNSUPPORTED = 2,   /* valid but not implemented (head_dim != 128, G > 64, ...) */
    MSGL_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (launch, copy) */
    MSGL_ERR_OUT_OF_RANGE = 4,  /* reported by msgl_read_status: device index error */
    MSGL_ERR_TIMEOUT = 5,       /* reported by msgl_read_status: a bounded wait gave up */
    MSGL_ERR_WORKSPACE = 6      /* workspace missing or smaller than the size query */
} msgl_status;

/* Bits of the device status word (uint32, caller-owned device memory). */
#define MSGL_DEVERR_SLOT_RANGE 0x1u  /* out_loc entry outside [0, num_slots) */
#define MSGL_DEVERR_PAGE_RANGE 0x2u  /* page index >= width, or page id outside the pool */
#define MSGL_DEVERR_LENGTH 0x4u      /* decode seq_len < 1, or lengths inconsistent with cu_ext */
#define MSGL_DEVERR_POSITION 0x8u    /* positions[t] != prefix_len + i for chunk row i */
#define MSGL_DEVERR_TIMEOUT 0x10u    /* a bounded in-kernel wait gave up */
#define MSGL_DEVERR_APPEND_SLOT 0x20u /* decode_append: new_loc[b] is not the slot of key seq_lens[b]-1 */

/*
 * The unified KV pool of one layer.  k_pool and v_pool are device bf16
 * [num_slots, num_kv_heads, head_dim], slot-major (the row of one slot is
 * num_kv_heads*head_dim contiguous elements).  num_slots must be a multiple
 * of page_size; page_size is a power of two in [1, 256]; head_dim must be 128.
 */
typedef struct msgl_kv_pool {
    void *k_pool;
    void *v_pool;
    int64_t num_slots;
    int32_t page_size;
    int32_t num_kv_heads;
    int32_t head_dim;
} msgl_kv_pool;

/*
 * Per-request page table: device int32 [num_reqs, stride]; row b lists the
 * page ids of request b in sequence order.  Only the first `width` entries
 * of a row may be read; a key whose page index reaches `width`, or whose
 * page id lies outside [0, num_slots/page_size), is a device index error.
 */
typedef struct msgl_page_table {
    const int32_t *page_ids;
    int32_t stride;
    int32_t width;
} msgl_page_table;

/*
 * Store step: write the new K/V rows of this forward into the pool
 * ("不懂SGLang？从miniSGLang开始", §1.3 item 1: the KV an attention call
 * reads is the pool's history plus the newly computed KV; every request
 * allocates from the one pool, §1.2 item 3).
 *
 *   k, v     device bf16 [n_tokens, num_kv_heads, head_dim]
 *   out_loc  device int32 [n_tokens]; row t goes to slot out_loc[t]
 *   status   device uint32 or NULL
 * Pool rows not named in out_loc are untouched.  Duplicate slots in out_loc
 * are undefined (one of the rows wins).  An out-of-range slot sets
 * MSGL_DEVERR_SLOT_RANGE and that row is skipped.  The copy is bit-exact.
 */
MSGL_API msgl_status msgl_store_kv(const msgl_kv_pool *pool, const void *k, const void *v,
                          const int32_t *out_loc, int32_t n_tokens, uint32_t *status,
                          msgl_stream_t stream);

/*
 * Extend (chunked prefill) step: request b has prefix_lens[b] tokens already
 * cached in its pages (a radix-cache hit or earlier chunks) and ext_lens[b]
 * new tokens whose K/V have already been stored in the pool by
 * msgl_store_kv.  Chunk row i of request b sits at absolute position
 * prefix_lens[b] + i and attends keys 0..prefix_lens[b]+i
 * ("Mini-SGLang 实战指南", §6.1 "Chunked Prefill", §6.5 "Radix Cache";
 * "不懂SGLang？从miniSGLang开始", §1.3).
 *
 *   q            device bf16 [total_tokens, num_q_heads, head_dim],
 *                request-major: request b owns rows cu_ext[b]..cu_ext[b+1]-1
 *   prefix_lens, ext_lens   device int32 [num_reqs]
 *   cu_ext       device int32 [num_reqs+1], cu_ext[0] = 0, prefix sums of ext_lens
 *   positions    device int32 [total_tokens] or NULL; when given, each row's
 *                entry must equal prefix_lens[b] + i (checked, else
 *                MSGL_DEVERR_POSITION; the mask always comes from the lengths)
 *   max_ext_len, max_seq_len   host upper bounds of ext_lens[b] and
 *                prefix_lens[b]+ext_lens[b]; they size the grid (a value
 *                that is too small is a device length error, never a wild read)
 *   scale        softmax scale (> 0, finite), normally 1/sqrt(head_dim)
 *   o            device bf16 [total_tokens, num_q_heads, head_dim] (output)
 *   lse          device fp32 [total_tokens, num_q_heads] (output), natural log
 *   workspace    device scratch of msgl_extend_workspace_size() bytes (may be
 *                NULL when that size is 0)
 */
MSGL_API size_t msgl_extend_workspace_size(int32_t num_reqs, int32_t total_tokens, int32_t num_q_heads,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t max_seq_len);

MSGL_API msgl_status msgl_attn_extend(const msgl_kv_pool *pool, const msgl_page_table *pages,
                             const void *q, int32_t num_q_heads, const int32_t *prefix_lens,
                             const int32_t *ext_lens, const int32_t *cu_ext,
                             const int32_t *positions, int32_t num_reqs, int32_t total_tokens,
                             int32_t max_ext_len, int32_t max_seq_len, float scale, void *o,
                             float *lse, void *workspace, size_t workspace_bytes,
                             uint32_t *status, msgl_stream_t stream);

/*
 * Decode step: one query row per request at position seq_lens[b]-1; it
 * attends all seq_lens[b] keys, the current token's included (stored by
 * msgl_store_kv first) ("Mini-SGLang 实战指南", §6.3 and §6.4: the decode
 * kernel is separate from prefill and is replayed under CUDA graphs, so the
 * grid depends only on the host scalars num_reqs and max_seq_len).
 * The keys are split into chunks processed in parallel, and the partial
 * results are merged by their log-sum-exp in a second kernel.
 *
 *   q          device bf16 [num_reqs, num_q_heads, head_dim]
 *   seq_lens   device int32 [num_reqs], each >= 1 and <= max_seq_len
 *   o, lse     device bf16 [num_reqs, num_q_heads, head_dim], fp32 [num_reqs, num_q_heads]
 *   workspace  device scratch of at least msgl_decode_workspace_size() bytes,
 *              256-byte aligned; it holds the split partials (fp32) and is
 *              fully rewritten by every call
 */
MSGL_API size_t msgl_decode_workspace_size(int32_t num_reqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_seq_len);

MSGL_API msgl_status msgl_attn_decode(const msgl_kv_pool *pool, const msgl_page_table *pages,
                             const void *q, int32_t num_q_heads, const int32_t *seq_lens,
                             int32_t num_reqs, int32_t max_seq_len, float scale, void *o,
                             float *lse, void *workspace, size_t workspace_bytes,
                             uint32_t *status, msgl_stream_t stream);

/*
 * Decode with the current token appended in the same launch: msgl_store_kv of
 * each request's new K/V row followed by msgl_attn_decode, fused.  The K/V an
 * attention call reads is the pool's history plus the newly computed K/V
 * ("不懂SGLang？从miniSGLang开始", §1.3 item 1), and decode runs once per
 * forward for every running request ("Mini-SGLang 实战指南", §6.3, §6.4).
 *
 *   k_new, v_new  device bf16 [num_reqs, num_kv_heads, head_dim]: the K/V of
 *                 each request's current token (key seq_lens[b]-1)
 *   new_loc       device int32 [num_reqs]: its pool slot, which must be the
 *                 page-table slot of key seq_lens[b]-1 (else
 *                 MSGL_DEVERR_APPEND_SLOT; an out-of-range slot sets
 *                 MSGL_DEVERR_SLOT_RANGE and nothing is written)
 * Every other argument, the outputs, the workspace and the status bits are
 * those of msgl_attn_decode.  Key seq_lens[b]-1 is attended from k_new/v_new
 * directly (it is not read back from the pool), and the row is written to
 * the pool bit-exact during the same launch.
 */
MSGL_API msgl_status msgl_attn_decode_append(const msgl_kv_pool *pool, const msgl_page_table *pages,
                                    const void *q, int32_t num_q_heads, const void *k_new,
                                    const void *v_new, const int32_t *new_loc,
                                    const int32_t *seq_lens, int32_t num_reqs, int32_t max_seq_len,
                                    float scale, void *o, float *lse, void *workspace,
                                    size_t workspace_bytes, uint32_t *status, msgl_stream_t stream);

/*
 * One batch of chunked-prefill rows or of decode rows, as the mixed step
 * below takes them.  Each field has the meaning, layout and ownership of
 * the msgl_attn_extend / msgl_attn_decode argument of the same name.  An
 * empty batch (num_reqs = 0) is allowed and launches nothing.
 */
typedef struct msgl_extend_batch {
    msgl_page_table pages;
    const void *q;                 /* device bf16 [total_tokens, num_q_heads, head_dim] */
    const int32_t *prefix_lens;    /* device int32 [num_reqs] */
    const int32_t *ext_lens;       /* device int32 [num_reqs] */
    const int32_t *cu_ext;         /* device int32 [num_reqs + 1] */
    const int32_t *positions;      /* device int32 [total_tokens] or NULL */
    int32_t num_reqs, total_tokens, max_ext_len, max_seq_len;
    void *o;                       /* device bf16 [total_tokens, num_q_heads, head_dim] (output) */
    float *lse;                    /* device fp32 [total_tokens, num_q_heads] (output) */
} msgl_extend_batch;

typedef struct msgl_decode_batch {
    msgl_page_table pages;
    const void *q;                 /* device bf16 [num_reqs, num_q_heads, head_dim] */
    const int32_t *seq_lens;       /* device int32 [num_reqs] */
    int32_t num_reqs, max_seq_len;
    void *o;                       /* device bf16 [num_reqs, num_q_heads, head_dim] (output) */
    float *lse;                    /* device fp32 [num_reqs, num_q_heads] (output) */
} msgl_decode_batch;

/*
 * Mixed step: the chunked-prefill batch and the decode batch of one forward
 * in a single call.  Under chunked prefill a forward carries prefill chunks
 * and decode rows together ("Mini-SGLang 实战指南", §6.1 "Chunked
 * Prefill"), and the engine works to keep the GPU from idling between the
 * pieces of a step (§6.6 "Overlap Scheduling").  The results are those of
 * msgl_attn_extend(ext) and msgl_attn_decode(dec) on the same inputs, bit
 * for bit; only the schedule differs.  The decode's key-range kernel runs
 * first; the extend is launched behind it with programmatic dependent
 * launch, so its CTAs take each SM as soon as that SM's decode range is
 * done instead of waiting for the slowest range; the decode's LSE merge
 * runs last.  Every launch shape depends on host scalars only, so the call
 * can be captured in a CUDA graph.
 *
 *   workspace   device scratch of at least
 *               msgl_decode_workspace_size(dec->num_reqs, ...) +
 *               msgl_extend_workspace_size(...) bytes, 256-byte aligned
 *               (NULL when that total is 0); fully rewritten by every call
 * Host validation and device status bits are those of the two calls.  On a
 * validation failure of either batch nothing is launched.
 */
MSGL_API msgl_status msgl_attn_mixed(const msgl_kv_pool *pool, const msgl_extend_batch *ext,
                                     const msgl_decode_batch *dec, int32_t num_q_heads, float scale,
                                     void *workspace, size_t workspace_bytes, uint32_t *status,
                                     msgl_stream_t stream);

/*
 * Decode for callers that cannot allocate device memory.  It has no
 * counterpart on the pages describing the engine: it is msgl_attn_decode
 * with its split scratch taken from a fixed array inside the library
 * instead of a caller workspace.  Meant for callers whose device memory is
 * all owned by a host pool planned up front, plugin-style interfaces that
 * receive only input and output pointers, and loops that cannot afford
 * cudaMalloc's implicit device synchronisation.
 *
 * Arguments, layouts, outputs and device status bits are those of
 * msgl_attn_decode, minus the workspace.  It allocates nothing: the scratch
 * is a static device array of MSGL_DECODE_NOALLOC_SCRATCH_BYTES that every
 * GPU loading the library holds until the process exits.  A call whose
 * msgl_decode_workspace_size() exceeds that size returns
 * MSGL_ERR_WORKSPACE (msgl_last_error() gives both sizes) without launching.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it.  Under
 * CUDA's lazy module loading that first call is also what loads the module
 * and places the 32 MiB on the device, an implicit allocation with its
 * possible synchronisation: make it once at start-up, before capturing any
 * stream and outside latency-critical loops.  The cached address assumes
 * one CUDA context per device for the life of the process; after a device
 * reset, or under a different driver-API context, use a fresh process.
 * All calls on a device share the array, which keeps the last call's
 * contents (no call relies on them); calls whose kernels overlap on the GPU
 * race on it, so order them.
 */
#define MSGL_DECODE_NOALLOC_SCRATCH_BYTES (32u << 20)

MSGL_API msgl_status msgl_attn_decode_noalloc(const msgl_kv_pool *pool, const msgl_page_table *pages,
                                     const void *q, int32_t num_q_heads, const int32_t *seq_lens,
                                     int32_t num_reqs, int32_t max_seq_len, float scale, void *o,
                                     float *lse, uint32_t *status, msgl_stream_t stream);

/*
 * Synchronises `stream`, reads the device status word into *flags (may be
 * NULL) and maps it to a status: MSGL_OK when it is zero, MSGL_ERR_TIMEOUT
 * when the timeout bit is set, else MSGL_ERR_OUT_OF_RANGE.  For tests and
 * debugging; not meant for the hot path.
 */
MSGL_API msgl_status msgl_read_status(const uint32_t *status, uint32_t *flags, msgl_stream_t stream);

/*
 * Self-test of the bounded wait every kernel uses (no counterpart on the
 * pages).  Launches one thread that waits on an mbarrier that nothing arrives
 * at, with a budget of budget_cycles SM clocks (0 < budget <= 4e9; ~1e7 is
 * about 5 ms).  The wait gives up, MSGL_DEVERR_TIMEOUT is ORed into *status,
 * and the kernel returns normally.  Use it to check that a lost arrival turns
 * into a status bit and the context stays usable.
 */
MSGL_API msgl_status msgl_selftest_wait_timeout(uint32_t *status, int64_t budget_cycles,
                                                msgl_stream_t stream);

/*
 * Host-side checks of one step's metadata, for tests and debugging.  They
 * read HOST copies of the arrays (copy the device arrays back first), launch
 * nothing, need no GPU and allocate nothing.  The kernels check the same
 * conditions on the device and report them through the status word; these
 * calls name the first offending entry in msgl_last_error().  Each returns
 * MSGL_OK, MSGL_ERR_INVALID_ARG (NULL array, bad scalar, inconsistent
 * lengths, wrong position, duplicate slot) or MSGL_ERR_OUT_OF_RANGE (a slot,
 * page index or page id outside the pool or the table).
 *
 * msgl_check_store_meta:  every out_loc[t] lies in [0, num_slots) and no
 *   slot is named twice (the store's result would depend on which row wins).
 * msgl_check_extend_meta:  prefix_lens[b] >= 0, ext_lens[b] >= 0,
 *   cu_ext[0] = 0, cu_ext[b+1] - cu_ext[b] = ext_lens[b], cu_ext[num_reqs] =
 *   total_tokens, ext_lens[b] <= max_ext_len, prefix_lens[b] + ext_lens[b]
 *   <= max_seq_len, positions[cu_ext[b] + i] = prefix_lens[b] + i (when
 *   positions is non-NULL), and every page that keys 0..prefix_lens[b] +
 *   ext_lens[b] - 1 fall on has an index below width and an id in
 *   [0, num_slots / page_size).
 * msgl_check_decode_meta:  1 <= seq_lens[b] <= max_seq_len and the pages of
 *   keys 0..seq_lens[b] - 1 are in range as above.
 *
 * page_ids is host int32 [num_reqs, stride]; only the first width entries of
 * a row are read.  The pages ("不懂SGLang？从miniSGLang开始", §1.3 item 3;
 * "Mini-SGLang 实战指南", §6.1, §6.2) define what the metadata means; these
 * checks have no counterpart there.
 */
MSGL_API msgl_status msgl_check_store_meta(int64_t num_slots, const int32_t *out_loc, int32_t n_tokens);

MSGL_API msgl_status msgl_check_extend_meta(int64_t num_slots, int32_t page_size, const int32_t *page_ids,
                                            int32_t stride, int32_t width, const int32_t *prefix_lens,
                                            const int32_t *ext_lens, const int32_t *cu_ext,
                                            const int32_t *positions, int32_t num_reqs, int32_t total_tokens,
                                            int32_t max_ext_len, int32_t max_seq_len);

MSGL_API msgl_status msgl_check_decode_meta(int64_t num_slots, int32_t page_size, const int32_t *page_ids,
                                            int32_t stride, int32_t width, const int32_t *seq_lens,
                                            int32_t num_reqs, int32_t max_seq_len);

/* Static description of a status code. */
MSGL_API const char *msgl_status_string(msgl_status s);

/* Thread-local text of the last failure in this thread (empty if none). */
MSGL_API const char *msgl_last_error(void);

/* MSGL_ABI_VERSION of the built library. */
MSGL_API int32_t msgl_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MSGL_ATTN_H */
