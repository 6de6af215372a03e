// Decode step: one query row per request over all of its pages.
//
// "Mini-SGLang 实战指南", §6.3: decode has its own attention kernel, apart
// from prefill; §6.4: decode is replayed under CUDA graphs, so the launch
// shape depends only on host scalars and the device (never on seq_lens).
//
// Design (bandwidth-bound: every cached K/V byte is read exactly once)
// ---------------------------------------------------------------------
// * Balanced split-KV.  The keys of all requests, laid end to end, are cut
//   into P equal ranges (at least 32 keys each), one per persistent CTA
//   (P = resident CTAs on the GPU).  A CTA's range covers one or more request segments; each segment
//   yields a partial (o, lse) per q head.  Request b's partials sit in rows
//   b + i of the workspace, i over the CTAs whose ranges touch it, and the
//   merge kernel folds them together by their log-sum-exp.
// * One CTA handles a group of up to 8 kv heads (all of them for Hkv <= 8).
//   A producer warp resolves slots through the page table (range-checked)
//   and fills a ring of 16-key stages; stages are handed over with mbarriers
//   (full: bytes landed; empty: every consumer warp has read the stage).
//   - page_size >= 16 ("box" path): a 16-key tile aligned to 16 keys lies in
//     one page, so its K (and V) arrive as two 3D TMA boxes of 64 dims x 16
//     keys x the group's heads (128-byte swizzle, head-major rows).  Four
//     copies per stage: a TMA unit issues about one copy per 80 cycles, which
//     held per-key copies near 50 GB/s per SM.
//     In the append mode the tile holding the current token lands on a
//     separate barrier, and the producer writes that key's rows from
//     k_new / v_new over the loaded ones before handing the stage over.
//   - page_size < 16: each key's pool row (the group's heads, contiguous in
//     the slot-major pool) arrives in one cp.async.bulk for K and one for V,
//     at a pitch of row + 16 bytes so that ldmatrix over 8 consecutive keys is
//     free of bank conflicts; in the append mode the current token's copies
//     read k_new / v_new instead.
// * One consumer warp per kv head computes S^T = K Q^T with m16n8k16 MMAs
//   (M = 16 keys, N = the group's 8 q-head slots, K = 128 dims), keeps a
//   base-2 online softmax per q head, transposes P to the B operand with
//   movmatrix, and accumulates O^T = V^T P^T (M = 16 dims x 8 tiles).
//   Packing the q heads of a kv head into N means each KV byte feeds all G
//   q heads at once.
#include <limits.h>
#include <math.h>
#include <string.h>

#include "kernels.h"
#include "ptx.cuh"

namespace msgl {

namespace {

constexpr int kTileKeys = 16;
constexpr int kMaxStages = 8;
constexpr int kMaxDecodeCtas = 512;       // bound on P, used to size the workspace
constexpr int kMaxHeadGroup = 8;
constexpr int kSmemBudget = 220 * 1024;

enum TileFlags { kFirst = 1, kLast = 2, kBad = 4, kEnd = 8 };

struct TileMeta {
    int32_t b;        // request
    int32_t slot;     // partial row (b + CTA index)
    int32_t n;        // keys in this tile
    int32_t flags;
    uint32_t mask;    // bit k: key k was loaded
    int32_t pad[3];
};

struct DecodeKernelArgs {
    PoolView pool;
    PageView pages;
    const __nv_bfloat16 *q;
    const int32_t *seq_lens;
    int32_t num_reqs, hq, group, max_seq_len, hg, stages;
    int32_t slices;   // consumer warps per kv head: each takes 8 of its G q heads
    float scale_log2;
    float *part_o;
    float *part_lse;
    uint32_t *status;
    // append mode (all three non-NULL): key seq_b-1 comes from k_new/v_new[b] and is
    // written to the pool at new_loc[b]
    const __nv_bfloat16 *k_new, *v_new;
    const int32_t *new_loc;
};

__device__ __forceinline__ int seq_valid(const int32_t *seq_lens, int b, int max_seq) {
    const int s = __ldg(seq_lens + b);
    return (s >= 1 && s <= max_seq) ? s : 0;
}

__device__ __forceinline__ long long warp_incl_scan(long long v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// Keys per CTA range: an equal share, but at least two tiles, so that a small
// batch does not scatter into hundreds of tiny partials for the merge to fold.
constexpr long long kMinKeysPerCta = 2 * kTileKeys;
__host__ __device__ __forceinline__ long long keys_per_cta(long long total, long long ctas) {
    const long long share = (total + ctas - 1) / ctas;
    return share > kMinKeysPerCta ? share : kMinKeysPerCta;
}

// Bytes of one stage: K and V of 16 keys for hg heads.  Box stages hold four swizzled
// 64-dim halves (K0, K1, V0, V1) of hg x 16 rows of 128 bytes; per-key stages hold
// padded rows.
size_t stage_bytes(int hg, bool box) {
    return box ? (size_t)4 * hg * kTileKeys * 128 : (size_t)2 * kTileKeys * (hg * 256 + 16);
}

// + 1024: the box path aligns the stage ring to 1024 bytes (128-byte swizzle atoms)
size_t decode_smem_bytes(int hg, int stages, bool box) {
    return 1024 + stages * stage_bytes(hg, box) + stages * sizeof(TileMeta) + (2 * stages + 1) * sizeof(uint64_t) +
           16;
}

template <bool kBox>
__global__ void __launch_bounds__(32 * (kMaxHeadGroup + 1), 1)
    decode_split_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                        const DecodeKernelArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const int hg = a.hg;
    const int pitch = hg * 256 + 16;
    const int half_bytes = hg * kTileKeys * 128;   // box path: one 64-dim half of K or V
    const int sbytes = kBox ? 4 * half_bytes : 2 * kTileKeys * pitch;
    const int S = a.stages;
    TileMeta *meta = reinterpret_cast<TileMeta *>(smem + (size_t)S * sbytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(meta + S);
    uint64_t *empty = full + S;
    uint64_t *patch = empty + S;   // box path, append mode: the current token's tile lands here first
    volatile int *abort_flag = reinterpret_cast<volatile int *>(patch + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g0 = blockIdx.y * hg;   // first kv head of this CTA
    // let the merge kernel launch now; it waits for this grid before reading partials
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(ptx::smem_u32(full + s), 1);
            ptx::mbar_init(ptx::smem_u32(empty + s), hg * a.slices);
        }
        ptx::mbar_init(ptx::smem_u32(patch), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();

    const int n_consumers = hg * a.slices;
    if (warp == n_consumers) {
        // ------------------------------------------------------------ producer
        const int B = a.num_reqs;
        long long total = 0;
        for (int c = 0; c < B; c += 32) {
            const int s = (c + lane < B) ? seq_valid(a.seq_lens, c + lane, a.max_seq_len) : 0;
            total += s;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
        const long long P = gridDim.x;
        const long long per = keys_per_cta(total, P);
        const long long r0 = per * blockIdx.x;
        const long long r1 = min(total, r0 + per);
        int it = 0;
        uint32_t patch_uses = 0;
        bool patch_pending = false;
        bool aborted = false;
        const uint32_t row_bytes = (uint32_t)hg * 256;
        // every K/V byte is read once: evict-first keeps the stream from displacing other lines
        const uint64_t stream_policy = ptx::l2_evict_first_policy();
        const long long slot_elems = (long long)a.pool.hkv * kHeadDim;

        auto stage_wait_empty = [&](int stage, int round) -> bool {
            if (ptx::mbar_wait(ptx::smem_u32(empty + stage), (round & 1) ^ 1)) return true;
            if (lane == 0) { report(a.status, MSGL_DEVERR_TIMEOUT); *abort_flag = 1; }
            return false;
        };

        if (r0 < r1) {
            // locate the request holding key r0
            long long base = 0, start_b = 0;
            int b = -1;
            for (int c = 0; c < B && b < 0; c += 32) {
                const int s = (c + lane < B) ? seq_valid(a.seq_lens, c + lane, a.max_seq_len) : 0;
                const long long incl = warp_incl_scan(s, lane);
                const long long tot = __shfl_sync(0xffffffffu, incl, 31);
                if (r0 < base + tot) {
                    const unsigned m = __ballot_sync(0xffffffffu, base + incl > r0);
                    const int l = __ffs(m) - 1;
                    b = c + l;
                    start_b = base + __shfl_sync(0xffffffffu, incl - s, l);
                }
                base += tot;
            }
            long long pos = r0;
            while (b >= 0 && b < B && pos < r1 && !aborted) {
                const int sb = seq_valid(a.seq_lens, b, a.max_seq_len);
                const long long end_b = start_b + sb;
                if (end_b > pos) {
                    const int lo = (int)(pos - start_b);
                    const int hi = (int)(min(r1, end_b) - start_b);
                    // page id of key `key` of request b (-1 when the page index is past the
                    // table's width, which then reads as a bad page)
                    auto load_pid = [&](int key) -> int {
                        const int pidx = key >> a.pool.log2_ps;
                        return pidx < a.pages.width ? __ldg(a.pages.ids + (int64_t)b * a.pages.stride + pidx) : -1;
                    };
                    if constexpr (kBox) {
                        // 16-key tiles aligned to 16 keys (each inside one page); keys outside
                        // [lo, hi) are loaded with the tile and masked.  Lane 0 does the work,
                        // with the next tile's page id looked up one tile ahead.
                        const int tlo = lo & ~(kTileKeys - 1);
                        int pid_cur = lane == 0 ? load_pid(tlo) : -1;
                        for (int t0 = tlo; t0 < hi; t0 += kTileKeys) {
                            const int stage = it % S, round = it / S;
                            const int t1 = t0 + kTileKeys;
                            const int pid_next = (lane == 0 && t1 < hi) ? load_pid(t1) : -1;
                            if (*abort_flag || !stage_wait_empty(stage, round)) { aborted = true; break; }
                            if (lane == 0) {
                                const int klo = max(lo, t0) - t0, khi = min(hi, t1) - t0;
                                const uint32_t keys = ((1u << khi) - 1u) & ~((1u << klo) - 1u);
                                const bool ok = pid_cur >= 0 && pid_cur < a.pool.num_pages;
                                const uint32_t full_bar = ptx::smem_u32(full + stage);
                                TileMeta &md = meta[stage];
                                md.b = b;
                                md.slot = b + (int)blockIdx.x;
                                md.n = khi - klo;
                                md.flags = (t0 == tlo ? kFirst : 0) | (t1 >= hi ? kLast : 0) | (ok ? 0 : kBad);
                                md.mask = ok ? keys : 0u;
                                if (!ok) report(a.status, MSGL_DEVERR_PAGE_RANGE);
                                // append mode: the tile holding the current token lands on the
                                // patch barrier; its row is overwritten below before the stage
                                // is handed over
                                const bool patch_tile = a.new_loc != nullptr && hi == sb && sb - 1 < t1;
                                const uint32_t land_bar = patch_tile ? ptx::smem_u32(patch) : full_bar;
                                ptx::mbar_arrive_expect_tx(land_bar, ok ? (uint32_t)sbytes : 0u);
                                if (ok) {
                                    const int slot0 = (pid_cur << a.pool.log2_ps) + (t0 & ((1 << a.pool.log2_ps) - 1));
                                    const uint32_t dst = ptx::smem_u32(smem + (size_t)stage * sbytes);
                                    ptx::tma_load_3d_hint(dst, &k_map, 0, slot0, g0, land_bar, stream_policy);
                                    ptx::tma_load_3d_hint(dst + half_bytes, &k_map, 64, slot0, g0, land_bar, stream_policy);
                                    ptx::tma_load_3d_hint(dst + 2 * half_bytes, &v_map, 0, slot0, g0, land_bar, stream_policy);
                                    ptx::tma_load_3d_hint(dst + 3 * half_bytes, &v_map, 64, slot0, g0, land_bar, stream_policy);
                                }
                            }
                            // (only the CTA whose range ends at key sb - 1 handles it)
                            if (a.new_loc != nullptr && hi == sb && sb - 1 < t1) {
                                // current token (key sb - 1): its K/V come from k_new / v_new.  Wait for
                                // the tile, write the token's rows of every head over the loaded ones
                                // (swizzled positions), store them into the pool at new_loc[b], then
                                // release the stage.
                                const bool page_ok = __shfl_sync(0xffffffffu, pid_cur, 0) >= 0 &&
                                                     __shfl_sync(0xffffffffu, pid_cur, 0) < a.pool.num_pages;
                                if (!ptx::mbar_wait(ptx::smem_u32(patch), patch_uses & 1)) {
                                    if (lane == 0) { report(a.status, MSGL_DEVERR_TIMEOUT); *abort_flag = 1; }
                                    patch_pending = true;
                                    aborted = true;
                                    break;
                                }
                                ++patch_uses;
                                const int kl = sb - 1 - t0;
                                const long long src = (long long)b * slot_elems + (long long)g0 * kHeadDim;
                                uint8_t *stage_p = smem + (size_t)stage * sbytes;
                                for (int x = lane; x < hg * 16; x += 32) {
                                    // x = (head, 16-byte chunk of the 128 dims)
                                    const int h = x >> 4, c16 = x & 15;
                                    const int hf = c16 >> 3, c = c16 & 7;
                                    const uint32_t off = (uint32_t)(hf * half_bytes + (h * kTileKeys + kl) * 128 +
                                                                    ((c ^ (kl & 7)) << 4));
                                    const uint4 kv = ld_stream_16(a.k_new + src + h * kHeadDim + 8 * c16);
                                    const uint4 vv = ld_stream_16(a.v_new + src + h * kHeadDim + 8 * c16);
                                    *reinterpret_cast<uint4 *>(stage_p + off) = kv;
                                    *reinterpret_cast<uint4 *>(stage_p + 2 * half_bytes + off) = vv;
                                }
                                const long long loc = __ldg(a.new_loc + b);
                                const long long page_slot =
                                    page_ok ? ((long long)__shfl_sync(0xffffffffu, pid_cur, 0) << a.pool.log2_ps) +
                                                  ((sb - 1) & ((1 << a.pool.log2_ps) - 1))
                                            : -1;
                                if (loc < 0 || loc >= a.pool.num_slots) {
                                    if (lane == 0) report(a.status, MSGL_DEVERR_SLOT_RANGE);
                                } else {
                                    if (lane == 0 && loc != page_slot) report(a.status, MSGL_DEVERR_APPEND_SLOT);
                                    const long long dst = loc * slot_elems + (long long)g0 * kHeadDim;
                                    for (int c = lane; c < hg * kHeadDim / 8; c += 32) {
                                        const uint4 kv = ld_stream_16(a.k_new + src + 8 * c);
                                        const uint4 vv = ld_stream_16(a.v_new + src + 8 * c);
                                        *reinterpret_cast<uint4 *>(const_cast<__nv_bfloat16 *>(a.pool.k) + dst + 8 * c) = kv;
                                        *reinterpret_cast<uint4 *>(const_cast<__nv_bfloat16 *>(a.pool.v) + dst + 8 * c) = vv;
                                    }
                                }
                                __syncwarp();
                                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(full + stage));
                            }
                            pid_cur = pid_next;
                            __syncwarp();
                            ++it;
                        }
                        pos = min(r1, end_b);
                        start_b = end_b;
                        ++b;
                        continue;
                    }
                    // the page ids of the next tile are loaded one tile ahead, so the table
                    // lookup overlaps the wait for a free stage
                    int pid_cur = lane < min(kTileKeys, hi - lo) ? load_pid(lo + lane) : -1;
                    for (int t0 = lo; t0 < hi; t0 += kTileKeys) {
                        const int stage = it % S, round = it / S;
                        const int n = min(kTileKeys, hi - t0);
                        const int t1 = t0 + kTileKeys;
                        const int pid_next = (t1 < hi && lane < min(kTileKeys, hi - t1)) ? load_pid(t1 + lane) : -1;
                        if (*abort_flag || !stage_wait_empty(stage, round)) { aborted = true; break; }
                        bool ok = false;
                        int64_t slot = -1;
                        if (lane < n && pid_cur >= 0 && pid_cur < a.pool.num_pages) {
                            slot = ((int64_t)pid_cur << a.pool.log2_ps) + ((t0 + lane) & ((1 << a.pool.log2_ps) - 1));
                            ok = true;
                        }
                        pid_cur = pid_next;
                        const uint32_t mask = __ballot_sync(0xffffffffu, ok);
                        const uint32_t badm = __ballot_sync(0xffffffffu, lane < n && !ok);
                        const uint32_t full_bar = ptx::smem_u32(full + stage);
                        if (lane == 0) {
                            TileMeta &md = meta[stage];
                            md.b = b;
                            md.slot = b + (int)blockIdx.x;
                            md.n = n;
                            md.flags = (t0 == lo ? kFirst : 0) | (t0 + kTileKeys >= hi ? kLast : 0) |
                                       (badm ? kBad : 0);
                            md.mask = mask;
                            if (badm) report(a.status, MSGL_DEVERR_PAGE_RANGE);
                            ptx::mbar_arrive_expect_tx(full_bar, __popc(mask) * row_bytes * 2);
                        }
                        __syncwarp();
                        // append mode: this tile holds the request's current token
                        const bool has_new = a.new_loc && t0 + n == sb;
                        const bool is_new = has_new && lane == n - 1;
                        if (ok) {
                            uint8_t *kdst = smem + (size_t)stage * sbytes + lane * pitch;
                            uint8_t *vdst = kdst + kTileKeys * pitch;
                            const long long off = slot * slot_elems + (long long)g0 * kHeadDim;
                            const long long noff = (long long)b * slot_elems + (long long)g0 * kHeadDim;
                            ptx::bulk_g2s_hint(ptx::smem_u32(kdst), is_new ? a.k_new + noff : a.pool.k + off,
                                               row_bytes, full_bar, stream_policy);
                            ptx::bulk_g2s_hint(ptx::smem_u32(vdst), is_new ? a.v_new + noff : a.pool.v + off,
                                               row_bytes, full_bar, stream_policy);
                        }
                        if (has_new) {
                            // write the new K/V rows of this head group into the pool at new_loc[b];
                            // only this CTA touches key seq_b-1 in this launch
                            const long long loc = __ldg(a.new_loc + b);
                            const long long page_slot = __shfl_sync(0xffffffffu, slot, n - 1);
                            if (loc < 0 || loc >= a.pool.num_slots) {
                                if (lane == 0) report(a.status, MSGL_DEVERR_SLOT_RANGE);
                            } else {
                                if (lane == 0 && loc != page_slot) report(a.status, MSGL_DEVERR_APPEND_SLOT);
                                const long long src = (long long)b * slot_elems + (long long)g0 * kHeadDim;
                                const long long dst = loc * slot_elems + (long long)g0 * kHeadDim;
                                for (int c = lane; c < (int)row_bytes / 16; c += 32) {
                                    const uint4 kv = ld_stream_16(a.k_new + src + 8 * c);
                                    const uint4 vv = ld_stream_16(a.v_new + src + 8 * c);
                                    *reinterpret_cast<uint4 *>(const_cast<__nv_bfloat16 *>(a.pool.k) + dst + 8 * c) = kv;
                                    *reinterpret_cast<uint4 *>(const_cast<__nv_bfloat16 *>(a.pool.v) + dst + 8 * c) = vv;
                                }
                            }
                        }
                        ++it;
                    }
                    pos = min(r1, end_b);
                }
                start_b = end_b;
                ++b;
            }
        }
        // end marker: an empty stage the consumers stop at
        if (!aborted) {
            const int stage = it % S, round = it / S;
            if (!*abort_flag && stage_wait_empty(stage, round)) {
                if (lane == 0) {
                    meta[stage].flags = kEnd;
                    ptx::mbar_arrive(ptx::smem_u32(full + stage));
                }
                ++it;
            } else {
                aborted = true;
            }
        }
        if (aborted) {
            // let every copy already issued land before the CTA exits (bounded)
            const int first = it > S ? it - S : 0;
            for (int k = first; k < it; ++k)
                ptx::mbar_wait(ptx::smem_u32(full + (k % S)), (k / S) & 1, 200000000LL);
            if (patch_pending) ptx::mbar_wait(ptx::smem_u32(patch), patch_uses & 1, 200000000LL);
        }
    } else if (warp < n_consumers) {
        // ----------------------------------------------------------- consumers
        const int kvh = warp / a.slices;         // this warp's kv head within the group
        const int g = g0 + kvh;
        const int hoff = (warp - kvh * a.slices) * 8;   // its 8 q heads start at g * G + hoff
        const int G = a.group;
        const int Gs = G - hoff;                 // q heads from hoff on (slots >= Gs are empty)
        const int qh = lane >> 2;                // q-head slot this lane loads for Q^T
        const int h0 = 2 * (lane & 3), h1 = h0 + 1;
        const int k0 = lane >> 2, k1 = k0 + 8;   // keys of this lane's S^T elements
        const int kv0 = 2 * (lane & 3), kv1 = kv0 + 8;  // keys of this lane's V^T fragment
        uint32_t qf[8][2];
        float acc[8][4];
        float m2[2], l[2];
        bool seg_bad = false;
        const uint32_t tiles = ptx::smem_u32(smem);
        // ldmatrix row addresses (per lane) inside a stage
        const int krow = (lane & 7) + 8 * ((lane >> 3) & 1);
        const int kcol = 8 * (lane >> 4);
        const int vrow = (lane & 7) + 8 * (lane >> 4);
        const int vcol = 8 * ((lane >> 3) & 1);
        const uint32_t k_lane = (uint32_t)(krow * pitch + kvh * 256 + kcol * 2);
        const uint32_t v_lane = (uint32_t)(kTileKeys * pitch + vrow * pitch + kvh * 256 + vcol * 2);
        // Box path: row (head w, key k) of a 64-dim half sits at (16 w + k) * 128 bytes, its
        // 16-byte chunk c at position c ^ (k & 7) (k & 7 = lane & 7 for every ldmatrix row
        // this lane addresses).  Offset of dims [d, d + 8) of this lane's K / V row:
        auto box_off = [&](int row, int d) -> uint32_t {
            return (uint32_t)((d >> 6) * half_bytes + (kvh * kTileKeys + row) * 128 +
                              ((((d & 63) >> 3) ^ (lane & 7)) << 4));
        };

        for (int it = 0;; ++it) {
            const int stage = it % S, round = it / S;
            if (*abort_flag) break;
            if (!ptx::mbar_wait(ptx::smem_u32(full + stage), round & 1)) {
                if (lane == 0) { report(a.status, MSGL_DEVERR_TIMEOUT); *abort_flag = 1; }
                break;
            }
            const int flags = meta[stage].flags;
            if (flags & kEnd) break;
            const int b = meta[stage].b;
            const int pslot = meta[stage].slot;
            const uint32_t mask = meta[stage].mask;

            if (flags & kFirst) {
                const __nv_bfloat16 *qp = a.q + ((long long)b * a.hq + (long long)g * G + hoff + qh) * kHeadDim;
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    if (qh < Gs) {
                        qf[ks][0] = *reinterpret_cast<const uint32_t *>(qp + 16 * ks + 2 * (lane & 3));
                        qf[ks][1] = *reinterpret_cast<const uint32_t *>(qp + 16 * ks + 8 + 2 * (lane & 3));
                    } else {
                        qf[ks][0] = qf[ks][1] = 0u;
                    }
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
                m2[0] = m2[1] = -INFINITY;
                l[0] = l[1] = 0.f;
                seg_bad = false;
            }
            seg_bad |= (flags & kBad) != 0;

            const uint32_t base = tiles + (uint32_t)(stage * sbytes);
            // Read the whole stage (K and V fragments) into registers, then hand it back:
            // the producer's next copies into this stage overlap the math below.  The
            // arrival's address depends on the loaded registers, so it cannot pass them.
            uint32_t kf[8][4], vf[8][4];
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t addr = kBox ? base + box_off(krow, 16 * ks + kcol) : base + k_lane + ks * 32;
                ptx::ldsm_x4(addr, kf[ks][0], kf[ks][1], kf[ks][2], kf[ks][3]);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t addr =
                    kBox ? base + 2 * half_bytes + box_off(vrow, 16 * i + vcol) : base + v_lane + i * 32;
                ptx::ldsm_x4_t(addr, vf[i][0], vf[i][1], vf[i][2], vf[i][3]);
            }
            {
                uint32_t any = 0u;
#pragma unroll
                for (int i = 0; i < 8; ++i) any |= kf[i][0] | vf[i][0];
                uint32_t zero;
                asm volatile("and.b32 %0, %1, 0;" : "=r"(zero) : "r"(any));
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(empty + stage) + zero);
            }
            // S^T (16 keys x 8 q-head slots) = K (16 x 128) * Q^T (128 x 8), two accumulation chains
            float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < 8; ks += 2) {
                ptx::mma_bf16_16816(s, kf[ks], qf[ks][0], qf[ks][1]);
                ptx::mma_bf16_16816(s2, kf[ks + 1], qf[ks + 1][0], qf[ks + 1][1]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) s[i] += s2[i];
            const bool v0 = (mask >> k0) & 1u, v1 = (mask >> k1) & 1u;
            const float x00 = v0 ? s[0] * a.scale_log2 : -INFINITY;   // key k0, head h0
            const float x01 = v0 ? s[1] * a.scale_log2 : -INFINITY;   // key k0, head h1
            const float x10 = v1 ? s[2] * a.scale_log2 : -INFINITY;   // key k1, head h0
            const float x11 = v1 ? s[3] * a.scale_log2 : -INFINITY;   // key k1, head h1
            float mx0 = fmaxf(x00, x10), mx1 = fmaxf(x01, x11);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m2[0], mx0), mn1 = fmaxf(m2[1], mx1);
            const float al0 = (mn0 == -INFINITY) ? 1.f : ptx::ex2(m2[0] - mn0);
            const float al1 = (mn1 == -INFINITY) ? 1.f : ptx::ex2(m2[1] - mn1);
            const float p00 = (x00 == -INFINITY) ? 0.f : ptx::ex2(x00 - mn0);
            const float p01 = (x01 == -INFINITY) ? 0.f : ptx::ex2(x01 - mn1);
            const float p10 = (x10 == -INFINITY) ? 0.f : ptx::ex2(x10 - mn0);
            const float p11 = (x11 == -INFINITY) ? 0.f : ptx::ex2(x11 - mn1);
            m2[0] = mn0;
            m2[1] = mn1;
            l[0] = l[0] * al0 + p00 + p10;
            l[1] = l[1] * al1 + p01 + p11;
            const uint32_t pb0 = ptx::movmatrix_t(ptx::pack_bf16(p00, p01));   // keys 0-7
            const uint32_t pb1 = ptx::movmatrix_t(ptx::pack_bf16(p10, p11));   // keys 8-15
            // zero V^T fragment entries of keys that were not loaded
            const uint32_t ma = ((mask >> kv0) & 1u ? 0x0000ffffu : 0u) | ((mask >> (kv0 + 1)) & 1u ? 0xffff0000u : 0u);
            const uint32_t mb = ((mask >> kv1) & 1u ? 0x0000ffffu : 0u) | ((mask >> (kv1 + 1)) & 1u ? 0xffff0000u : 0u);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                vf[i][0] &= ma;
                vf[i][1] &= ma;
                vf[i][2] &= mb;
                vf[i][3] &= mb;
                acc[i][0] *= al0;
                acc[i][1] *= al1;
                acc[i][2] *= al0;
                acc[i][3] *= al1;
                ptx::mma_bf16_16816(acc[i], vf[i], pb0, pb1);
            }

            if (flags & kLast) {
                float lt0 = l[0], lt1 = l[1];
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
                    lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
                }
                const float inv0 = lt0 > 0.f ? 1.f / lt0 : 0.f;
                const float inv1 = lt1 > 0.f ? 1.f / lt1 : 0.f;
                const long long hb = (long long)pslot * a.hq + (long long)g * G + hoff;
                float *po = a.part_o + hb * kHeadDim;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int d0 = 16 * i + (lane >> 2), d1 = d0 + 8;
                    if (h0 < Gs) {
                        po[h0 * kHeadDim + d0] = acc[i][0] * inv0;
                        po[h0 * kHeadDim + d1] = acc[i][2] * inv0;
                    }
                    if (h1 < Gs) {
                        po[h1 * kHeadDim + d0] = acc[i][1] * inv1;
                        po[h1 * kHeadDim + d1] = acc[i][3] * inv1;
                    }
                }
                if (lane < 4) {
                    const float nan = __int_as_float(0x7fc00000);
                    if (h0 < Gs)
                        a.part_lse[hb + h0] = (seg_bad || !(lt0 > 0.f)) ? nan : (m2[0] + log2f(lt0)) * kLn2;
                    if (h1 < Gs)
                        a.part_lse[hb + h1] = (seg_bad || !(lt1 > 0.f)) ? nan : (m2[1] + log2f(lt1)) * kLn2;
                }
            }
        }
    }
    __syncthreads();
}

// Fold the partials of request b, q head h: weights exp(lse_i - max),
// o = sum w_i o_i / sum w_i, lse = max + ln(sum w_i).  A NaN partial lse
// marks a segment that hit a bad index: the row is written as o = 0, lse = -inf.
// One warp per (request, q head).  The lanes first share out the partials (max,
// weights and their sum by warp reductions, weights kept in shared memory), then
// each lane owns 4 of the 128 dims and sums the weighted partial rows, four
// partials at a time so their loads overlap.
constexpr int kMergeMaxParts = kMaxDecodeCtas + 1;

__global__ void __launch_bounds__(256) decode_merge_kernel(
    const int32_t *__restrict__ seq_lens, int32_t num_reqs, int32_t max_seq_len, int32_t hq,
    int32_t num_ctas, const float *__restrict__ part_o, const float *__restrict__ part_lse,
    __nv_bfloat16 *__restrict__ o, float *__restrict__ lse, uint32_t *status) {
    __shared__ long long s_start, s_total;
    __shared__ float s_w[8][kMergeMaxParts];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    if (warp == 0) {
        long long total = 0, before = 0;
        for (int c = 0; c < num_reqs; c += 32) {
            const int idx = c + lane;
            const int s = idx < num_reqs ? seq_valid(seq_lens, idx, max_seq_len) : 0;
            total += s;
            if (idx < b) before += s;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            total += __shfl_xor_sync(0xffffffffu, total, off);
            before += __shfl_xor_sync(0xffffffffu, before, off);
        }
        if (lane == 0) { s_total = total; s_start = before; }
    }
    __syncthreads();
    const int h = blockIdx.x * 8 + warp;
    if (h >= hq) return;
    const int sb = seq_valid(seq_lens, b, max_seq_len);
    const long long row = (long long)b * hq + h;
    __nv_bfloat16 *orow = o + row * kHeadDim + lane * 4;
    if (sb == 0) {
        if (blockIdx.x == 0 && warp == 0 && lane == 0) report(status, MSGL_DEVERR_LENGTH);
        *reinterpret_cast<uint2 *>(orow) = make_uint2(0u, 0u);
        if (lane == 0) lse[row] = -INFINITY;
        return;
    }
    // the split kernel's partials are complete and visible after this point
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const long long per = keys_per_cta(s_total, num_ctas);
    const int first = (int)(s_start / per);
    const int count = (int)((s_start + sb - 1) / per) - first + 1;   // <= num_ctas
    if (count <= 4) {
        // few partials (the usual case): every lane loads all partial LSEs and its four dims
        // of every partial row at once, so the fold costs one memory round trip
        const float *lp = part_lse + (long long)(b + first) * hq + h;
        const float *op = part_o + ((long long)(b + first) * hq + h) * kHeadDim + lane * 4;
        const long long stride = (long long)hq * kHeadDim;
        float x[4];
        float4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[i] = i < count ? lp[(long long)i * hq] : -INFINITY;
            v[i] = i < count ? *reinterpret_cast<const float4 *>(op + i * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        bool bad = false;
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            bad |= isnan(x[i]);
            M = fmaxf(M, x[i]);
        }
        float L = 0.f, acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
        if (!bad && M != -INFINITY) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float w = x[i] == -INFINITY ? 0.f : __expf(x[i] - M);
                L += w;
                acc0 += w * v[i].x;
                acc1 += w * v[i].y;
                acc2 += w * v[i].z;
                acc3 += w * v[i].w;
            }
        }
        const bool zero = bad || !(L > 0.f);
        const float inv = zero ? 0.f : 1.f / L;
        *reinterpret_cast<uint2 *>(orow) =
            make_uint2(ptx::pack_bf16(acc0 * inv, acc1 * inv), ptx::pack_bf16(acc2 * inv, acc3 * inv));
        if (lane == 0) lse[row] = zero ? -INFINITY : M + logf(L);
        return;
    }
    // max over the partial LSEs (NaN = failed segment)
    float M = -INFINITY;
    bool failed = false;
    for (int i = lane; i < count; i += 32) {
        const float x = part_lse[(long long)(b + first + i) * hq + h];
        if (isnan(x)) failed = true;
        else M = fmaxf(M, x);
    }
    failed = __any_sync(0xffffffffu, failed);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float L = 0.f;
    if (!failed && M != -INFINITY) {
        for (int i = lane; i < count; i += 32) {
            const float x = part_lse[(long long)(b + first + i) * hq + h];
            const float w = x == -INFINITY ? 0.f : __expf(x - M);
            s_w[warp][i] = w;
            L += w;
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
    }
    __syncwarp();
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const bool zero = failed || !(L > 0.f);
    if (!zero) {
        const float *base = part_o + ((long long)(b + first) * hq + h) * kHeadDim + lane * 4;
        const long long stride = (long long)hq * kHeadDim;
        int i = 0;
        for (; i + 4 <= count; i += 4) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const float4 *>(base + (i + u) * stride);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float w = s_w[warp][i + u];
                acc[0] += w * v[u].x;
                acc[1] += w * v[u].y;
                acc[2] += w * v[u].z;
                acc[3] += w * v[u].w;
            }
        }
        for (; i < count; ++i) {
            const float4 v = *reinterpret_cast<const float4 *>(base + i * stride);
            const float w = s_w[warp][i];
            acc[0] += w * v.x;
            acc[1] += w * v.y;
            acc[2] += w * v.z;
            acc[3] += w * v.w;
        }
    }
    const float inv = zero ? 0.f : 1.f / L;
    const uint32_t lo = ptx::pack_bf16(acc[0] * inv, acc[1] * inv);
    const uint32_t hi = ptx::pack_bf16(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2 *>(orow) = make_uint2(lo, hi);
    if (lane == 0) lse[row] = zero ? -INFINITY : M + logf(L);
}

struct Launch {
    int hg, stages, ctas;
    size_t smem;
};

// Consumer warps per kv head: each covers 8 of its G q heads (the N = 8 MMA slots).
int decode_slices(int group) { return (group + 7) / 8; }

// kv heads per CTA: the largest divisor of hkv whose consumer warps (hg x slices) fit in 8.
int decode_head_group(int hkv, int slices) {
    int hg = kMaxHeadGroup / slices;
    if (hg < 1) hg = 1;
    while (hkv % hg) --hg;
    return hg;
}

Launch decode_launch_shape(int hkv, int slices, bool box) {
    Launch L;
    L.hg = decode_head_group(hkv, slices);
    int st = (int)((kSmemBudget - 1024 - 64) / (stage_bytes(L.hg, box) + sizeof(TileMeta) + 16));
    L.stages = st < 2 ? 2 : (st > kMaxStages ? kMaxStages : st);
    L.smem = decode_smem_bytes(L.hg, L.stages, box);
    const int sms = sm_count();
    const int groups = hkv / L.hg;
    int ctas = sms / groups;
    if (ctas < 1) ctas = 1;
    L.ctas = ctas > kMaxDecodeCtas ? kMaxDecodeCtas : ctas;
    return L;
}

}  // namespace

DecodePlan plan_decode(int32_t num_reqs, int32_t hq, int32_t hkv, int32_t max_seq_len) {
    (void)max_seq_len;
    (void)hkv;
    DecodePlan p;
    const size_t rows = (size_t)num_reqs + kMaxDecodeCtas;
    p.o_bytes = (rows * hq * kHeadDim * sizeof(float) + 255) / 256 * 256;
    const size_t l_bytes = (rows * hq * sizeof(float) + 255) / 256 * 256;
    p.workspace = p.o_bytes + l_bytes;
    return p;
}

cudaError_t launch_decode(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream, DecodePhase phase) {
    if (a.num_reqs == 0) return cudaSuccess;
    const int hkv = a.pool.hkv;
    const int slices = decode_slices(a.hq / hkv);
    if (slices > kMaxHeadGroup) return cudaErrorInvalidValue;   // G > 64
    // Box path: whole 16-key tiles by 3D TMA (page_size >= 16, not the append mode).  Its
    // tensor maps view each pool as [kv head][slot][128 dims] (innermost last), so a box
    // lands head-major: 16 consecutive keys of one head form 16 consecutive smem rows.
    const int hg = decode_head_group(hkv, slices);
    bool box = (1 << a.pool.log2_ps) >= kTileKeys && a.pool.num_slots < INT_MAX;
    CUtensorMap km, vm;
    memset(&km, 0, sizeof km);
    memset(&vm, 0, sizeof vm);
    if (box) {
        PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
        if (!enc) return cudaErrorNotSupported;
        for (int which = 0; which < 2; ++which) {
            cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)a.pool.num_slots, (cuuint64_t)hkv};
            cuuint64_t strides[2] = {(cuuint64_t)hkv * kHeadDim * 2, (cuuint64_t)kHeadDim * 2};
            cuuint32_t boxd[3] = {64, (cuuint32_t)kTileKeys, (cuuint32_t)hg};
            cuuint32_t es[3] = {1, 1, 1};
            if (enc(which ? &vm : &km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<__nv_bfloat16 *>(which ? a.pool.v : a.pool.k), dims, strides, boxd, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        }
    }
    const Launch L = decode_launch_shape(hkv, slices, box);
    static bool attr_set[64];   // per device; idempotent, racing setters write the same value
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<false>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_split_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kSmemBudget);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    DecodeKernelArgs k{};
    k.pool = a.pool;
    k.pages = a.pages;
    k.q = a.q;
    k.seq_lens = a.seq_lens;
    k.num_reqs = a.num_reqs;
    k.hq = a.hq;
    k.group = a.hq / hkv;
    k.max_seq_len = a.max_seq_len;
    k.hg = L.hg;
    k.slices = slices;
    k.stages = L.stages;
    k.scale_log2 = a.scale * kLog2e;
    k.part_o = a.part_o;
    k.part_lse = a.part_lse;
    k.status = a.status;
    k.k_new = a.k_new;
    k.v_new = a.v_new;
    k.new_loc = a.new_loc;
    (void)plan;
    if (L.smem > (size_t)kSmemBudget) return cudaErrorInvalidValue;
    if (phase != DecodePhase::kMerge) {
        dim3 grid(L.ctas, hkv / L.hg);
        if (box)
            decode_split_kernel<true><<<grid, 32 * (L.hg * slices + 1), L.smem, stream>>>(km, vm, k);
        else
            decode_split_kernel<false><<<grid, 32 * (L.hg * slices + 1), L.smem, stream>>>(km, vm, k);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess || phase == DecodePhase::kSplit) return e;
    }
    // programmatic dependent launch: the merge's launch and its seq_lens scan overlap the
    // tail of the kernel before it (the split, or the extend of a mixed step)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.hq + 7) / 8, a.num_reqs);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel, a.seq_lens, a.num_reqs, a.max_seq_len, a.hq,
                              L.ctas, (const float *)a.part_o, (const float *)a.part_lse, a.o, a.lse,
                              a.status);
}

}  // namespace msgl
