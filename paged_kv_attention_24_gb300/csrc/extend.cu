// Extend (chunked prefill) step on the 5th-generation tensor cores.
//
// Chunk row i of request b attends keys 0..prefix_b + i of the request's
// pages: the cached (radix-shared) prefix plus its own causal part
// ("Mini-SGLang 实战指南", §6.1 "Chunked Prefill" and §6.5 "Radix Cache";
// "不懂SGLang？从miniSGLang开始", §1.3: K/V come from the pool, located
// through the page table).
//
// Design
// ------
// * GQA packing: a 128-row Q tile holds R = floor(128 / G) consecutive
//   tokens x the G q heads of one kv head (row r = token r / G, head r % G),
//   loaded by one 3D TMA box per 64-dim half straight from q[T, Hq, 128].
//   Every K/V byte staged in shared memory feeds all G heads.
// * A CTA owns two such tiles (2R tokens) of one request and one kv head and
//   streams 128-key K and V tiles through 2-stage (K) and 3-stage (V) rings.
//   At page_size >= 16 a page that is a contiguous, fully valid run of pool
//   rows arrives in tiled TMA boxes (K: one per 64-dim half; V: both halves
//   of 16 or 32 keys per box, into V's 16-key block layout), and any other
//   keys are gathered four pool rows per copy (TMA gather4).  Below 16 every
//   key is its own run, and 16-byte cp.async copies replace the gathers (a
//   TMA instruction per four 128-byte rows cannot keep up).  A key beyond the
//   causal range, or behind a bad page id, reads as zeros.
// * tcgen05.mma (M = N = 128, K = 16 per instruction, bf16 in, fp32 out):
//   S_t = Q_t K^T lands in TMEM (columns 0-127 for tile 0, 128-255 for tile
//   1); O_t accumulates in columns 256-383 / 384-511 (the whole 512-column
//   TMEM of the SM).  P is written back over S_t as packed bf16 and fed to
//   O_t += P_t V from TMEM, with V as an MN-major shared-memory operand.
// * Warp roles: warp 0 loads Q and K, warp 3 loads V (warp 2 shares the K
//   tiles on the cp.async path), one thread of warp 1 issues the MMAs,
//   warps 4-7 and 8-11 run the online softmax of tile 0 and tile 1 (one
//   TMEM lane = one row per thread).  While one warpgroup exponentiates,
//   the tensor core works on the other tile.  O is rescaled lazily: only
//   when a row's running max grows by more than 2^8 (so P stays <= 256);
//   after the first K/V tile the row max is taken only when a row sum
//   shows that some score may have grown that much.
// * The issuing thread runs at the tensor pipe's pace and shares its SM
//   sub-partition with two softmax warps, so every instruction it executes
//   between MMA groups idles the pipe: it tests the next group's barrier
//   while the current group is queued, releases no K/V stage itself (the
//   last tile's softmax warp does, on seeing S complete), commits O only
//   after a tile's last PV, and runs a steady-state loop without per-tile
//   conditions.
// * Every mbarrier wait is bounded; a timeout sets MSGL_DEVERR_TIMEOUT and
//   the CTA winds down after its copies and MMAs have landed.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <limits.h>
#include <math.h>
#include <string.h>

#include "kernels.h"
#include "ptx.cuh"

namespace msgl {

namespace {

constexpr int kRows = 128;                 // rows per Q tile (MMA M)
constexpr int kKeys = 128;                 // keys per K/V tile (MMA N of S, K of PV)
constexpr int kStages = 2;                 // K tiles in flight
constexpr int kVStages = 3;                // V tiles in flight (V is needed later than K)
constexpr int kThreads = 384;              // 12 warps
constexpr uint32_t kHalf = 16384;          // 128 rows x 128 bytes (64 bf16)
constexpr uint32_t kTile = 2 * kHalf;      // 128 x 128 bf16
// With tiled page copies (page size >= 16), V tiles are stored as 8 blocks of 16 keys,
// each block [half][16 keys][128 B], so that one copy brings both 64-dim halves of up to
// 32 keys and every PV MMA (16 keys) reads one block, its halves kVHalf bytes apart.  At
// 16 keys per page the copy engine's per-copy cost bounds the loads, and this halves the
// V copies.  The 16-byte-copy path (smaller pages) lays V out as K.
constexpr uint32_t kVBlock = 4096, kVHalf = 2048;
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + 2 * kTile;
constexpr uint32_t kOffV = kOffK + kStages * kTile;
constexpr uint32_t kOffBar = kOffV + kVStages * kTile;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;   // + slack to align the base to 1024

// barrier slots
constexpr int kQFull = 0, kKFull = 1, kKEmpty = 3, kVFull = 5, kVEmpty = 8, kSFull = 11, kPFull = 13,
              kOFull = 15, kDrain = 17, kNumBars = 18;

struct ExtendKernelArgs {
    PoolView pool;
    PageView pages;
    const int32_t *prefix_lens, *ext_lens, *cu_ext, *positions;
    int32_t hq, group, rows_per_tile, q_box_rows, total_tokens, num_reqs, nblk, oob_row;
    int32_t box_rows;     // rows of one tiled pool box (min(page_size, 128)); 0 = gather only
    int32_t v_blocks;     // V tiles in blocks of 16 keys (tiled page copies); 0 = laid out as K
    float scale_log2;
    __nv_bfloat16 *o;
    float *lse;
    uint32_t *status;
    int32_t pdl_wait;     // launched behind a kernel it must not outlive (see the kernel's start)
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              uint32_t *status) {
    if (ptx::mbar_wait(bar, parity)) return true;
    report(status, MSGL_DEVERR_TIMEOUT);
    *abort_flag = 1;
    return false;
}

__global__ void __launch_bounds__(kThreads, 1)
    extend_tc_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap k_map,
                     const __grid_constant__ CUtensorMap v_map, const __grid_constant__ CUtensorMap kt_map,
                     const __grid_constant__ CUtensorMap vt_map, const ExtendKernelArgs a) {
    extern __shared__ uint8_t smem_raw[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Launched with programmatic dependent launch behind the decode split of a mixed step,
    // this grid may start before the split has finished.  The last CTA waits for it, so the
    // grid cannot complete before the split has: whatever the stream runs next after this
    // grid sees the split's partials.  It reads nothing the split writes.  The last CTA is
    // handed out last, long after the split is done, so the wait returns at once.
    if (a.pdl_wait && blockIdx.x == gridDim.x - 1 && threadIdx.x == 0)
        asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- work item: heaviest token blocks first, then kv head, then request
    const int per_rank = a.pool.hkv * a.num_reqs;
    const int rank = blockIdx.x / per_rank;
    const int rest = blockIdx.x - rank * per_rank;
    const int g = rest % a.pool.hkv;
    const int b = rest / a.pool.hkv;
    const int blk = a.nblk - 1 - rank;
    const int R = a.rows_per_tile, G = a.group;
    const int ext = __ldg(a.ext_lens + b);
    const int pre = __ldg(a.prefix_lens + b);
    const int cu_b = __ldg(a.cu_ext + b);
    const int i0 = blk * 2 * R;
    if (blk == 0 && g == 0 && threadIdx.x == 0) {
        if (ext > a.nblk * 2 * R || __ldg(a.cu_ext + b + 1) - cu_b != ext || pre < 0 || cu_b < 0 ||
            (long long)cu_b + ext > a.total_tokens)
            report(a.status, MSGL_DEVERR_LENGTH);
    }
    if (i0 >= ext || pre < 0 || cu_b < 0 || (long long)cu_b + ext > a.total_tokens) return;

    const int nA = min(R, ext - i0);
    const int nB = max(0, min(R, ext - i0 - R));
    const int nkv0 = (pre + i0 + nA + kKeys - 1) / kKeys;          // K/V tiles tile 0 needs
    const int nkv1 = nB > 0 ? (pre + i0 + R + nB + kKeys - 1) / kKeys : 0;
    const int nkv = max(nkv0, nkv1);
    const int nkeys = nB > 0 ? pre + i0 + R + nB : pre + i0 + nA;
    const int tok0 = cu_b + i0;

    const uint32_t raw = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + kOffBar;
    auto bar = [&](int i) -> uint32_t { return bar0 + 8u * (uint32_t)i; };
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(smem + kOffBar + 8 * kNumBars);
    volatile int *min_bad = reinterpret_cast<volatile int *>(smem + kOffBar + 8 * kNumBars + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + kOffBar + 8 * kNumBars + 8);

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(kQFull), 1);
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar(kKFull + s), 1);
            ptx::mbar_init(bar(kKEmpty + s), 1);
        }
        for (int s = 0; s < kVStages; ++s) {
            ptx::mbar_init(bar(kVFull + s), 1);
            ptx::mbar_init(bar(kVEmpty + s), 1);
        }
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bar(kSFull + t), 1);
            ptx::mbar_init(bar(kPFull + t), 4);
            ptx::mbar_init(bar(kOFull + t), 1);
        }
        ptx::mbar_init(bar(kDrain), 1);
        *min_bad = INT_MAX;
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 2) {
        ptx::tc_alloc(ptx::smem_u32((const void *)tmem_slot), 512);
        ptx::tc_relinquish();
    }
    if (warp == 2 || warp == 3) {
        // zero the Q rows a TMA box does not cover (GQA padding rows)
        const int used = a.q_box_rows * G;
        const int pad_bytes = (kRows - used) * 128;
        for (int t = 0; t < 2; ++t)
            for (int h = 0; h < 2; ++h) {
                uint8_t *p = smem + kOffQ + t * kTile + h * kHalf + used * 128;
                for (int x = (threadIdx.x - 64) * 16; x < pad_bytes; x += 64 * 16)
                    *reinterpret_cast<uint4 *>(p + x) = make_uint4(0, 0, 0, 0);
            }
        ptx::fence_proxy_async_smem();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Loaders: warp 0 brings Q and the K tiles, warp 3 the V tiles (one issuing warp per
    // operand; a single warp issuing both was the bottleneck at small page sizes).  With
    // no tiled boxes (page_size < 16) K/V rows are copied with 16-byte cp.async instead
    // of TMA gathers, and warp 2 takes the odd K tiles so two K copies are in flight.
    const bool lsu = a.box_rows == 0;
    if (warp == 0 || warp == 3 || (lsu && warp == 2)) {
        // ---------------------------------------------------------------- K/V loaders
        const bool is_v = warp == 3;
        if (warp == 0 && lane == 0) {
            const uint32_t box = 64u * G * a.q_box_rows * 2u;
            ptx::mbar_arrive_expect_tx(bar(kQFull), box * (nB > 0 ? 4u : 2u));
            for (int t = 0; t < (nB > 0 ? 2 : 1); ++t)
                for (int h = 0; h < 2; ++h)
                    ptx::tma_load_3d(sbase + kOffQ + t * kTile + h * kHalf, &q_map, 64 * h, g * G,
                                     tok0 + t * R, bar(kQFull));
        }
        // Pool rows of the tile's keys, four consecutive keys per lane.  A key past the
        // causal range or behind a bad page id gets oob_row (zero fill).
        auto key_rows = [&](int j, int (&rows)[4], bool &all_ok, int64_t &slot0) {
            all_ok = true;
            slot0 = 0;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = j * kKeys + 4 * lane + e;
                rows[e] = a.oob_row;
                if (key < nkeys) {
                    bool badp = false;
                    const int64_t slot = slot_of(a.pool, a.pages, b, key, badp);
                    if (badp) {
                        atomicMin((int *)min_bad, key);
                        all_ok = false;
                    } else {
                        rows[e] = (int)(slot * a.pool.hkv + g);
                        if (e == 0) slot0 = slot;
                    }
                } else {
                    all_ok = false;
                }
            }
        };
        int rows[4];
        bool all_ok;
        int64_t slot0;
        if (lsu) {
            // 16-byte cp.async copies into the SWIZZLE_128B K-major layout: per step, lanes
            // 0-15 copy key 2i and lanes 16-31 key 2i + 1, one 16-byte chunk each (each key's
            // 256-byte row is contiguous in the pool).  The rows of the next tile are looked
            // up while the copies fly; writer-side proxy fence, then one arrival.
            const __nv_bfloat16 *pool = is_v ? a.pool.v : a.pool.k;
            const int step = is_v ? 1 : 2, first = warp == 2 ? 1 : 0;
            const int hi = lane >> 4, c = lane & 15;
            const uint32_t col_off = (uint32_t)(c >> 3) * kHalf;
            int next[4];
            if (first < nkv) key_rows(first, rows, all_ok, slot0);
            for (int j = first; j < nkv && !*abort_flag; j += step) {
                const int sv = j % kVStages;
                const uint32_t empty = is_v ? bar(kVEmpty + sv) : bar(kKEmpty + (j & 1));
                const uint32_t parity = is_v ? ((j / kVStages) & 1) ^ 1 : ((j >> 1) & 1) ^ 1;
                if (!wait_or_abort(empty, parity, abort_flag, a.status)) break;
                const uint32_t dst = is_v ? sbase + kOffV + sv * kTile : sbase + kOffK + (j & 1) * kTile;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const int e0 = (i & 1) * 2;
                    const int r0 = __shfl_sync(0xffffffffu, rows[e0], i >> 1);
                    const int r1 = __shfl_sync(0xffffffffu, rows[e0 + 1], i >> 1);
                    const int row = hi ? r1 : r0;
                    const int r = 2 * i + hi;
                    const bool valid = row < a.oob_row;
                    ptx::cp_async_16(dst + col_off + (uint32_t)r * 128u + ((uint32_t)((c & 7) ^ (r & 7)) << 4),
                                     pool + (valid ? (int64_t)row * kHeadDim + c * 8 : 0), valid ? 16u : 0u);
                }
                ptx::cp_async_commit();
                if (j + step < nkv) key_rows(j + step, next, all_ok, slot0);
                ptx::cp_async_wait_all();
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(is_v ? bar(kVFull + sv) : bar(kKFull + (j & 1)));
#pragma unroll
                for (int e = 0; e < 4; ++e) rows[e] = next[e];
            }
            ptx::cp_async_wait_all();
            if (*abort_flag && warp == 0) ptx::mbar_wait(bar(kQFull), 0, 200000000LL);
        } else {
            // TMA: a page that is a contiguous run of pool rows and fully valid arrives in
            // one tiled copy per 64-dim half, issued by its first lane; any other 4-key
            // group is gathered four rows at a time.
            const int BR = a.box_rows;
            const int lanes_per_box = BR / 4;
            const int box_lead = (lane / lanes_per_box) * lanes_per_box;
            const unsigned box_bits =
                lanes_per_box >= 32 ? 0xffffffffu : ((1u << lanes_per_box) - 1u) << box_lead;
            const CUtensorMap *gm = is_v ? &v_map : &k_map;
            const CUtensorMap *tm = is_v ? &vt_map : &kt_map;
            int issued = 0;
            for (int j = 0; j < nkv && !*abort_flag; ++j) {
                key_rows(j, rows, all_ok, slot0);
                const unsigned ok_mask = __ballot_sync(0xffffffffu, all_ok);
                const bool tiled = (ok_mask & box_bits) == box_bits;
                const int sv = j % kVStages;
                const uint32_t empty = is_v ? bar(kVEmpty + sv) : bar(kKEmpty + (j & 1));
                const uint32_t parity = is_v ? ((j / kVStages) & 1) ^ 1 : ((j >> 1) & 1) ^ 1;
                if (!wait_or_abort(empty, parity, abort_flag, a.status)) break;
                const uint32_t full = is_v ? bar(kVFull + sv) : bar(kKFull + (j & 1));
                // this lane's four keys: rows 4 lane .. 4 lane + 3 (K), or their place in V's blocks
                const bool vb = is_v && a.v_blocks;
                const uint32_t dst = vb ? sbase + kOffV + sv * kTile + (uint32_t)(lane >> 2) * kVBlock +
                                              (uint32_t)(lane & 3) * 512u
                                        : (is_v ? sbase + kOffV + sv * kTile : sbase + kOffK + (j & 1) * kTile) +
                                              lane * 512;
                const uint32_t half_off = vb ? kVHalf : kHalf;
                if (lane == 0) ptx::mbar_arrive_expect_tx(full, kTile);
                __syncwarp();
                if (!tiled) {
                    ptx::tma_gather4(dst, gm, 0, rows[0], rows[1], rows[2], rows[3], full);
                    ptx::tma_gather4(dst + half_off, gm, 64, rows[0], rows[1], rows[2], rows[3], full);
                } else if (lane == box_lead) {
                    if (vb) {
                        // the page's blocks, two (8 KB) at most per copy: {64 dims, head g, 16
                        // slots, 2 halves, 1 or 2 blocks}.  Larger copies held up the K copies
                        // queued behind them on the same copy engine.
                        for (int n = 0; n < (BR > 32 ? BR / 32 : 1); ++n)
                            ptx::tma_load_5d(dst + (uint32_t)n * 2u * kVBlock, tm, 0, g, (int)slot0 + 32 * n, 0, 0,
                                             full);
                    } else {
                        ptx::tma_load_3d(dst, tm, 0, g, (int)slot0, full);
                        ptx::tma_load_3d(dst + kHalf, tm, 64, g, (int)slot0, full);
                    }
                }
                issued = j + 1;
            }
            if (*abort_flag) {
                // let issued copies land before shared memory goes away (bounded waits)
                if (warp == 0) ptx::mbar_wait(bar(kQFull), 0, 200000000LL);
                const int depth = is_v ? kVStages : kStages;
                for (int j = max(0, issued - depth); j < issued; ++j)
                    ptx::mbar_wait(is_v ? bar(kVFull + j % kVStages) : bar(kKFull + (j & 1)),
                                   is_v ? (j / kVStages) & 1 : (j >> 1) & 1, 200000000LL);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = ptx::umma_idesc_bf16(128, 128, false, false);
            constexpr uint32_t idesc_o = ptx::umma_idesc_bf16(128, 128, false, true);
            bool ok = wait_or_abort(bar(kQFull), 0, abort_flag, a.status);
            ptx::tc_fence_after();
            // The issuing thread runs at the tensor pipe's pace (an MMA issues once the one
            // before it is nearly done), so every cycle it spends between two groups is a
            // cycle the pipe idles.  Each group therefore tests, after its 4th MMA and with the
            // non-blocking test_wait, the barrier the next group needs: the test's latency
            // hides behind the MMAs still queued, and the bounded wait runs only when the
            // phase has not completed yet.  Descriptors are built once and advanced by adding
            // the offset (address >> 4) to their start-address field.
            const uint64_t qdesc = ptx::umma_desc_sw128(sbase + kOffQ, 16, 1024);
            const uint64_t kdesc = ptx::umma_desc_sw128(sbase + kOffK, 16, 1024);
            const uint64_t vdesc = ptx::umma_desc_sw128(sbase + kOffV, a.v_blocks ? kVHalf : kHalf, 1024);
            const uint32_t vstep = (a.v_blocks ? kVBlock : 16u * 128u) >> 4;   // MMA kk's 16 keys
            // S_t = Q_t K^T for tile t from the K stage at descriptor kd (8 MMAs over the 128
            // dims); returns the test of (pb, pp), or false when pb is 0
            auto s_group = [&](int t, uint64_t kd, uint32_t pb, uint32_t pp) -> bool {
                const uint64_t qd = qdesc + (uint64_t)(t * (kTile >> 4));
                bool r = false;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
                    ptx::tc_mma_ss(tmem + 128 * t, qd + off, kd + off, idesc_s, kk > 0);
                    if (kk == 3 && pb) r = ptx::mbar_test_wait(pb, pp);
                }
                ptx::tc_commit(bar(kSFull + t));
                return r;
            };
            // O_t += P_t V from the V stage at descriptor vd (P from TMEM, 8 MMAs over the 128
            // keys); acc = 0 starts O_t
            auto pv_group = [&](int t, uint64_t vd, bool acc, uint32_t pb, uint32_t pp) -> bool {
                bool r = false;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    ptx::tc_mma_ts(tmem + 256 + 128 * t, tmem + 128 * t + kk * 8, vd + (uint64_t)(kk * vstep),
                                   idesc_o, (acc || kk > 0) ? 1u : 0u);
                    if (kk == 3 && pb) r = ptx::mbar_test_wait(pb, pp);
                }
                return r;
            };
            auto issue_s = [&](int t, int j, uint32_t pb, uint32_t pp) -> bool {
                return s_group(t, kdesc + (uint64_t)((j & 1) * (kTile >> 4)), pb, pp);
            };
            auto issue_pv = [&](int t, int j, uint32_t pb, uint32_t pp) -> bool {
                const bool r = pv_group(t, vdesc + (uint64_t)((j % kVStages) * (kTile >> 4)), j > 0, pb, pp);
                // only the epilogue waits for O_t: the completion of S_t(j+1), issued after
                // PV_t(j) by this thread, already tells the softmax that PV_t(j) is done
                if (j == (t ? nkv1 : nkv0) - 1) ptx::tc_commit(bar(kOFull + t));
                return r;
            };
            // Order per K/V tile j: PV_0(j), S_0(j+1), PV_1(j), S_1(j+1).  The next S of a
            // tile goes in right after its PV (same TMEM columns; tcgen05 MMAs from one
            // thread execute in order), so tile 0's next softmax overlaps tile 1's.
            bool v_ok = false;   // V_j's barrier, tested during S_1(j)
            if (ok && (ok = wait_or_abort(bar(kKFull + 0), 0, abort_flag, a.status))) {
                ptx::tc_fence_after();
                if (nkv0 > 0) issue_s(0, 0, 0, 0);
                if (nkv1 > 0) v_ok = issue_s(1, 0, bar(kVFull + 0), 0);
            }
            int j = 0;
            {
                // Steady state: both tiles have K/V tiles j and j + 1, so all four groups run
                // and none is a tile's last; the stages advance by counters.
                const int jss = nB > 0 ? nkv0 - 1 : 0;
                uint32_t vs = 0, vpar = 0;   // V stage of tile j and the parity of its phase
                uint32_t ks = 1, kpar = 0;   // K stage of tile j + 1 and the parity of its phase
                for (; ok && j < jss; ++j) {
                    if (!v_ok && !(ok = wait_or_abort(bar(kVFull) + 8u * vs, vpar, abort_flag, a.status))) break;
                    if (!(ok = wait_or_abort(bar(kPFull + 0), j & 1, abort_flag, a.status))) break;
                    ptx::tc_fence_after();
                    const uint64_t vd = vdesc + (uint64_t)(vs * (kTile >> 4));
                    const uint32_t b_k = bar(kKFull) + 8u * ks;
                    if (!pv_group(0, vd, j > 0, b_k, kpar) && !(ok = wait_or_abort(b_k, kpar, abort_flag, a.status)))
                        break;
                    ptx::tc_fence_after();
                    const uint64_t kd = kdesc + (uint64_t)(ks * (kTile >> 4));
                    if (!s_group(0, kd, bar(kPFull + 1), j & 1) &&
                        !(ok = wait_or_abort(bar(kPFull + 1), j & 1, abort_flag, a.status)))
                        break;
                    ptx::tc_fence_after();
                    pv_group(1, vd, j > 0, 0, 0);
                    vs = vs == kVStages - 1 ? 0 : vs + 1;
                    vpar ^= vs == 0 ? 1u : 0u;
                    v_ok = s_group(1, kd, bar(kVFull) + 8u * vs, vpar);
                    ks ^= 1u;
                    kpar ^= ks == 0 ? 1u : 0u;
                }
            }
            for (; ok && j < nkv; ++j) {
                const int jn = j + 1, sn = jn & 1, phn = (jn >> 1) & 1;
                const bool more = jn < nkv;
                if (!v_ok && !(ok = wait_or_abort(bar(kVFull + j % kVStages), (j / kVStages) & 1, abort_flag, a.status)))
                    break;
                bool k_ok = false, p1_ok = false;
                if (j < nkv0) {
                    if (!(ok = wait_or_abort(bar(kPFull + 0), j & 1, abort_flag, a.status))) break;
                    ptx::tc_fence_after();
                    k_ok = issue_pv(0, j, more ? bar(kKFull + sn) : 0u, phn);
                }
                if (more) {
                    if (!k_ok && !(ok = wait_or_abort(bar(kKFull + sn), phn, abort_flag, a.status))) break;
                    ptx::tc_fence_after();
                    if (jn < nkv0) p1_ok = issue_s(0, jn, j < nkv1 ? bar(kPFull + 1) : 0u, j & 1);
                }
                if (j < nkv1) {
                    if (!p1_ok && !(ok = wait_or_abort(bar(kPFull + 1), j & 1, abort_flag, a.status))) break;
                    ptx::tc_fence_after();
                    issue_pv(1, j, 0, 0);
                }
                v_ok = false;
                if (more && jn < nkv1) v_ok = issue_s(1, jn, bar(kVFull + jn % kVStages), (jn / kVStages) & 1);
            }
            // drain: every MMA issued above has completed once this fires
            ptx::tc_commit(bar(kDrain));
            ptx::mbar_wait(bar(kDrain), 0, 400000000LL);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- softmax
        const int t = (warp - 4) >> 2;                 // Q tile of this warpgroup
        const int quad = warp & 3;
        const int r = quad * 32 + lane;                // TMEM lane = tile row
        const int tok_l = r / G, jh = r - tok_l * G;
        const int n_t = t == 0 ? nA : nB;
        const int i_row = i0 + t * R + tok_l;
        const bool row_valid = (r < R * G) && (tok_l < n_t);
        const int limit = pre + i_row;                 // last key this row may see
        const int jm = (pre + i0 + t * R + 1) >> 7;    // tiles >= jm may need masking
        const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
        const uint32_t tS = tmem + lane_base + 128 * t;
        const uint32_t tO = tmem + lane_base + 256 + 128 * t;
        float m_ref = -INFINITY, l = 0.f;
        const int my_nkv = t ? nkv1 : nkv0;
        bool ok = true;
        // The K/V stages are released from here, not by commits of the MMA thread (whose
        // every instruction between two MMA groups leaves the tensor pipe idle): the
        // completion of S_r(j), r the last tile (it has the most K/V tiles), means every
        // MMA issued before it is done, so K_j (read by S_0(j) and S_r(j)) and V_{j-1} (read
        // by PV_0(j-1) and PV_r(j-1)) are free.
        const bool releaser = lane == 0 && warp == (nB > 0 ? 8 : 4);
        for (int j = 0; j < my_nkv; ++j) {
            // S_t(j) complete: PV_t(j-1), issued before it by the same thread, is done too
            if (!(ok = wait_or_abort(bar(kSFull + t), j & 1, abort_flag, a.status))) break;
            ptx::tc_fence_after();
            if (releaser) {
                ptx::mbar_arrive(bar(kKEmpty + (j & 1)));
                if (j > 0) ptx::mbar_arrive(bar(kVEmpty + (j - 1) % kVStages));
            }
            const bool masked = j >= jm;             // uniform: only tiles past the first row's limit
            const int lim = limit - j * kKeys;       // key c of this tile is visible iff c <= lim
            // one TMEM read of the row's 128 scores
            uint32_t v[128];
            ptx::tc_ld32(tS + 0, *reinterpret_cast<uint32_t(*)[32]>(v + 0));
            ptx::tc_ld32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
            ptx::tc_ld32(tS + 64, *reinterpret_cast<uint32_t(*)[32]>(v + 64));
            ptx::tc_ld32(tS + 96, *reinterpret_cast<uint32_t(*)[32]>(v + 96));
            ptx::tc_wait_ld();
            if (masked) {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (i > lim) v[i] = __float_as_uint(-INFINITY);
            }
            // row max in four independent 3-input chains (16 deep each), scaled to log2 units
            auto row_max = [&]() -> float {
                float mxa = -INFINITY, mxb = -INFINITY, mxc = -INFINITY, mxd = -INFINITY;
#pragma unroll
                for (int i = 0; i < 128; i += 8) {
                    mxa = ptx::max3(mxa, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                    mxb = ptx::max3(mxb, __uint_as_float(v[i + 2]), __uint_as_float(v[i + 3]));
                    mxc = ptx::max3(mxc, __uint_as_float(v[i + 4]), __uint_as_float(v[i + 5]));
                    mxd = ptx::max3(mxd, __uint_as_float(v[i + 6]), __uint_as_float(v[i + 7]));
                }
                return fmaxf(fmaxf(mxa, mxb), fmaxf(mxc, mxd)) * a.scale_log2;
            };
            // The first tile sets the reference m_ref to the row max.  Later tiles write P from
            // the reference straight away: a score more than 2^8 above it makes some p > 256
            // and so the row sum >= 256 (a NaN fails the test too).  Only then is the row max
            // taken; a row whose max passes m_ref + 8 moves its reference there, its O and l
            // are rescaled, and P is written again.  Every p stays below 2^8 either way.
            if (j == 0) m_ref = fmaxf(m_ref, row_max());
            float ls = 0.f;
#pragma unroll 1
            for (int pass = 0;; ++pass) {
                // P = 2^(s * scale_log2 - m_ref) (masked scores are -inf -> 0), back over S as bf16
                const uint64_t sc2 = ptx::f2_pack(a.scale_log2, a.scale_log2);
                const uint64_t nm2 = ptx::f2_pack(-m_ref, -m_ref);
                uint64_t l2 = ptx::f2_pack(0.f, 0.f);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int e = 32 * c + 2 * i;
                        const uint64_t x2 = ptx::f2_fma(ptx::f2_pack(__uint_as_float(v[e]), __uint_as_float(v[e + 1])),
                                                        sc2, nm2);
                        float x0, x1;
                        ptx::f2_unpack(x2, x0, x1);
                        const float p0 = ptx::ex2(x0), p1 = ptx::ex2(x1);
                        l2 = ptx::f2_add(l2, ptx::f2_pack(p0, p1));
                        pk[i] = ptx::pack_bf16(p0, p1);
                    }
                    ptx::tc_st16(tS + 16 * c, pk);
                }
                float la, lb;
                ptx::f2_unpack(l2, la, lb);
                ls = la + lb;
                if (pass == 1 || j == 0 || __all_sync(0xffffffffu, ls < 256.f)) break;
                const float m_new = fmaxf(m_ref, row_max());
                const bool need = m_new > m_ref + 8.f;
                if (!__any_sync(0xffffffffu, need)) break;
                const float alpha = need ? ptx::ex2(m_ref - m_new) : 1.f;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t o32[32];
                    ptx::tc_ld32(tO + 32 * c, o32);
                    ptx::tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o32[i] = __float_as_uint(__uint_as_float(o32[i]) * alpha);
                    ptx::tc_st32(tO + 32 * c, o32);
                }
                ptx::tc_wait_st();
                l *= alpha;
                if (need) m_ref = m_new;
            }
            l += ls;
            ptx::tc_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(kPFull + t));
        }
        // epilogue: O / l -> bf16, lse = ln(sum exp(s))
        if (ok && my_nkv > 0 && wait_or_abort(bar(kOFull + t), 0, abort_flag, a.status)) {
            ptx::tc_fence_after();
            const int tok_g = tok0 + t * R + tok_l;
            const bool store = row_valid && tok_g < a.total_tokens;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const long long orow = ((long long)tok_g * a.hq + (long long)g * G + jh);
            const bool o_aligned32 = (reinterpret_cast<uintptr_t>(a.o) & 31u) == 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                ptx::tc_ld32(tO + 32 * c, v);
                ptx::tc_wait_ld();
                if (store) {
                    __nv_bfloat16 *dst = a.o + orow * kHeadDim + 32 * c;
                    uint32_t w[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        w[q] = ptx::pack_bf16(__uint_as_float(v[2 * q]) * inv, __uint_as_float(v[2 * q + 1]) * inv);
                    if (o_aligned32) {
                        // 32-byte stores: half the store instructions of 16-byte ones
                        ptx::st_v8(dst, w);
                        ptx::st_v8(dst + 16, w + 8);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            reinterpret_cast<uint4 *>(dst)[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
                    }
                }
            }
            if (store) {
                a.lse[orow] = (m_ref + log2f(l)) * kLn2;
                if (a.positions && jh == 0 && __ldg(a.positions + tok_g) != limit)
                    report(a.status, MSGL_DEVERR_POSITION);
            }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp >= 4) {
        // rows that would have read a key behind a bad page id: o = 0, lse = -inf
        const int bad_key = *min_bad;
        if (bad_key != INT_MAX) {
            const int t = (warp - 4) >> 2;
            const int r = (warp & 3) * 32 + lane;
            const int tok_l = r / G, jh = r - tok_l * G;
            const int n_t = t == 0 ? nA : nB;
            const int tok_g = tok0 + t * R + tok_l;
            if (r < R * G && tok_l < n_t && tok_g < a.total_tokens && pre + i0 + t * R + tok_l >= bad_key) {
                const long long orow = ((long long)tok_g * a.hq + (long long)g * G + jh);
                uint4 *dst = reinterpret_cast<uint4 *>(a.o + orow * kHeadDim);
                for (int q = 0; q < 16; ++q) dst[q] = make_uint4(0, 0, 0, 0);
                a.lse[orow] = -INFINITY;
            }
            if (threadIdx.x == 128) report(a.status, MSGL_DEVERR_PAGE_RANGE);
        }
    }
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tc_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------- host side

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

size_t extend_workspace_bytes(int32_t, int32_t, int32_t, int32_t, int32_t) { return 0; }

cudaError_t launch_extend(const ExtendArgs &a, cudaStream_t stream) {
    if (a.num_reqs == 0 || a.total_tokens == 0 || a.max_ext_len == 0) return cudaSuccess;
    const int hkv = a.pool.hkv;
    const int G = a.hq / hkv;
    const int R = kRows / G;
    const int q_box_rows = R < a.total_tokens ? R : a.total_tokens;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;

    CUtensorMap qm, km, vm;
    {
        cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)a.hq, (cuuint64_t)a.total_tokens};
        cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)a.hq * kHeadDim * 2};
        cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)q_box_rows};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void *)a.q, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const long long pool_rows = a.pool.num_slots * hkv;
    if (pool_rows >= INT_MAX) return cudaErrorInvalidValue;
    // 2D view {128 dims, slots x heads} for four-row gathers
    for (int which = 0; which < 2; ++which) {
        cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)pool_rows};
        cuuint64_t strides[1] = {(cuuint64_t)kHeadDim * 2};
        cuuint32_t box[2] = {64, 1};
        cuuint32_t es[2] = {1, 1};
        if (enc(which ? &vm : &km, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                (void *)(which ? a.pool.v : a.pool.k), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // tiled 3D view {128 dims, Hkv heads, slots}: one box = box_rows slots of one head
    CUtensorMap ktm, vtm;
    memset(&ktm, 0, sizeof ktm);
    memset(&vtm, 0, sizeof vtm);
    const int page = 1 << a.pool.log2_ps;
    const int box_rows = page >= 16 ? (page < kKeys ? page : kKeys) : 0;
    const int v_blocks = box_rows > 0;
    if (box_rows > 0) {
        cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)hkv, (cuuint64_t)a.pool.num_slots};
        cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)hkv * kHeadDim * 2};
        cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
        cuuint32_t es[3] = {1, 1, 1};
        if (enc(&ktm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void *)a.pool.k, dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
        if (v_blocks) {
            // V: 5D view {64 dims, Hkv heads, 16 slots, 2 halves (128 bytes apart), blocks of
            // 16 slots}: one box brings one or two blocks in V's layout.  The view aliases slots
            // across its 3rd and 5th dimensions, so its bounds do not guard the pool: the
            // kernel uses a box only for a page whose slots are all valid.
            cuuint64_t vdims[5] = {64, (cuuint64_t)hkv, (cuuint64_t)a.pool.num_slots, 2, (cuuint64_t)(kKeys / 16)};
            cuuint64_t vstrides[4] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)hkv * kHeadDim * 2, 128,
                                      (cuuint64_t)16 * hkv * kHeadDim * 2};
            cuuint32_t vbox[5] = {64, 1, 16, 2, (cuuint32_t)(box_rows > 32 ? 2 : box_rows / 16)};
            cuuint32_t ves[5] = {1, 1, 1, 1, 1};
            if (enc(&vtm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, (void *)a.pool.v, vdims, vstrides, vbox, ves,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cudaErrorInvalidValue;
        } else if (enc(&vtm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void *)a.pool.v, dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            return cudaErrorInvalidValue;
        }
    }
    static bool attr_set[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(extend_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    ExtendKernelArgs k{};
    k.pool = a.pool;
    k.pages = a.pages;
    k.prefix_lens = a.prefix_lens;
    k.ext_lens = a.ext_lens;
    k.cu_ext = a.cu_ext;
    k.positions = a.positions;
    k.hq = a.hq;
    k.group = G;
    k.rows_per_tile = R;
    k.q_box_rows = q_box_rows;
    k.total_tokens = a.total_tokens;
    k.num_reqs = a.num_reqs;
    k.nblk = (a.max_ext_len + 2 * R - 1) / (2 * R);
    k.oob_row = (int)pool_rows;
    k.box_rows = box_rows;
    k.v_blocks = v_blocks;
    k.scale_log2 = a.scale * kLog2e;
    k.o = a.o;
    k.lse = a.lse;
    k.status = a.status;
    k.pdl_wait = a.pdl ? 1 : 0;
    const long long grid = (long long)k.nblk * hkv * a.num_reqs;
    if (grid >= INT_MAX) return cudaErrorInvalidValue;
    if (!a.pdl) {
        extend_tc_kernel<<<(unsigned)grid, kThreads, kSmemBytes, stream>>>(qm, km, vm, ktm, vtm, k);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, extend_tc_kernel, qm, km, vm, ktm, vtm, k);
}

}  // namespace msgl
