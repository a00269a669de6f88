// decode_sm103.cu -- paged MLA decode over the latent cache on the 5th-generation tensor cores.
//
// What it computes ([vLLM-MLA, two-algorithms section]; [vLLM-MLA, FlashMLA section]): for one
// query row (request b, query position t) and all H <= 128 heads, MQA attention over the
// row's visible tokens [j0, j1) (one split of it), every head reading the same 576-element
// cached row:  S = scale * Q K^T,  P = softmax(S),  O = P V  with V = the first 512 dims.
//
// One thread-block cluster of two CTAs per (query row, split) unit. Pages are taken four at a
// time ("groups" of 256 tokens) so that every tensor-core instruction has N = 256: with N = 256
// the tensor core holds enough queued work to hide the ~130-cycle gap that each blocking
// synchronisation of the issuing thread leaves, so the pipe stays busy between ring slots.
//
//   CTA 0 ("scores")  Q: the 512 latent dims (128 heads x 512 bf16) are loaded once by TMA and
//                     kept in tensor memory; the 64 rope dims stay in shared memory.
//                     K: a ring of four 32 KB slots, one slot = one 64-dim panel of a group's
//                     four pages (256 rows, 128-byte swizzle), refilled panel by panel by TMA as
//                     the MMAs release them.
//                     S = Q K^T per group: 36 tcgen05.mma of M=128 heads x N=256 tokens x K=16
//                     (32 with A from TMEM, 4 with A = rope dims from shared memory) into a
//                     256-column TMEM buffer.
//                     Softmax: eight warps, two per TMEM lane quarter, each owning two pages of
//                     the group for 32 heads; fp32 online softmax with a lazily moved running
//                     max (rescale only when a row's max grows by more than 2^8). Each thread
//                     writes its head's P row (bf16, in the MMA's swizzled K-major layout) and
//                     rescale factor into a local staging buffer for the page (one of four, one
//                     per page of the group); one thread per half then sends the whole buffer
//                     to CTA 1's P buffer for the page with a single bulk copy, whose bytes
//                     complete CTA 1's barrier for that buffer. One bulk copy moves the 17 KB
//                     about twice as fast as 128 threads' st.async stores, and the softmax
//                     warps are free as soon as their shared-memory writes are done.
//   CTA 1 ("output")  holds the 128 x 512 fp32 output accumulator -- all 512 TMEM columns of its
//                     SM, the reason the work is split over two SMs -- streams the pages'
//                     first 512 dims (mostly L2 hits), and accumulates O += P V per page with
//                     tcgen05.mma (M=128, N=2x256, K=64; V read as an MN-major operand straight
//                     from the TMA tile). Its MMA thread waits for P, the helpers and V; four
//                     helper warps re-arm the P buffers, rescale O, zero the V rows past the
//                     last token, and (with four more warps) run the epilogue. Until the
//                     epilogue those four other warps prefetch into L2 the pages that CTA 0
//                     will load about one group later, so that its K loads hit L2.
// Per page the pair issues exactly the algorithm's 2*128*64*(576+512) flops.
//
// Rows past the split's last visible token are masked by index (S = -inf) and, in the last
// partial page, zeroed in CTA 1's V tile so that stale or NaN bytes cannot leak through 0 * NaN.
// All waits are bounded (see sm103_ptx.cuh); on a timeout the kernel winds down and reports
// MLA_DEV_WAIT_TIMEOUT instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <cstring>

#include "decode_common.cuh"
#include "internal.h"
#include "sm103_ptx.cuh"

namespace mla {

cudaError_t encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128);

namespace {

using namespace ptx;
using namespace dec;

// Hint: bring the 128-byte line at `ptr` into L2 (no effect on correctness).
__device__ __forceinline__ void prefetch_l2(const void* ptr) { asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr)); }

// A 32-bit global load through the non-coherent path, issued where it stands in program order
// (the asm is volatile), for data that no kernel of the grid writes.
__device__ __forceinline__ int ld_nc_s32(const int32_t* ptr) {
    int v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(ptr));
    return v;
}

constexpr int kThreads = 320;        // warp 0 TMA, warp 1 MMA, warps 2-9 softmax (CTA 0) / 2-5 helpers, 2-9 epilogue (CTA 1)
constexpr int kPPG = 4;              // pages per group
constexpr int kSlots = 4;            // CTA 0 K ring slots (32 KB each)
constexpr int kPageBox = 64 * 128;   // one page's rows of one 64-dim panel (8 KB)
constexpr int kSlotBytes = kPPG * kPageBox;  // 32 KB
constexpr int kQPanelBytes = 128 * 128;      // 128 heads x 64 dims of Q (16 KB)
constexpr int kPBufs = 5;            // CTA 1 P buffers (one page each): P arrives up to 5 pages ahead
constexpr int kVStages = 2;          // CTA 1 V ring stages of kVRows tokens x 512 dims
constexpr int kVRows = 64;           // one page per V stage
constexpr int kVPerPage = kPage / kVRows;        // V stages per page
constexpr int kVBox = kVRows * 128;             // one 64-dim panel of a V stage (8 KB)
constexpr int kVStageBytes = 8 * kVBox;         // 64 KB
constexpr int kPBytes = 128 * 128;              // P page: 128 heads x 64 tokens bf16
constexpr int kPMsgBytes = (kPBytes + 512 + 4 + 15) / 16 * 16;  // P + alpha[128] + flag word, in 16-byte units
constexpr int kPBufStride = 17 * 1024;
constexpr int kCtrlBytes = 4096;
// CTA 0 layout
constexpr int OFF_QROPE = kCtrlBytes;                      // 16 KB
constexpr int OFF_RING = OFF_QROPE + kQPanelBytes;         // 4 x 32 KB
constexpr int OFF_STAGE = OFF_RING + kSlots * kSlotBytes;  // 4 P staging buffers, kPBufStride apart
constexpr int kSmem0 = OFF_STAGE + 4 * kPBufStride;
// CTA 1 layout
constexpr int OFF_V = kCtrlBytes;
constexpr int OFF_PB = OFF_V + kVStages * kVStageBytes;
constexpr int kSmem1 = OFF_PB + kPBufs * kPBufStride;
constexpr int kSmemBytes = kSmem0 > kSmem1 ? kSmem0 : kSmem1;
static_assert(kSmemBytes <= 232448, "over the per-CTA shared memory limit");
static_assert(kPMsgBytes <= kPBufStride, "P message");
// Q's latent panels land in the four staging buffers (panels 0-3) and ring slots 2-3 (panels
// 4-7), so that the first K panels can load into slots 0 and 1 at once; P is staged only after
// the first S, which needs Q in tensor memory.
static_assert(kSlots == 4 && kPBufStride >= kQPanelBytes && 4 * kQPanelBytes == 2 * kSlotBytes, "Q panel homes");
static_assert(OFF_RING % 1024 == 0 && OFF_STAGE % 1024 == 0 && OFF_PB % 1024 == 0 && kPBufStride % 1024 == 0 && kVBox % 1024 == 0,
              "128-byte swizzled tiles need 1024-byte alignment");
// the epilogue stages its output tiles over the V ring and the P buffers
static_assert(OFF_V + 8 * 128 * 128 <= kSmem1, "epilogue tiles");
__device__ __forceinline__ uint32_t q_panel_off(int pn) {
    return pn < 4 ? OFF_STAGE + pn * kPBufStride : OFF_RING + 2 * kSlotBytes + (pn - 4) * kQPanelBytes;
}

// Barrier slots (8 bytes each); one layout for both CTAs so that a multicast commit from CTA 1
// lands on CTA 0's B_PEMPTY slots.
enum : int {
    B_SLOTFULL = 0,                    // [kSlots] CTA0: ring slot landed (TMA tx)
    B_SLOTEMPTY = B_SLOTFULL + kSlots, // [kSlots] CTA0: ring slot consumed by the QK MMAs
    B_SFULL = B_SLOTEMPTY + kSlots,    // CTA0: S ready
    B_SEMPTY,                          // CTA0: S read into registers by the softmax warps (256)
    B_QFULL,                           // CTA0: Q landed in shared memory (TMA tx)
    B_QREADY,                          // CTA0: Q latent dims moved to TMEM, ring free for K (256)
    B_PEMPTY,                          // [kPBufs] both CTAs: PV MMA of the page in P buffer b completed
    B_VFULL = B_PEMPTY + kPBufs,       // [kVStages] CTA1: V stage landed
    B_VEMPTY = B_VFULL + kVStages,     // [kVStages] CTA1: V stage consumed
    B_PFULL = B_VEMPTY + kVStages,     // [kPBufs] CTA1: P message landed (bulk copy bytes from CTA0)
    B_READY = B_PFULL + kPBufs,        // [kPBufs] CTA1: page ready for its PV MMA (128 helper threads)
    B_STATS = B_READY + kPBufs,        // CTA1: final row statistics written by CTA0 (one cluster-scope arrive)
    B_STAGEFREE,                       // [4] CTA0: staging buffer's copy has landed (remote arrive from CTA1)
    B_COUNT = B_STAGEFREE + 4
};
static_assert(8 * B_COUNT <= 512, "barrier slots");
constexpr int OFF_TMEM = 512;
constexpr int OFF_ABORT = 516;
constexpr int OFF_PROG = 520;     // CTA1: pages made ready by the helper warps (paces the L2 prefetch)
constexpr int OFF_MX = 1024;       // CTA0: f32 [2][128] exchange between the two warp halves
constexpr int OFF_STAT_M = 2048;   // CTA1: f32 [128] final running max (log2 units)
constexpr int OFF_STAT_L = 2560;   // CTA1: f32 [128] row sum of the bf16-rounded P (normalises O)
constexpr int OFF_STAT_LT = 3072;  // CTA1: f32 [128] row sum of the unrounded P (gives the LSE)

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 256;  // CTA0: Q latent in columns [0, 256), S in [256, 512)
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 256, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, false, true);
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kBarMax = 1, kBarOr = 2, kBarHalf0 = 3;  // named barriers of the softmax warps
constexpr uint32_t kBarStage0 = 5;                          // [2] one per softmax half: P staged
constexpr uint32_t kBarEpi = 4;                             // named barrier of CTA 1's helper warps
constexpr int kEpiPanelBytes = 128 * 128;                   // 128 rows x 128 B output tile
constexpr int kPrefetchAhead = 8;  // pages (two groups) between the helpers' progress and the page prefetched into L2

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_sm103_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap kvh_map,
                        const __grid_constant__ CUtensorMap q_map,
                        const __grid_constant__ CUtensorMap o_map, const __grid_constant__ CUtensorMap p_map,
                        const DecodeArgs p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    if (sbase & 1023u) {  // the swizzled layouts need 1024-byte aligned tiles; never expected
        if (tid == 0 && p.dev_status) atomicOr(p.dev_status, MLA_DEV_WAIT_TIMEOUT);
        return;  // both CTAs of the cluster see the same alignment and leave together
    }
    const int unit = (int)(blockIdx.x >> 1);
    // The first split of a row starts at page 0 whatever the row's length, so the K producer
    // fetches the first group's block-table entries while the length is still on its way
    // (validated once the page count is known).
    int blk_early[kPPG] = {-1, -1, -1, -1};
    const bool early_blocks = p.plan_units == nullptr && p.qsl == nullptr && unit % p.num_splits == 0;
    if (early_blocks && tid == 0 && rank == 0) {
        const int32_t* row = p.block_table + (size_t)(unit / p.num_splits / p.Sq) * p.max_blocks;
#pragma unroll
        for (int q = 0; q < kPPG; ++q)
            if (q < p.max_blocks) blk_early[q] = ld_nc_s32(row + q);
    }
    RowGeom g{};
    if (!p.plan_units) g = row_geometry(p, unit, tid == 0 && rank == 0);  // its loads overlap the set-up
    volatile int* abort = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
    int32_t* ds = p.dev_status;
    auto bar = [&](int i) -> uint32_t { return sbase + 8u * (uint32_t)i; };

    if (tid == 0) {
        *abort = 0;
        *reinterpret_cast<volatile int*>(smem + OFF_PROG) = 0;
        for (int i = 0; i < B_COUNT; ++i) {
            uint32_t cnt = 1;
            if (i == B_SEMPTY || i == B_QREADY) cnt = 256;
            if (i >= B_READY && i < B_READY + kPBufs) cnt = 128;
            bar_init(bar(i), cnt);
        }
        if (rank == 1)  // P buffers armed for their first message before CTA 0 can send one
            for (int b = 0; b < kPBufs; ++b) bar_arrive_expect_tx(bar(B_PFULL + b), kPMsgBytes);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(sbase + OFF_TMEM, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // both CTAs' barriers exist before any remote arrive or copy
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);
    if (tid == 0) griddep_launch_dependents();
    if (p.plan_units) {
        // The schedule is the preceding kernel's output: the set-up above overlapped it.
        // Clusters past its unit count leave together (both CTAs read the same count).
        griddep_wait();
        if (unit >= *p.plan_count) {
            if (warp == 0) tmem_dealloc(tmem, kTmemCols);
            cluster_sync();
            return;
        }
        g = row_geometry(p, unit, tid == 0 && rank == 0);
    }
    const int npages = g.npages;
    const int ngroups = (npages + kPPG - 1) / kPPG;

    if (rank == 0) {
        // ============================== scores CTA ==============================
        if (warp == 0) {
            if (lane == 0 && npages > 0) {
                tma_prefetch_desc(&kv_map);
                // The K panels go out before the preceding kernel (which may be writing q) has
                // finished: no kernel of this library writes the cache. CTA 1 prefetches the
                // pages into L2 ahead of these loads, with plain prefetch instructions: bulk
                // prefetches issued here would queue in this SM's TMA unit, the narrow point of
                // the K stream.
                const int oob = (int)(p.num_blocks * kPage);  // one past the cache: TMA fills zeros
                int issued = 0;  // K panels issued
                bool ok = true;
                for (int gi = 0; gi < ngroups && ok; ++gi) {
                    int y[kPPG];
                    const int np = min(kPPG, npages - kPPG * gi);
                    for (int q = 0; q < np; ++q) {
                        int blk;
                        if (gi == 0 && early_blocks) {  // the entry fetched early: same checks as page_block
                            blk = blk_early[q];
                            if (blk < 0 || (int64_t)blk >= p.num_blocks) {
                                if (p.dev_status) atomicOr(p.dev_status, MLA_DEV_BAD_BLOCK_ID);
                                blk = -1;
                            }
                        } else {
                            blk = page_block(p, g.b, g.page0 + kPPG * gi + q);
                        }
                        y[q] = blk < 0 ? oob : blk * kPage;
                    }
                    for (int pn = 0; pn < 9; ++pn) {
                        const int m = 9 * gi + pn, slot = m % kSlots, k = m / kSlots;
                        // first use of slots 2-3: Q's panels have been moved out to TMEM
                        ok = k > 0      ? wait_bar(bar(B_SLOTEMPTY + slot), (k - 1) & 1, abort, ds)
                             : slot >= 2 ? wait_bar(bar(B_QREADY), 0, abort, ds)
                                         : true;
                        if (!ok) break;
                        const uint32_t full = bar(B_SLOTFULL + slot);
                        const uint32_t dst = sbase + OFF_RING + slot * kSlotBytes;
                        bar_arrive_expect_tx(full, np * kPageBox);
                        for (int q = 0; q < np; ++q) tma_load_2d(dst + q * kPageBox, &kv_map, full, pn * 64, y[q]);
                        ++issued;
                    }
                }
                if (*abort) {  // let the copies in flight land before the CTA can exit
                    volatile int dummy = 0;
                    for (int m = (issued > kSlots ? issued - kSlots : 0); m < issued; ++m) {
                        dummy = 0;
                        wait_bar(bar(B_SLOTFULL + m % kSlots), (m / kSlots) & 1, &dummy, nullptr);
                    }
                }
            }
        } else if (warp == 1) {
            if (lane == 0 && npages > 0) {
                // Q, the preceding kernel's output, is loaded from here so that it goes out at
                // once, in parallel with the producer's block-table reads and first K panels.
                tma_prefetch_desc(&q_map);
                griddep_wait();
                bar_arrive_expect_tx(bar(B_QFULL), 9 * kQPanelBytes);
                for (int qn = 0; qn < 8; ++qn)
                    tma_load_2d(sbase + q_panel_off(qn), &q_map, bar(B_QFULL), qn * 64, g.r * p.H);
                tma_load_2d(sbase + OFF_QROPE, &q_map, bar(B_QFULL), 8 * 64, g.r * p.H);
                int done = 0;
                bool ok = wait_bar(bar(B_QREADY), 0, abort, ds);
                if (ok) tc_fence_after();
                for (int gi = 0; gi < ngroups && ok; ++gi) {
                    if (gi > 0) {  // the softmax warps have read the previous S out of TMEM
                        if (!(ok = wait_bar(bar(B_SEMPTY), (gi - 1) & 1, abort, ds))) break;
                        tc_fence_after();
                    }
                    const uint32_t d = tmem + kSCol;
                    for (int pn = 0; pn < 9; ++pn) {
                        const int m = 9 * gi + pn, slot = m % kSlots, k = m / kSlots;
                        // TMA-written operands are ordered by the barrier itself: no tcgen05 fence
                        if (!(ok = wait_bar(bar(B_SLOTFULL + slot), k & 1, abort, ds))) break;
                        const uint32_t kb = sbase + OFF_RING + slot * kSlotBytes;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint64_t bd = smem_desc_sw128(kb + 32 * j, 16, 1024);
                            if (pn < 8) {
                                mma_ts(d, tmem + 8u * (4 * pn + j), bd, kIdescQK, (pn | j) ? 1u : 0u);
                            } else {
                                const uint64_t ad = smem_desc_sw128(sbase + OFF_QROPE + 32 * j, 16, 1024);
                                mma_ss(d, ad, bd, kIdescQK, 1u);
                            }
                        }
                        mma_commit(bar(B_SLOTEMPTY + slot));
                        ++done;
                    }
                    if (ok) mma_commit(bar(B_SFULL));
                }
                volatile int dummy = 0;  // drain: the last commits have landed before teardown
                for (int m = (done > kSlots ? done - kSlots : 0); m < done; ++m) {
                    dummy = 0;
                    wait_bar(bar(B_SLOTEMPTY + m % kSlots), (m / kSlots) & 1, &dummy, nullptr);
                }
                if (*abort) {  // and Q has landed
                    dummy = 0;
                    wait_bar(bar(B_QFULL), 0, &dummy, nullptr);
                }
            }
        } else {
            // ------------------------- softmax warps (256 threads) -------------------------
            const int half = (warp - 2) >> 2;            // pages 2 half, 2 half + 1 of each group
            const int row = 32 * (warp & 3) + lane;      // head
            const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
            const bool live = row < p.H;
            float* mx = reinterpret_cast<float*>(smem + OFF_MX);
            if (npages > 0) {
                // Q latent dims: this half moves panels 4 half .. 4 half + 3 into TMEM
                const bool okq = warp_wait(bar(B_QFULL), 0, abort, ds);
#pragma unroll 1
                for (int pn = 4 * half; pn < 4 * half + 4; ++pn) {
                    uint32_t v[32];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 x = make_uint4(0, 0, 0, 0);
                        if (live && okq)
                            x = *reinterpret_cast<const uint4*>(smem + q_panel_off(pn) + row * 128 +
                                                                ((c ^ (row & 7)) << 4));
                        v[4 * c] = x.x;
                        v[4 * c + 1] = x.y;
                        v[4 * c + 2] = x.z;
                        v[4 * c + 3] = x.w;
                    }
                    tmem_st32(tmem + lane_base + 32u * pn, v);
                }
                if (!live && half == 0) {  // heads past H: zero rope rows too (S rows stay finite)
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        *reinterpret_cast<uint4*>(smem + OFF_QROPE + row * 128 + c * 16) = make_uint4(0, 0, 0, 0);
                    fence_proxy_async_cta();
                }
                tmem_wait_st();
                tc_fence_before();
                bar_arrive(bar(B_QREADY));
            }
            const float sl2 = p.scale * 1.4426950408889634f;  // exp2 domain
            // l sums P as the PV MMA sees it (bf16) so that o = P V / l stays consistent when one
            // token dominates; lt sums the unrounded P for the LSE. Each half keeps its own sums
            // (same running max); they are added at the end.
            float m_run = -CUDART_INF_F, l_run = 0.f, lt_run = 0.f;
            const uint32_t pbuf_remote = map_to_rank(sbase + OFF_PB, 1);
            const uint32_t pfull_remote = map_to_rank(bar(B_PFULL), 1);
            for (int gi = 0; gi < ngroups; ++gi) {
                // No early exit from this loop: all 256 threads must pass the same named barriers
                // (which cannot time out); after an abort the waits return at once and the work
                // is skipped.
                const bool okS = warp_wait(bar(B_SFULL), gi & 1, abort, ds);
                uint32_t s[4][32];
                if (okS) {
                    tc_fence_after();
                    const uint32_t scol = tmem + lane_base + kSCol + 128u * half;
#pragma unroll
                    for (int c = 0; c < 4; ++c) tmem_ld32(scol + 32u * c, s[c]);
                    tmem_wait_ld();
                    tc_fence_before();
                    bar_arrive(bar(B_SEMPTY));
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int j = 0; j < 32; ++j) s[c][j] = __float_as_uint(-CUDART_INF_F);
                }
                const int pg0 = kPPG * gi + 2 * half;  // first of this half's two pages
                const int valid0 = valid_rows(g, pg0), valid1 = valid_rows(g, pg0 + 1);
                float lm = -CUDART_INF_F;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int v = c < 2 ? valid0 - 32 * c : valid1 - 32 * (c - 2);
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (j >= v) s[c][j] = __float_as_uint(-CUDART_INF_F);
                        lm = fmaxf(lm, __uint_as_float(s[c][j]));
                    }
                }
                mx[half * 128 + row] = lm;
                named_bar(kBarMax, 256);
                const float mt = fmaxf(lm, mx[(1 - half) * 128 + row]) * sl2;  // scale > 0
                const bool resc = mt > m_run + kRescaleThreshold;
                float alpha = 1.f;
                if (resc) {
                    alpha = fast_exp2(m_run - mt);  // 0 on the first group (m_run = -inf)
                    m_run = mt;
                }
                l_run *= alpha;
                lt_run *= alpha;
                // does any row of this group move its max (then CTA 1 rescales O first); the
                // barrier also keeps the next group's writes of mx behind this group's reads
                const bool any = named_bar_or(kBarOr, 256, resc && gi > 0);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int page = pg0 + q;
                    uint32_t pk[32];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float a0 = fast_exp2(fmaf(__uint_as_float(s[2 * q][2 * c]), sl2, -m_run));
                        const float a1 = fast_exp2(fmaf(__uint_as_float(s[2 * q][2 * c + 1]), sl2, -m_run));
                        const float b0 = fast_exp2(fmaf(__uint_as_float(s[2 * q + 1][2 * c]), sl2, -m_run));
                        const float b1 = fast_exp2(fmaf(__uint_as_float(s[2 * q + 1][2 * c + 1]), sl2, -m_run));
                        pk[c] = pack_bf16x2(a0, a1);
                        pk[16 + c] = pack_bf16x2(b0, b1);
                        lt_run += (a0 + a1) + (b0 + b1);
                        l_run += (bf16_lo_f(pk[c]) + bf16_hi_f(pk[c])) +
                                 (bf16_lo_f(pk[16 + c]) + bf16_hi_f(pk[16 + c]));
                    }
                    {
                        // staging buffer sbi takes page sbi of every group; it is free again once
                        // the previous group's copy out of it has landed in CTA 1
                        const int sbi = 2 * half + q;
                        const int htid = tid - 64 - 128 * half;
                        uint8_t* stage = smem + OFF_STAGE + sbi * kPBufStride;
                        if (page < npages) {  // pages past the end send nothing and leave the buffer alone
                            if (gi > 0) warp_wait<true>(bar(B_STAGEFREE + sbi), (gi - 1) & 1, abort, ds);
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                *reinterpret_cast<uint4*>(stage + row * 128 + ((c ^ (row & 7)) << 4)) =
                                    make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                            // every page carries the group's rescale factors; the group's first
                            // page also carries the flag that tells CTA 1 to rescale O first
                            reinterpret_cast<float*>(stage + kPBytes)[row] = alpha;
                            if (row == 0)
                                *reinterpret_cast<uint32_t*>(stage + kPBytes + 512) = (half == 0 && q == 0 && any) ? 1u : 0u;
                            fence_proxy_async_cta();  // generic writes before the bulk copy reads them
                        }
                        named_bar(kBarStage0 + half, 128);
                        if (htid == 0 && page < npages && okS) {
                            // CTA 1's buffer for this page is free once the PV of the page kPBufs
                            // earlier has completed (multicast commit)
                            const int pb = page % kPBufs, up = page / kPBufs;
                            if (up == 0 || wait_bar<true>(bar(B_PEMPTY + pb), (up - 1) & 1, abort, ds))
                                bulk_copy_to_peer(pbuf_remote + pb * kPBufStride,
                                                  sbase + OFF_STAGE + sbi * kPBufStride, kPMsgBytes,
                                                  pfull_remote + 8u * pb);
                        }
                    }
                }
            }
            // combine the two halves' sums, ship the final statistics
            named_bar(kBarMax, 256);
            if (half == 1) {
                mx[row] = l_run;
                mx[128 + row] = lt_run;
            }
            named_bar(kBarMax, 256);
            if (half == 0) {
                l_run += mx[row];
                lt_run += mx[128 + row];
                st_cluster_u32(map_to_rank(sbase + OFF_STAT_M, 1) + 4u * row, __float_as_uint(m_run));
                st_cluster_u32(map_to_rank(sbase + OFF_STAT_L, 1) + 4u * row, __float_as_uint(l_run));
                st_cluster_u32(map_to_rank(sbase + OFF_STAT_LT, 1) + 4u * row, __float_as_uint(lt_run));
                named_bar(kBarHalf0, 128);
                if (tid == 64) {
                    bar_arrive_remote(bar(B_STATS), 1);
                    // nothing may still be on its way to this CTA when it exits: CTA 1's last
                    // multicast commits
                    for (int pg = (npages > kPBufs ? npages - kPBufs : 0); pg < npages; ++pg) {
                        volatile int dummy = 0;
                        wait_bar<true>(bar(B_PEMPTY + pg % kPBufs), (pg / kPBufs) & 1, *abort ? &dummy : abort, ds);
                    }
                }
            }
        }
    } else {
        // ============================== output CTA ==============================
        if (warp == 0) {
            if (lane == 0 && npages > 0) {
                tma_prefetch_desc(&kvh_map);
                // kVRows tokens x 512 dims per stage: stage hs holds rows
                // [kVRows (hs % kVPerPage), + kVRows) of page hs / kVPerPage
                int issued = 0;
                bool ok = true;
                for (int i = 0; i < npages && ok; ++i) {
                    const int blk = page_block(p, g.b, g.page0 + i);
                    const int y = blk < 0 ? (int)(p.num_blocks * kPage) : blk * kPage;  // TMA fills zeros
                    for (int hf = 0; hf < kVPerPage; ++hf) {
                        const int hs = kVPerPage * i + hf, st = hs % kVStages, kv = hs / kVStages;
                        if (kv > 0 && !(ok = wait_bar(bar(B_VEMPTY + st), (kv - 1) & 1, abort, ds))) break;
                        const uint32_t full = bar(B_VFULL + st);
                        bar_arrive_expect_tx(full, kVStageBytes);
                        const uint32_t dst = sbase + OFF_V + st * kVStageBytes;
#pragma unroll
                        for (int pn = 0; pn < 8; ++pn)
                            tma_load_2d(dst + pn * kVBox, &kvh_map, full, pn * 64, y + kVRows * hf);
                        issued = hs + 1;
                    }
                }
                if (*abort) {
                    for (int i = (issued > kVStages ? issued - kVStages : 0); i < issued; ++i) {
                        volatile int dummy = 0;
                        wait_bar(bar(B_VFULL + i % kVStages), (i / kVStages) & 1, &dummy, nullptr);
                    }
                }
            }
        } else if (warp == 1) {
            // MMA thread: per page one wait for P (PFULL) and the helpers (READY), then for each of
            // its V stages the stage's wait and its MMAs of N = 256 (K steps x 2 column halves)
            if (lane == 0) {
                int done = 0;  // V stages whose MMAs were issued
                bool ok = true;
                for (int i = 0; i < npages && ok; ++i) {
                    const int pb = i % kPBufs;
                    // V and P were written by the async proxy (TMA / bulk copy): the MMA thread
                    // observes their barriers itself; READY adds the helpers' rescale / zeroing.
                    if (!(ok = wait_bar(bar(B_PFULL + pb), (i / kPBufs) & 1, abort, ds))) break;
                    if (!(ok = wait_bar(bar(B_READY + pb), (i / kPBufs) & 1, abort, ds))) break;
                    tc_fence_after();  // after a rescale by the helper warps' tcgen05.st
                    const uint32_t pbuf = sbase + OFF_PB + pb * kPBufStride;
                    for (int hf = 0; hf < kVPerPage && ok; ++hf) {
                        const int hs = kVPerPage * i + hf, st = hs % kVStages;
                        if (!(ok = wait_bar(bar(B_VFULL + st), (hs / kVStages) & 1, abort, ds))) break;
                        const uint32_t vb = sbase + OFF_V + st * kVStageBytes;
#pragma unroll
                        for (int k = 0; k < kVRows / 16; ++k) {
                            const int kk = (kVRows / 16) * hf + k;  // K step of the page
                            const uint64_t ad = smem_desc_sw128(pbuf + kk * 32, 16, 1024);
#pragma unroll
                            for (int nh = 0; nh < 2; ++nh) {
                                const uint64_t bd = smem_desc_sw128(vb + nh * 4 * kVBox + k * 2048, kVBox, 1024);
                                mma_ss(tmem + 256u * nh, ad, bd, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                        mma_commit(bar(B_VEMPTY + st));
                        done = hs + 1;
                    }
                    if (!ok) break;
                    // P buffer pb is free again (CTA 0) and O holds page i (helper warps, CTA 1).
                    // One barrier per P buffer keeps every waiter within one phase of it: a
                    // page's P only arrives after the PV of the page kPBufs earlier completed.
                    mma_commit_multicast(bar(B_PEMPTY + pb), (uint16_t)0x3);
                }
                volatile int dummy = 0;  // drain the V-ring commits before teardown
                for (int i = (done > kVStages ? done - kVStages : 0); i < done; ++i) {
                    dummy = 0;
                    wait_bar(bar(B_VEMPTY + i % kVStages), (i / kVStages) & 1, &dummy, nullptr);
                }
            }
        } else {
            // ------------- helper warps 2-5: P / V arrival, rescale, tail zeroing -------------
            // ------------- warps 2-9: the epilogue (each warp set stages half of the panels) ----
            const int row = 32 * (warp & 3) + lane;
            const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
            const int ctid = tid - 64;  // 0..255; 0..127 are the helper warps
            const int eset = warp >= 6 ? 1 : 0;
            int pages_ready = warp >= 6 ? npages : 0;
            for (int i = 0; i < npages && warp < 6; ++i) {
                const int pb = i % kPBufs, up = i / kPBufs;
                if (!warp_wait(bar(B_PFULL + pb), up & 1, abort, ds)) break;
                if (ctid == 0) {
                    bar_arrive_expect_tx(bar(B_PFULL + pb), kPMsgBytes);  // re-arm for the next message
                    bar_arrive_remote(bar(B_STAGEFREE + (i & 3)), 0);     // CTA 0's staging buffer is free
                }
                const uint8_t* pmsg = smem + OFF_PB + pb * kPBufStride;
                const bool fix = i > 0 && *reinterpret_cast<const volatile uint32_t*>(pmsg + kPBytes + 512) != 0;
                const int valid = valid_rows(g, i);
                if (fix) {  // O must hold every earlier PV product before it is rescaled
                    if (!warp_wait(bar(B_PEMPTY + (i - 1) % kPBufs), ((i - 1) / kPBufs) & 1, abort, ds)) break;
                    tc_fence_after();
                    const float a = reinterpret_cast<const volatile float*>(pmsg + kPBytes)[row];
#pragma unroll 1
                    for (int c = 0; c < kL / 32; ++c) {
                        uint32_t v[32];
                        tmem_ld32(tmem + lane_base + 32u * c, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * a);
                        tmem_st32(tmem + lane_base + 32u * c, v);
                    }
                    tmem_wait_st();
                }
                bool vok = true;
                for (int hf = 0; hf < kVPerPage && vok; ++hf) {
                    const int hs = kVPerPage * i + hf, st = hs % kVStages;
                    if (!(vok = warp_wait(bar(B_VFULL + st), (hs / kVStages) & 1, abort, ds))) break;
                    // rows of this half past the last visible token: zero them in all 8 panels
                    const int vh = min(kVRows, max(0, valid - kVRows * hf));
                    if (vh < kVRows) {
                        const uint32_t vb = OFF_V + st * kVStageBytes;
                        const int chunks = (kVRows - vh) * 8 * 8;
                        for (int q = ctid; q < chunks; q += 128) {
                            const int rr = vh + q / 64, pn = (q / 8) % 8, cc = q % 8;
                            *reinterpret_cast<uint4*>(smem + vb + pn * kVBox + rr * 128 + cc * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                        fence_proxy_async_cta();
                    }
                }
                if (!vok) break;
                tc_fence_before();
                bar_arrive(bar(B_READY + pb));
                pages_ready = i + 1;
                if (ctid == 0) *reinterpret_cast<volatile int*>(smem + OFF_PROG) = pages_ready;
            }
            if (warp >= 6 && npages > kPPG) {
                // Warps 6-9 have nothing to do until the epilogue: they prefetch into L2 the page
                // kPrefetchAhead pages past the helpers' progress, which is about one group past
                // the page the scores CTA's K producer loads, so that its TMA loads hit L2. Plain
                // prefetch instructions, not bulk prefetches: those would queue in the TMA unit.
                // Only a hint: the loop gives up quietly if it falls behind or the unit aborts.
                const int ptid = tid - 192;
                const volatile int* prog = reinterpret_cast<const volatile int*>(smem + OFF_PROG);
                const int32_t* brow = p.block_table + (size_t)g.b * p.max_blocks + g.page0;
                int spins = 0;
                for (int t = kPPG; t < npages; ++t) {
                    bool go = true;
                    while (*prog < t - kPrefetchAhead) {
                        if (*abort || ++spins > (1 << 20)) {
                            go = false;
                            break;
                        }
                        __nanosleep(128);
                    }
                    if (!go) break;
                    const int32_t blk = brow[t];
                    if (blk < 0 || (int64_t)blk >= p.num_blocks) continue;
                    const uint8_t* page = p.cache + (size_t)blk * (kPage * kBf16RowBytes);
                    for (int l = ptid; l < kPage * kBf16RowBytes / 128; l += 128) prefetch_l2(page + 128 * l);
                }
            }
            // epilogue (outputs may still be read by the preceding kernel until it completes)
            griddep_wait();
            const bool has_o = npages > 0 && pages_ready == npages && !*abort;
            wait_bar<true>(bar(B_STATS), 0, abort, ds);
            const bool o_ok =
                has_o && wait_bar(bar(B_PEMPTY + (npages - 1) % kPBufs), ((npages - 1) / kPBufs) & 1, abort, ds);
            tc_fence_after();
            const float m = reinterpret_cast<volatile float*>(smem + OFF_STAT_M)[row];
            const float l = reinterpret_cast<volatile float*>(smem + OFF_STAT_L)[row];
            const float lt = reinterpret_cast<volatile float*>(smem + OFF_STAT_LT)[row];
            const bool use_o = __all_sync(0xffffffffu, o_ok);
            const bool empty = !use_o || !(l > 0.f);
            const float inv = empty ? 0.f : 1.f / l;
            const float lse_v = empty ? -CUDART_INF_F : (m + log2f(lt)) * 0.6931471805599453f;
            const bool live = row < p.H;
            if (live && eset == 0) {
                const float lse_out = lse_v;
                if (g.slot >= 0)
                    p.part_lse[(size_t)g.slot * p.H + row] = lse_out;
                else if (p.lse)
                    p.lse[(size_t)g.r * p.H + row] = lse_out;
            }
            // O / l leaves through TMA stores: each 128-byte-wide column panel of the 128 x 512
            // result is written to a swizzled shared tile (the V ring is idle now) and stored as
            // one box of H rows, so that global writes are whole 128-byte lines. fp32 output:
            // two rounds of eight 32-column panels; bf16: one round of eight 64-column panels.
            const bool out_f32 = g.slot >= 0 || p.o_dtype == MLA_DT_F32;
            const int rounds = out_f32 ? 2 : 1;
            const int zc = g.slot >= 0 ? g.slot : g.r;
            const CUtensorMap* omap = g.slot >= 0 ? &p_map : &o_map;
            for (int rd = 0; rd < rounds; ++rd) {
                if (rd > 0) {  // the previous round's stores have read their tiles
                    if (ctid == 0) bulk_wait_group_read<0>();
                    named_bar(kBarEpi, 256);
                }
                if (out_f32) {
                    // this warp set's four 32-column panels: all TMEM loads, one wait, the stores
                    uint32_t v[4][32];
                    if (use_o) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            tmem_ld32(tmem + lane_base + (uint32_t)(rd * 256 + (4 * eset + q) * 32), v[q]);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[q][j] = 0u;
                    }
                    if (live) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint8_t* tile = smem + OFF_V + (4 * eset + q) * kEpiPanelBytes;
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                *reinterpret_cast<uint4*>(tile + row * 128 + ((c ^ (row & 7)) << 4)) = make_uint4(
                                    __float_as_uint(__uint_as_float(v[q][4 * c]) * inv),
                                    __float_as_uint(__uint_as_float(v[q][4 * c + 1]) * inv),
                                    __float_as_uint(__uint_as_float(v[q][4 * c + 2]) * inv),
                                    __float_as_uint(__uint_as_float(v[q][4 * c + 3]) * inv));
                        }
                    }
                } else {
                    // bf16: this warp set's four 64-column panels, one at a time
#pragma unroll 1
                    for (int pl = 4 * eset; pl < 4 * eset + 4; ++pl) {
                        uint8_t* tile = smem + OFF_V + pl * kEpiPanelBytes;
                        const int col0 = pl * 64;
                        uint32_t v[2][32];
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            if (use_o) {
                                tmem_ld32(tmem + lane_base + (uint32_t)(col0 + 32 * h2), v[h2]);
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j) v[h2][j] = 0u;
                            }
                        }
                        if (use_o) tmem_wait_ld();
                        if (live) {
#pragma unroll
                            for (int c = 0; c < 8; ++c) {
                                const uint32_t* w = &v[c >> 2][8 * (c & 3)];
                                *reinterpret_cast<uint4*>(tile + row * 128 + ((c ^ (row & 7)) << 4)) = make_uint4(
                                    pack_bf16x2(__uint_as_float(w[0]) * inv, __uint_as_float(w[1]) * inv),
                                    pack_bf16x2(__uint_as_float(w[2]) * inv, __uint_as_float(w[3]) * inv),
                                    pack_bf16x2(__uint_as_float(w[4]) * inv, __uint_as_float(w[5]) * inv),
                                    pack_bf16x2(__uint_as_float(w[6]) * inv, __uint_as_float(w[7]) * inv));
                            }
                        }
                    }
                }
                fence_proxy_async_cta();
                named_bar(kBarEpi, 256);
                if (ctid == 0) {
                    const int cpp = out_f32 ? 32 : 64;  // columns per panel
                    for (int pl = 0; pl < 8; ++pl)
                        tma_store_3d(omap, sbase + OFF_V + pl * kEpiPanelBytes, rd * 256 + pl * cpp, 0, zc);
                    bulk_commit_group();
                }
            }
            if (ctid == 0) bulk_wait_group<0>();  // the stores are complete before the CTA exits
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    cluster_sync();
}

int g_attr_done[64] = {};

}  // namespace

cudaError_t launch_decode_sm103(const DecodeArgs& a, cudaStream_t s) {
    auto* kernel = decode_sm103_kernel;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !g_attr_done[dev]) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        g_attr_done[dev] = 1;
    }
    CUtensorMap kv_map, kvh_map, q_map, o_map, p_map;
    memset(&kv_map, 0, sizeof kv_map);
    memset(&kvh_map, 0, sizeof kvh_map);
    memset(&q_map, 0, sizeof q_map);
    memset(&o_map, 0, sizeof o_map);
    memset(&p_map, 0, sizeof p_map);
    const bool planned = a.plan_units != nullptr;
    const int64_t units = planned ? a.plan_max_units : (int64_t)a.rows * a.num_splits;
    {
        // final rows [row][head][512] of o_latent; one box is one 128-byte-wide column panel
        // of one row's H heads
        const bool f32 = a.o_dtype == MLA_DT_F32;
        const uint64_t es = f32 ? 4 : 2;
        const uint64_t dims[3] = {(uint64_t)kL, (uint64_t)a.H, (uint64_t)a.rows};
        const uint64_t strides[2] = {(uint64_t)kL * es, (uint64_t)a.H * kL * es};
        const uint32_t box[3] = {(uint32_t)(128 / es), (uint32_t)a.H, 1u};
        e = encode_tmap(&o_map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        a.o_latent, dims, strides, box, true);
        if (e != cudaSuccess) return e;
    }
    if (a.part_o) {
        // fp32 partial rows [slot][head][512] of the split units
        const uint64_t dims[3] = {(uint64_t)kL, (uint64_t)a.H, (uint64_t)units};
        const uint64_t strides[2] = {(uint64_t)kL * 4, (uint64_t)a.H * kL * 4};
        const uint32_t box[3] = {32u, (uint32_t)a.H, 1u};
        e = encode_tmap(&p_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.part_o, dims, strides, box, true);
        if (e != cudaSuccess) return e;
    }
    if (a.num_blocks > 0 && a.max_seq_len > 0) {
        // the cache's bf16 rows
        const uint64_t rows = (uint64_t)a.num_blocks * kPage;
        const uint64_t dims[2] = {(uint64_t)kD, rows};
        const uint64_t strides[1] = {(uint64_t)kBf16RowBytes};
        const uint32_t box[2] = {64, 64};
        e = encode_tmap(&kv_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.cache, dims,
                        strides, box, true);
        if (e != cudaSuccess) return e;
        // the same rows in boxes of kVRows tokens (CTA 1's V stages)
        const uint32_t hbox[2] = {64, (uint32_t)kVRows};
        e = encode_tmap(&kvh_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.cache, dims,
                        strides, hbox, true);
        if (e != cudaSuccess) return e;
        const uint64_t qdims[2] = {(uint64_t)kD, (uint64_t)a.rows * a.H};
        const uint32_t qbox[2] = {64, 128};
        e = encode_tmap(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, qdims, strides, qbox, true);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kernel, dim3((unsigned)(2 * units)), dim3(kThreads), kSmemBytes, s, kv_map, kvh_map, q_map, o_map,
                      p_map, a);
}

}  // namespace mla
