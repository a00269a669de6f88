// decode_fp8_sm103.cu -- paged MLA decode over the FP8 latent cache, dequantised on chip.
//
// What it computes ([vLLM-MLA, cache-shape section]: a 584-byte row holds the 576 e4m3 codes of
// one token's [kv_c || k_pe] plus its fp32 k_scale and v_scale; [vLLM-MLA, FlashMLA section]:
// the codes are widened to bf16 in shared memory before the tensor-core MMAs): for one query row
// and all H <= 128 heads,
//     S = scale * (Q . codes) * k_scale,   P = softmax(S),   O = sum_j P_j v_scale_j codes_j[:512].
// Every e4m3 value is a bf16 value, so the widened operands are exact; k_scale multiplies the
// fp32 score and v_scale the fp32 softmax weight before its one rounding to bf16, and the row sums
// that normalise O and give the LSE are of the unscaled weights.
//
// Same split as the bf16-cache kernel: one cluster of two CTAs per (query row, split) unit, CTA 0
// computing S and the softmax, CTA 1 accumulating O = P V in its 512 TMEM columns. What differs:
//   - Pages go two at a time ("groups" of 128 tokens) and S is double-buffered in TMEM (Q latent
//     in columns [0, 256), S in [256, 384) and [384, 512)), so the QK MMAs of the next group run
//     while the softmax reads the current one. The QK MMAs have N = 128.
//   - CTA 0 loads raw e4m3 rows by TMA. A 584-byte row stride cannot be tiled, so the cache is
//     viewed as 1168-byte row pairs: a 208-byte box at x = 192 t reads panel triple t (dims
//     [192 t, 192 t + 192)) of the even rows, and at x = 576 + 192 t the same dims of the odd rows
//     shifted by 8 bytes. Four converter warps widen each triple into three 128-byte swizzled bf16
//     K panels (the MMA's K-major layout) and, for the last triple, copy the scales out.
//   - CTA 1 copies whole half pages (18,688 contiguous bytes) with one bulk copy each; eight
//     converter warps widen the first 512 dims into the MN-major V tile and zero the rows past the
//     last visible token.
//   - Each softmax half stages its page of P (and the rescale factors) in its own shared memory
//     and sends it with one bulk shared-to-shared copy: per-thread remote stores would queue in
//     the same memory pipe as the converter warps' loads and stores.
// All waits are bounded; on a timeout the kernel winds down and reports MLA_DEV_WAIT_TIMEOUT.
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

// warps: 0 producer, 1 MMA; CTA 0: 2-9 softmax, 10-13 K converters;
// CTA 1: 2-5 helpers, 6-13 V converters, 2-9 epilogue
constexpr int kThreads = 448;
constexpr int kPPG = 2;                           // pages per group
constexpr int kPairBytes = 2 * kFp8RowBytes;      // 1168: one row pair of the cache
constexpr int kBoxW = 208;                        // raw box width (bytes): 192 dims + 16
constexpr int kBoxBytes = 32 * kBoxW;             // one box: 32 row pairs of one page (6,656 B)
constexpr int kRawSlotBytes = 2 * 2 * kBoxBytes;  // one triple of a group: [page][parity] boxes
constexpr int kRawSlots = 3;
constexpr int kKPanelBytes = 128 * 128;           // one 64-dim panel of a group's 128 rows, bf16
constexpr int kKSlotBytes = 3 * kKPanelBytes;     // one triple (48 KB)
constexpr int kKSlots = 2;
constexpr int kQPanelBytes = 128 * 128;           // 128 heads x 64 dims of Q
constexpr int kHalfPageBytes = 32 * kFp8RowBytes; // 18,688
constexpr int kVRawSlots = 3;
constexpr int kVRows = 32;                        // tokens per V stage (half a page)
constexpr int kVBox = kVRows * 128;               // one 64-dim panel of a V stage (4 KB)
constexpr int kVStageBytes = 8 * kVBox;           // 32 KB
constexpr int kVStages = 2;
constexpr int kPBufs = 5;                         // CTA 1 P buffers (one page each)
constexpr int kPBytes = 128 * 128;                // P page: 128 heads x 64 tokens bf16
// P + alpha[128] + flag word, padded to a multiple of 16 bytes: one bulk copy per page
constexpr int kPMsgBytes = (kPBytes + 512 + 4 + 15) / 16 * 16;
constexpr int kPBufStride = 17 * 1024;
constexpr int kCtrlBytes = 3584;                             // barriers and small arrays, last
// CTA 0 layout
constexpr int OFF_QROPE = 0;                                 // 16 KB
constexpr int OFF_KRING = OFF_QROPE + kQPanelBytes;          // 2 x 48 KB
constexpr int OFF_RAW = OFF_KRING + kKSlots * kKSlotBytes;   // 3 x 26 KB
constexpr int OFF_STAGE = OFF_RAW + kRawSlots * kRawSlotBytes;  // 2 x P message (one per half)
constexpr int OFF_CTRL = OFF_STAGE + 2 * kPMsgBytes;
constexpr int kSmem0 = OFF_CTRL + kCtrlBytes;
// CTA 1 layout (the control block sits at the same offset in both CTAs)
constexpr int OFF_V = 0;                                     // 2 x 32 KB
constexpr int OFF_VRAW = OFF_V + kVStages * kVStageBytes;    // 3 x 18,688 B
constexpr int OFF_PB = (OFF_VRAW + kVRawSlots * kHalfPageBytes + 1023) / 1024 * 1024;
constexpr int kSmem1 = OFF_PB + kPBufs * kPBufStride;
static_assert(kSmem1 <= OFF_CTRL, "CTA 1's buffers end below the control block");
constexpr int kSmemBytes = kSmem0;
static_assert(kSmemBytes <= 232448, "over the per-CTA shared memory limit");
static_assert(kPMsgBytes <= kPBufStride, "P message");
static_assert(kPairBytes % 16 == 0 && kBoxW % 16 == 0 && (576 % 16) == 0 && (192 % 16) == 0,
              "TMA: row-pair stride, box width and every box's x offset are multiples of 16 bytes");
static_assert(kHalfPageBytes % 16 == 0 && OFF_VRAW % 16 == 0, "bulk copies of half pages");
static_assert(OFF_STAGE % 1024 == 0 && kPMsgBytes % 16 == 0 && kPMsgBytes <= kPBufStride,
              "P staging: bulk copies of whole messages; Q panels 6-7 land there first");
static_assert(OFF_KRING % 1024 == 0 && OFF_RAW % 1024 == 0 && kRawSlotBytes % 1024 == 0 && OFF_PB % 1024 == 0 &&
                  kPBufStride % 1024 == 0 && kVBox % 1024 == 0 && OFF_V % 1024 == 0,
              "128-byte swizzled tiles need 1024-byte alignment");
static_assert(kBoxBytes % 128 == 0, "TMA boxes start on 128-byte boundaries");
// Q's latent panels land in the K ring (panels 0-5) and the P staging area (panels 6-7) until
// the softmax warps move them to TMEM.
static_assert(6 * kQPanelBytes == kKSlots * kKSlotBytes && 2 * kQPanelBytes <= 2 * kPMsgBytes, "Q panel homes");
// the epilogue stages its output tiles over the V ring, the raw ring and the P buffers
static_assert(OFF_V + 8 * 128 * 128 <= kSmem1, "epilogue tiles");
__device__ __forceinline__ uint32_t q_panel_off(int pn) {
    return pn < 6 ? OFF_KRING + pn * kQPanelBytes : OFF_STAGE + (pn - 6) * kQPanelBytes;
}

// Barrier slots (8 bytes each); one layout for both CTAs so that a multicast commit from CTA 1
// lands on CTA 0's B_PEMPTY slots.
enum : int {
    B_RAWFULL = 0,                       // [kRawSlots] CTA0: raw triple landed (TMA tx)
    B_RAWEMPTY = B_RAWFULL + kRawSlots,  // [kRawSlots] CTA0: raw triple widened (128 converter threads)
    B_KFULL = B_RAWEMPTY + kRawSlots,    // [kKSlots] CTA0: bf16 triple written (128 converter threads)
    B_KEMPTY = B_KFULL + kKSlots,        // [kKSlots] CTA0: bf16 triple consumed by the QK MMAs
    B_SFULL = B_KEMPTY + kKSlots,        // [2] CTA0: S buffer ready
    B_SEMPTY = B_SFULL + 2,              // [2] CTA0: S buffer read by the softmax warps (256)
    B_SCFULL = B_SEMPTY + 2,             // [2] CTA0: a group's scales written (128 converter threads)
    B_SCEMPTY = B_SCFULL + 2,            // [2] CTA0: a group's scales read (256 softmax threads)
    B_QFULL = B_SCEMPTY + 2,             // CTA0: Q landed in shared memory (TMA tx)
    B_QREADY,                            // CTA0: Q latent dims moved to TMEM (256)
    B_PEMPTY,                            // [kPBufs] both CTAs: PV MMA of the page in P buffer b completed
    B_VRAWFULL = B_PEMPTY + kPBufs,      // [kVRawSlots] CTA1: raw half page landed (bulk tx)
    B_VRAWEMPTY = B_VRAWFULL + kVRawSlots,  // [kVRawSlots] CTA1: raw half page widened (256)
    B_VFULL = B_VRAWEMPTY + kVRawSlots,  // [kVStages] CTA1: V stage written (256 converter threads)
    B_VEMPTY = B_VFULL + kVStages,       // [kVStages] CTA1: V stage consumed
    B_PFULL = B_VEMPTY + kVStages,       // [kPBufs] CTA1: P message landed (bulk copy bytes from CTA0)
    B_READY = B_PFULL + kPBufs,          // [kPBufs] CTA1: O rescaled for the page (128 helper threads)
    B_STATS = B_READY + kPBufs,          // CTA1: final row statistics written by CTA0
    B_STAGEFREE,                         // [2] CTA0: a half's last P message has landed in CTA 1
    B_COUNT = B_STAGEFREE + 2
};
static_assert(8 * B_COUNT <= 384, "barrier slots");
constexpr int OFF_TMEM = OFF_CTRL + 384;
constexpr int OFF_ABORT = OFF_CTRL + 388;
constexpr int OFF_VRAW_OK = OFF_CTRL + 392;   // CTA1: int [kVRawSlots] raw half page copied (0: bad block)
constexpr int OFF_MX = OFF_CTRL + 512;        // CTA0: f32 [2][128] exchange between the two warp halves
constexpr int OFF_KSC = OFF_CTRL + 1536;      // CTA0: f32 [2 groups][128 tokens] k_scale
constexpr int OFF_VSC = OFF_CTRL + 2560;      // CTA0: f32 [2 groups][128 tokens] v_scale
constexpr int OFF_STAT_M = OFF_CTRL + 512;    // CTA1: f32 [128] final running max (log2 units)
constexpr int OFF_STAT_L = OFF_CTRL + 1024;   // CTA1: f32 [128] row sum of P (normalises O)
constexpr int OFF_STAT_LT = OFF_CTRL + 1536;  // CTA1: f32 [128] the same sum (gives the LSE)
static_assert(OFF_VSC + 1024 <= OFF_CTRL + kCtrlBytes && OFF_VRAW_OK + 4 * kVRawSlots <= OFF_MX, "control block");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 256;  // CTA0: S buffer sb in columns [256 + 128 sb, + 128)
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, false, true);
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kBarMax = 1, kBarOr = 2, kBarHalf0 = 3;  // named barriers of the softmax warps
constexpr uint32_t kBarStage0 = 5;                          // + half: one half's P staging
constexpr uint32_t kBarEpi = 4;                             // named barrier of CTA 1's epilogue warps
constexpr int kEpiPanelBytes = 128 * 128;

// Eight e4m3 codes -> eight bf16 (exact), as one 16-byte chunk of a bf16 row.
__device__ __forceinline__ uint4 widen8(uint2 v) {
    uint4 o;
    e4m3x4_to_bf16x4(v.x, o.x, o.y);
    e4m3x4_to_bf16x4(v.y, o.z, o.w);
    return o;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_fp8_kernel(const __grid_constant__ CUtensorMap raw_map, const __grid_constant__ CUtensorMap q_map,
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
    RowGeom g{};
    if (!p.plan_units) g = row_geometry(p, unit, tid == 0 && rank == 0);  // its loads overlap the set-up
    volatile int* abort = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
    int32_t* ds = p.dev_status;
    auto bar = [&](int i) -> uint32_t { return sbase + OFF_CTRL + 8u * (uint32_t)i; };

    if (tid == 0) {
        *abort = 0;
        for (int i = 0; i < B_COUNT; ++i) {
            uint32_t cnt = 1;
            if ((i >= B_RAWEMPTY && i < B_RAWEMPTY + kRawSlots) || (i >= B_KFULL && i < B_KFULL + kKSlots) ||
                (i >= B_SCFULL && i < B_SCFULL + 2) || (i >= B_READY && i < B_READY + kPBufs))
                cnt = 128;
            if ((i >= B_SEMPTY && i < B_SEMPTY + 2) || (i >= B_SCEMPTY && i < B_SCEMPTY + 2) || i == B_QREADY ||
                (i >= B_VRAWEMPTY && i < B_VRAWEMPTY + kVRawSlots) || (i >= B_VFULL && i < B_VFULL + kVStages))
                cnt = 256;
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
    cluster_sync();  // both CTAs' barriers exist before any remote arrive or store
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
                // raw K triples: group gi, triple t -> ring slot (3 gi + t) % kRawSlots; the cache
                // is never written by this library's kernels, so the loads start before the
                // preceding kernel has finished; Q (that kernel's output) waits for it
                tma_prefetch_desc(&q_map);
                tma_prefetch_desc(&raw_map);
                bool q_issued = false;
                int issued = 0;
                bool ok = true;
                const int oob = (int)(p.num_blocks * (kPage / 2));  // first row pair past the cache
                for (int gi = 0; gi < ngroups && ok; ++gi) {
                    const int np = min(kPPG, npages - kPPG * gi);
                    int y[kPPG];
                    for (int q = 0; q < np; ++q) {
                        const int blk = page_block(p, g.b, g.page0 + kPPG * gi + q);
                        y[q] = blk < 0 ? oob : blk * (kPage / 2);  // out of range: TMA fills zeros
                    }
                    for (int t = 0; t < 3; ++t) {
                        const int m = 3 * gi + t, slot = m % kRawSlots, k = m / kRawSlots;
                        if (!q_issued && m == 2) {
                            griddep_wait();
                            bar_arrive_expect_tx(bar(B_QFULL), 9 * kQPanelBytes);
                            for (int qn = 0; qn < 8; ++qn)
                                tma_load_2d(sbase + q_panel_off(qn), &q_map, bar(B_QFULL), qn * 64, g.r * p.H);
                            tma_load_2d(sbase + OFF_QROPE, &q_map, bar(B_QFULL), 8 * 64, g.r * p.H);
                            q_issued = true;
                        }
                        if (k > 0 && !(ok = wait_bar(bar(B_RAWEMPTY + slot), (k - 1) & 1, abort, ds))) break;
                        const uint32_t full = bar(B_RAWFULL + slot);
                        const uint32_t dst = sbase + OFF_RAW + slot * kRawSlotBytes;
                        bar_arrive_expect_tx(full, np * 2 * kBoxBytes);
                        for (int q = 0; q < np; ++q) {
                            tma_load_2d(dst + (2 * q) * kBoxBytes, &raw_map, full, 192 * t, y[q]);
                            tma_load_2d(dst + (2 * q + 1) * kBoxBytes, &raw_map, full, 576 + 192 * t, y[q]);
                        }
                        ++issued;
                    }
                }
                if (*abort) {  // let the copies in flight land before the CTA can exit
                    volatile int dummy = 0;
                    if (q_issued) wait_bar(bar(B_QFULL), 0, &dummy, nullptr);
                    for (int m = (issued > kRawSlots ? issued - kRawSlots : 0); m < issued; ++m) {
                        dummy = 0;
                        wait_bar(bar(B_RAWFULL + m % kRawSlots), (m / kRawSlots) & 1, &dummy, nullptr);
                    }
                }
            }
        } else if (warp == 1) {
            if (lane == 0 && npages > 0) {
                int done = 0;  // triples whose MMAs were issued
                bool ok = wait_bar(bar(B_QREADY), 0, abort, ds);
                if (ok) tc_fence_after();
                for (int gi = 0; gi < ngroups && ok; ++gi) {
                    const int sb = gi & 1;
                    if (gi >= 2) {  // the softmax warps have read this S buffer's previous group
                        if (!(ok = wait_bar(bar(B_SEMPTY + sb), ((gi >> 1) - 1) & 1, abort, ds))) break;
                        tc_fence_after();
                    }
                    const uint32_t d = tmem + kSCol + 128u * sb;
                    for (int t = 0; t < 3; ++t) {
                        const int m = 3 * gi + t, ks = m % kKSlots;
                        // written by the converter warps (generic stores + proxy fence + arrive)
                        if (!(ok = wait_bar(bar(B_KFULL + ks), (m / kKSlots) & 1, abort, ds))) break;
                        tc_fence_after();
                        const uint32_t kb = sbase + OFF_KRING + ks * kKSlotBytes;
#pragma unroll
                        for (int i = 0; i < 3; ++i) {
                            const int pn = 3 * t + i;
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint64_t bd = smem_desc_sw128(kb + i * kKPanelBytes + 32 * j, 16, 1024);
                                if (pn < 8) {
                                    mma_ts(d, tmem + 8u * (4 * pn + j), bd, kIdescQK, (pn | j) ? 1u : 0u);
                                } else {
                                    const uint64_t ad = smem_desc_sw128(sbase + OFF_QROPE + 32 * j, 16, 1024);
                                    mma_ss(d, ad, bd, kIdescQK, 1u);
                                }
                            }
                        }
                        mma_commit(bar(B_KEMPTY + ks));
                        ++done;
                    }
                    if (ok) mma_commit(bar(B_SFULL + sb));
                }
                volatile int dummy = 0;  // drain: the last commits have landed before teardown
                for (int m = (done > kKSlots ? done - kKSlots : 0); m < done; ++m) {
                    dummy = 0;
                    wait_bar(bar(B_KEMPTY + m % kKSlots), (m / kKSlots) & 1, &dummy, nullptr);
                }
            }
        } else if (warp < 10) {
            // ------------------------- softmax warps (256 threads) -------------------------
            const int half = (warp - 2) >> 2;            // page 2 gi + half of each group
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
            // Both sums are of the unscaled weights exp(s - m): v_scale only enters P as the MMA
            // sees it. Each half keeps its own sums (same running max); they are added at the end.
            float m_run = -CUDART_INF_F, l_run = 0.f, lt_run = 0.f;
            const uint32_t pbuf_remote = map_to_rank(sbase + OFF_PB, 1);
            const uint32_t pfull_remote = map_to_rank(bar(B_PFULL), 1);
            for (int gi = 0; gi < ngroups; ++gi) {
                // No early exit from this loop: all 256 threads must pass the same named barriers
                // (which cannot time out); after an abort the waits return at once and the work
                // is skipped.
                const int sb = gi & 1;
                const bool okS = warp_wait(bar(B_SFULL + sb), (gi >> 1) & 1, abort, ds);
                uint32_t s[2][32];
                if (okS) {
                    tc_fence_after();
                    const uint32_t scol = tmem + lane_base + kSCol + 128u * sb + 64u * half;
                    tmem_ld32(scol, s[0]);
                    tmem_ld32(scol + 32u, s[1]);
                    tmem_wait_ld();
                    tc_fence_before();
                    bar_arrive(bar(B_SEMPTY + sb));
                } else {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int j = 0; j < 32; ++j) s[c][j] = __float_as_uint(-CUDART_INF_F);
                }
                const int page = kPPG * gi + half;
                const int valid = valid_rows(g, page);
                // the group's scales (written by the converter warps with the last triple)
                const bool okSc = warp_wait(bar(B_SCFULL + sb), (gi >> 1) & 1, abort, ds);
                const float* ksc = reinterpret_cast<const float*>(smem + OFF_KSC) + 128 * sb + 64 * half;
                const float* vsc = reinterpret_cast<const float*>(smem + OFF_VSC) + 128 * sb + 64 * half;
                float lm = -CUDART_INF_F;
#pragma unroll
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        // K = e4m3 * k_scale: the scale multiplies the score (same address in
                        // every lane: a broadcast read)
                        const float4 k4 = okSc ? *reinterpret_cast<const float4*>(ksc + 32 * c + 4 * j4)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                        const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int j = 4 * j4 + u;
                            float x = __uint_as_float(s[c][j]) * kk[u];
                            if (32 * c + j >= valid) x = -CUDART_INF_F;
                            s[c][j] = __float_as_uint(x);
                            lm = fmaxf(lm, x);
                        }
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
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int j4 = 0; j4 < 8; ++j4) {
                        // V = e4m3 * v_scale: the scale multiplies the weight before its one rounding
                        const float4 v4 = okSc ? *reinterpret_cast<const float4*>(vsc + 32 * c + 4 * j4)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                        const int j = 4 * j4;
                        const float a0 = fast_exp2(fmaf(__uint_as_float(s[c][j]), sl2, -m_run));
                        const float a1 = fast_exp2(fmaf(__uint_as_float(s[c][j + 1]), sl2, -m_run));
                        const float a2 = fast_exp2(fmaf(__uint_as_float(s[c][j + 2]), sl2, -m_run));
                        const float a3 = fast_exp2(fmaf(__uint_as_float(s[c][j + 3]), sl2, -m_run));
                        pk[16 * c + 2 * j4] = pack_bf16x2(a0 * v4.x, a1 * v4.y);
                        pk[16 * c + 2 * j4 + 1] = pack_bf16x2(a2 * v4.z, a3 * v4.w);
                        const float sum = (a0 + a1) + (a2 + a3);
                        lt_run += sum;
                        l_run += sum;
                    }
                }
                bar_arrive(bar(B_SCEMPTY + sb));
                // P goes to CTA 1 as one bulk copy per page from this half's staging buffer (the
                // copy engine moves it; per-thread remote stores would queue behind the converter
                // warps' shared-memory traffic). The buffer is rewritten only after the previous
                // group's message from this half has landed (CTA 1's helpers signal it).
                const int htid = tid - 64 - 128 * half;  // 0..127 within the half
                uint8_t* stage = smem + OFF_STAGE + half * kPMsgBytes;
                if (gi > 0) warp_wait<true>(bar(B_STAGEFREE + half), (gi - 1) & 1, abort, ds);
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4*>(stage + row * 128 + ((c ^ (row & 7)) << 4)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                // every page carries the group's rescale factors; the group's first page also
                // carries the flag that tells CTA 1 to rescale O first
                reinterpret_cast<float*>(stage + kPBytes)[row] = alpha;
                if (row == 0) *reinterpret_cast<uint32_t*>(stage + kPBytes + 512) = (half == 0 && any) ? 1u : 0u;
                fence_proxy_async_cta();  // generic writes before the copy engine reads them
                named_bar(kBarStage0 + half, 128);
                if (htid == 0 && page < npages && okS) {
                    // CTA 1's buffer for this page is free once the PV of the page kPBufs earlier
                    // has completed (multicast commit)
                    const int pb = page % kPBufs, up = page / kPBufs;
                    if (up == 0 || wait_bar<true>(bar(B_PEMPTY + pb), (up - 1) & 1, abort, ds)) {
                        bulk_copy_to_peer(pbuf_remote + pb * kPBufStride, sbase + OFF_STAGE + half * kPMsgBytes,
                                          kPMsgBytes, pfull_remote + 8u * pb);
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
        } else {
            // ---------------- K converter warps 10-13 (128 threads) ----------------
            // Triple m = 3 gi + t of group gi: raw slot m % kRawSlots -> bf16 slot m % kKSlots,
            // three 64-dim panels x 128 rows (two pages) x 8 chunks of 8 dims. Rows of a page past
            // the unit's last page stay stale: their scores are masked by index.
            const int ctid = tid - 320;
            if (npages > 0) {
                bool ok = true;
                for (int gi = 0; gi < ngroups && ok; ++gi) {
                    const int np = min(kPPG, npages - kPPG * gi);
                    for (int t = 0; t < 3 && ok; ++t) {
                        const int m = 3 * gi + t, rs = m % kRawSlots, ks = m % kKSlots;
                        if (!(ok = warp_wait(bar(B_RAWFULL + rs), (m / kRawSlots) & 1, abort, ds))) break;
                        // the bf16 slot: its previous triple's MMAs have completed (the first two
                        // uses: Q's panels have been moved out to TMEM)
                        ok = m >= kKSlots ? warp_wait(bar(B_KEMPTY + ks), ((m / kKSlots) - 1) & 1, abort, ds)
                                          : warp_wait(bar(B_QREADY), 0, abort, ds);
                        if (!ok) break;
                        const uint32_t raw = sbase + OFF_RAW + rs * kRawSlotBytes;
                        const uint32_t kb = sbase + OFF_KRING + ks * kKSlotBytes;
                        // eight loads, then eight widen-and-store: the compiler cannot move a load
                        // above an earlier store to shared memory, so batching keeps loads in flight
#pragma unroll 1
                        for (int k0 = 0; k0 < 24; k0 += 8) {
                            uint2 v[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                const int item = ctid + 128 * (k0 + u);
                                const int c = item & 7, R = (item >> 3) & 127, i = item >> 10;
                                const int q = R >> 6, r = R & 63, e = r & 1, j = r >> 1;
                                // even rows start at the box's first byte, odd rows 8 bytes in
                                v[u] = q < np ? lds_u2(raw + (2 * q + e) * kBoxBytes + j * kBoxW + 8 * e + 64 * i + 8 * c)
                                              : make_uint2(0u, 0u);
                            }
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                const int item = ctid + 128 * (k0 + u);
                                const int c = item & 7, R = (item >> 3) & 127, i = item >> 10;
                                if ((R >> 6) < np) sts_u4(kb + i * kKPanelBytes + R * 128 + ((c ^ (R & 7)) << 4), widen8(v[u]));
                            }
                        }
                        if (t == 2) {
                            // the group's scales, for the softmax warps: (k_scale, v_scale) sit in the
                            // 8 bytes after the row's 576 codes. Rows past the last visible token get
                            // 0, so that a stale or NaN scale cannot reach P through 0 * NaN.
                            const int sb = gi & 1;
                            if (gi >= 2 && !(ok = warp_wait(bar(B_SCEMPTY + sb), ((gi >> 1) - 1) & 1, abort, ds)))
                                break;
                            const int q = ctid >> 6, r = ctid & 63, e = r & 1, j = r >> 1;
                            float2 sc = make_float2(0.f, 0.f);
                            if (q < np && r < valid_rows(g, kPPG * gi + q)) {
                                const uint2 w = lds_u2(raw + (2 * q + e) * kBoxBytes + j * kBoxW + 8 * e + 192);
                                sc = make_float2(__uint_as_float(w.x), __uint_as_float(w.y));
                            }
                            reinterpret_cast<float*>(smem + OFF_KSC)[128 * sb + ctid] = sc.x;
                            reinterpret_cast<float*>(smem + OFF_VSC)[128 * sb + ctid] = sc.y;
                            bar_arrive(bar(B_SCFULL + sb));
                        }
                        fence_proxy_async_cta();  // generic-proxy writes before the MMAs read them
                        bar_arrive(bar(B_KFULL + ks));
                        bar_arrive(bar(B_RAWEMPTY + rs));
                    }
                }
            }
        }
    } else {
        // ============================== output CTA ==============================
        if (warp == 0) {
            if (lane == 0 && npages > 0) {
                // raw half pages: half page hs = 2 i + hf of page i -> slot hs % kVRawSlots; a page
                // whose block-table entry is out of range is not copied (its flag tells the
                // converters to write zeros)
                int issued = 0;
                bool ok = true;
                int* raw_ok = reinterpret_cast<int*>(smem + OFF_VRAW_OK);
                for (int i = 0; i < npages && ok; ++i) {
                    const int blk = page_block(p, g.b, g.page0 + i);
                    for (int hf = 0; hf < 2; ++hf) {
                        const int hs = 2 * i + hf, slot = hs % kVRawSlots, k = hs / kVRawSlots;
                        if (k > 0 && !(ok = wait_bar(bar(B_VRAWEMPTY + slot), (k - 1) & 1, abort, ds))) break;
                        const uint32_t full = bar(B_VRAWFULL + slot);
                        raw_ok[slot] = blk >= 0;
                        if (blk >= 0) {
                            bar_arrive_expect_tx(full, kHalfPageBytes);
                            bulk_load(sbase + OFF_VRAW + slot * kHalfPageBytes,
                                      p.cache + (size_t)blk * (kPage * kFp8RowBytes) + hf * kHalfPageBytes,
                                      kHalfPageBytes, full);
                        } else {
                            bar_arrive(full);
                        }
                        issued = hs + 1;
                    }
                }
                if (*abort) {
                    for (int i = (issued > kVRawSlots ? issued - kVRawSlots : 0); i < issued; ++i) {
                        volatile int dummy = 0;
                        wait_bar(bar(B_VRAWFULL + i % kVRawSlots), (i / kVRawSlots) & 1, &dummy, nullptr);
                    }
                }
            }
        } else if (warp == 1) {
            // MMA thread: per page one wait for P (PFULL) and the helpers (READY), then for each of
            // its two V stages the stage's wait and its MMAs of N = 256 (K steps x 2 column halves)
            if (lane == 0) {
                int done = 0;  // V stages whose MMAs were issued
                bool ok = true;
                for (int i = 0; i < npages && ok; ++i) {
                    const int pb = i % kPBufs;
                    if (!(ok = wait_bar(bar(B_PFULL + pb), (i / kPBufs) & 1, abort, ds))) break;
                    if (!(ok = wait_bar(bar(B_READY + pb), (i / kPBufs) & 1, abort, ds))) break;
                    tc_fence_after();  // after a rescale by the helper warps' tcgen05.st
                    const uint32_t pbuf = sbase + OFF_PB + pb * kPBufStride;
                    for (int hf = 0; hf < 2 && ok; ++hf) {
                        const int hs = 2 * i + hf, st = hs % kVStages;
                        if (!(ok = wait_bar(bar(B_VFULL + st), (hs / kVStages) & 1, abort, ds))) break;
                        tc_fence_after();  // V was written by the converter warps
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
                    // P buffer pb is free again (CTA 0) and O holds page i (helper warps, CTA 1)
                    mma_commit_multicast(bar(B_PEMPTY + pb), (uint16_t)0x3);
                }
                volatile int dummy = 0;  // drain the V-ring commits before teardown
                for (int i = (done > kVStages ? done - kVStages : 0); i < done; ++i) {
                    dummy = 0;
                    wait_bar(bar(B_VEMPTY + i % kVStages), (i / kVStages) & 1, &dummy, nullptr);
                }
            }
        } else {
            const int row = 32 * (warp & 3) + lane;
            const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
            int pages_ready = warp >= 6 ? npages : 0;
            if (warp < 6) {
                // ------------- helper warps 2-5: re-arm the P buffers, rescale O -------------
                const int ctid = tid - 64;  // 0..127
                for (int i = 0; i < npages; ++i) {
                    const int pb = i % kPBufs, up = i / kPBufs;
                    if (!warp_wait(bar(B_PFULL + pb), up & 1, abort, ds)) break;
                    if (ctid == 0) {
                        bar_arrive_expect_tx(bar(B_PFULL + pb), kPMsgBytes);  // the next message
                        bar_arrive_remote(bar(B_STAGEFREE + (i & 1)), 0);   // CTA 0 may restage
                    }
                    const uint8_t* pmsg = smem + OFF_PB + pb * kPBufStride;
                    const bool fix = i > 0 && *reinterpret_cast<const volatile uint32_t*>(pmsg + kPBytes + 512) != 0;
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
                    tc_fence_before();
                    bar_arrive(bar(B_READY + pb));
                    pages_ready = i + 1;
                }
            } else {
                // ------------- V converter warps 6-13 (256 threads) -------------
                // half page hs: raw slot hs % kVRawSlots -> V stage hs % kVStages, 32 rows x 8
                // panels x 8 chunks; rows past the last visible token (or of a page that was not
                // copied) are zero, so that stale or NaN bytes cannot leak through 0 * NaN
                const int ctid = tid - 192;  // 0..255
                const int* raw_ok = reinterpret_cast<const int*>(smem + OFF_VRAW_OK);
                bool ok = true;
                for (int i = 0; i < npages && ok; ++i) {
                    const int valid = valid_rows(g, i);
                    for (int hf = 0; hf < 2; ++hf) {
                        const int hs = 2 * i + hf, rs = hs % kVRawSlots, st = hs % kVStages;
                        if (!(ok = warp_wait(bar(B_VRAWFULL + rs), (hs / kVRawSlots) & 1, abort, ds))) break;
                        if (hs >= kVStages &&
                            !(ok = warp_wait(bar(B_VEMPTY + st), ((hs / kVStages) - 1) & 1, abort, ds)))
                            break;
                        const bool copied = *reinterpret_cast<const volatile int*>(raw_ok + rs) != 0;
                        const uint32_t raw = sbase + OFF_VRAW + rs * kHalfPageBytes;
                        const uint32_t vb = sbase + OFF_V + st * kVStageBytes;
                        // all eight loads first (see the K converters)
                        uint2 v[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int item = ctid + 256 * k;
                            const int c = item & 7, pn = (item >> 3) & 7, r = item >> 6;
                            v[k] = copied && kVRows * hf + r < valid ? lds_u2(raw + r * kFp8RowBytes + 64 * pn + 8 * c)
                                                                     : make_uint2(0u, 0u);
                        }
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int item = ctid + 256 * k;
                            const int c = item & 7, pn = (item >> 3) & 7, r = item >> 6;
                            sts_u4(vb + pn * kVBox + r * 128 + ((c ^ (r & 7)) << 4), widen8(v[k]));
                        }
                        fence_proxy_async_cta();  // generic-proxy writes before the MMAs read them
                        bar_arrive(bar(B_VFULL + st));
                        bar_arrive(bar(B_VRAWEMPTY + rs));
                    }
                }
            }
            if (warp < 10) {
                // ------------- epilogue, warps 2-9 (each warp set stages half of the panels) -------------
                const int etid = tid - 64;  // 0..255
                const int eset = warp >= 6 ? 1 : 0;
                // outputs may still be read by the preceding kernel until it completes
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
                    if (g.slot >= 0)
                        p.part_lse[(size_t)g.slot * p.H + row] = lse_v;
                    else if (p.lse)
                        p.lse[(size_t)g.r * p.H + row] = lse_v;
                }
                // O / l leaves through TMA stores: each 128-byte-wide column panel of the 128 x 512
                // result is written to a swizzled shared tile (the rings are idle now) and stored as
                // one box of H rows. fp32 output: two rounds of eight 32-column panels; bf16: one
                // round of eight 64-column panels.
                const bool out_f32 = g.slot >= 0 || p.o_dtype == MLA_DT_F32;
                const int rounds = out_f32 ? 2 : 1;
                const int zc = g.slot >= 0 ? g.slot : g.r;
                const CUtensorMap* omap = g.slot >= 0 ? &p_map : &o_map;
                for (int rd = 0; rd < rounds; ++rd) {
                    if (rd > 0) {  // the previous round's stores have read their tiles
                        if (etid == 0) bulk_wait_group_read<0>();
                        named_bar(kBarEpi, 256);
                    }
                    if (out_f32) {
                        // this warp set's four 32-column panels, two at a time (register budget)
#pragma unroll 1
                        for (int q0 = 0; q0 < 4; q0 += 2) {
                            uint32_t v[2][32];
                            if (use_o) {
#pragma unroll
                                for (int q = 0; q < 2; ++q)
                                    tmem_ld32(tmem + lane_base + (uint32_t)(rd * 256 + (4 * eset + q0 + q) * 32), v[q]);
                                tmem_wait_ld();
                            } else {
#pragma unroll
                                for (int q = 0; q < 2; ++q)
#pragma unroll
                                    for (int j = 0; j < 32; ++j) v[q][j] = 0u;
                            }
                            if (live) {
#pragma unroll
                                for (int q = 0; q < 2; ++q) {
                                    uint8_t* tile = smem + OFF_V + (4 * eset + q0 + q) * kEpiPanelBytes;
#pragma unroll
                                    for (int c = 0; c < 8; ++c)
                                        *reinterpret_cast<uint4*>(tile + row * 128 + ((c ^ (row & 7)) << 4)) =
                                            make_uint4(__float_as_uint(__uint_as_float(v[q][4 * c]) * inv),
                                                       __float_as_uint(__uint_as_float(v[q][4 * c + 1]) * inv),
                                                       __float_as_uint(__uint_as_float(v[q][4 * c + 2]) * inv),
                                                       __float_as_uint(__uint_as_float(v[q][4 * c + 3]) * inv));
                                }
                            }
                        }
                    } else {
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
                    if (etid == 0) {
                        const int cpp = out_f32 ? 32 : 64;  // columns per panel
                        for (int pl = 0; pl < 8; ++pl)
                            tma_store_3d(omap, sbase + OFF_V + pl * kEpiPanelBytes, rd * 256 + pl * cpp, 0, zc);
                        bulk_commit_group();
                    }
                }
                if (etid == 0) bulk_wait_group<0>();  // the stores are complete before the CTA exits
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    cluster_sync();
}

int g_attr_done[64] = {};

}  // namespace

cudaError_t launch_decode_fp8_sm103(const DecodeArgs& a, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !g_attr_done[dev]) {
        e = cudaFuncSetAttribute(decode_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        g_attr_done[dev] = 1;
    }
    CUtensorMap raw_map, q_map, o_map, p_map;
    memset(&raw_map, 0, sizeof raw_map);
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
        // the cache as 1168-byte row pairs (bytes), boxes of 208 bytes x 32 row pairs, unswizzled
        const uint64_t dims[2] = {(uint64_t)kPairBytes, (uint64_t)a.num_blocks * (kPage / 2)};
        const uint64_t strides[1] = {(uint64_t)kPairBytes};
        const uint32_t box[2] = {(uint32_t)kBoxW, 32u};
        e = encode_tmap(&raw_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, a.cache, dims, strides, box, false);
        if (e != cudaSuccess) return e;
        const uint64_t qdims[2] = {(uint64_t)kD, (uint64_t)a.rows * a.H};
        const uint64_t qstrides[1] = {(uint64_t)kBf16RowBytes};
        const uint32_t qbox[2] = {64, 128};
        e = encode_tmap(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, qdims, qstrides, qbox, true);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(decode_fp8_kernel, dim3((unsigned)(2 * units)), dim3(kThreads), kSmemBytes, s, raw_map, q_map,
                      o_map, p_map, a);
}

}  // namespace mla
