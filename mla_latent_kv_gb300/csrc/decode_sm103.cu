// decode_sm103.cu -- paged MLA decode over the latent cache on the 5th-generation tensor cores.
//
// What it computes ([vLLM-MLA, two-algorithms section]; [vLLM-MLA, FlashMLA section]): for one
// query row (request b, query position t) and all H <= 128 heads, MQA attention over the
// row's visible tokens [j0, j1) (one split of it), every head reading the same 576-element
// cached row:  S = scale * Q K^T,  P = softmax(S),  O = P V  with V = the first 512 dims.
//
// Design (one thread-block cluster of two CTAs per (query row, split) unit):
//   CTA 0 ("scores")  loads Q (128 heads x 576 bf16) once by TMA and keeps it resident in tensor
//                     memory, streams the row's 64-token pages through a 3-stage TMA ring (9
//                     panels of 64 dims, 128-byte swizzle), computes S = Q K^T per page with
//                     tcgen05.mma (M=128 heads, N=64 tokens, K=576, A from TMEM) into a
//                     double-buffered TMEM accumulator, and runs the fp32 online softmax (one
//                     thread per head). It writes P (bf16, already in the MMA's swizzled K-major
//                     layout) straight into CTA 1's shared memory (4 buffers deep), with the
//                     per-head rescale factors, and releases each buffer with one cluster-scope
//                     arrive.
//   CTA 1 ("output")  holds the 128 x 512 fp32 output accumulator -- all 512 TMEM columns of its
//                     SM, which is why the work is split over two SMs -- streams the same pages'
//                     first 512 dims (mostly L2 hits, 2-stage ring), and accumulates O += P V with
//                     tcgen05.mma (M=128, N=2x256, K=64, V read as an MN-major operand straight
//                     from the TMA tile). Its four other warps only act on request: rescale O,
//                     zero the V rows past the end of the last page, and the epilogue.
// Neither CTA repeats the other's tensor-core work: per page the pair issues exactly the
// algorithm's 2*128*64*(576+512) flops. The softmax rescales O lazily: the running max only moves
// (and O is rescaled) when a row's max grows by more than 2^8, which keeps every exp2 argument
// <= 8 and makes rescaling rare after the first page.
//
// Rows past the split's last visible token are masked by index (S = -inf) and, in the last
// partial page, zeroed in CTA 1's V tile so that stale or NaN bytes cannot leak through 0 * NaN.
// All waits are bounded (see sm103_ptx.cuh); on a timeout the kernel winds down and reports
// MLA_DEV_WAIT_TIMEOUT instead of hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include <cstring>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mla {

cudaError_t encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box, bool swizzle128);

namespace {

using namespace ptx;

constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 softmax / correction+epilogue
constexpr int kKStages = 3;    // CTA 0 ring of full pages (K = all 576 dims)
constexpr int kVStages = 2;    // CTA 1 ring of V (first 512 dims)
constexpr int kPBufs = 4;      // P buffers in CTA 1
constexpr int kPanelBytes = 64 * 128;          // 64 rows x 64 bf16 (one 128-byte swizzle span)
constexpr int kKStageBytes = 9 * kPanelBytes;  // 73,728
constexpr int kVStageBytes = 8 * kPanelBytes;  // 65,536
constexpr int kQPanelBytes = 128 * 128;        // 128 heads x 64 dims of Q
constexpr int kPBytes = 128 * 128;             // P: 128 heads x 64 tokens
constexpr int kCtrlBytes = 4096;
constexpr int kSmem0 = kCtrlBytes + kKStages * kKStageBytes;                     // 225,280
constexpr int kSmem1 = kCtrlBytes + kVStages * kVStageBytes + kPBufs * kPBytes;  // 200,704
constexpr int kSmemBytes = kSmem0 > kSmem1 ? kSmem0 : kSmem1;
static_assert(kSmemBytes <= 232448, "over the per-CTA shared memory limit");
static_assert(9 * kQPanelBytes <= 2 * kKStageBytes, "Q is staged in the first two K stages");

// Barrier slots (8 bytes each). Both CTAs use one layout so that a multicast commit from CTA 1
// lands on CTA 0's B_PEMPTY slot.
enum : int {
    B_KFULL = 0,     // [3] CTA0: K stage landed (TMA tx)
    B_KEMPTY = 3,    // [3] CTA0: K stage consumed by the QK MMA
    B_SFULL = 6,     // [2] CTA0: S buffer ready
    B_SEMPTY = 8,    // [2] CTA0: S buffer read by the softmax warps (128)
    B_PEMPTY = 10,   // [4] CTA0: P buffer consumed by CTA1's PV MMA (multicast commit)
    B_QFULL = 14,    // CTA0: Q tile landed in shared memory (TMA tx)
    B_QREADY = 15,   // CTA0: Q moved to TMEM, its shared memory free again (128)
    B_VFULL = 16,    // [2] CTA1: V stage landed
    B_VEMPTY = 18,   // [2] CTA1: V stage consumed
    B_PFULL = 20,    // [4] CTA1: P + rescale data written by CTA0 (one cluster-scope arrive)
    B_REQ = 24,      // CTA1: request to the helper warps (MMA thread arrives)
    B_DONE = 25,     // CTA1: request served (128)
    B_OSTEP = 26,    // CTA1: PV MMAs issued so far completed
    B_STATS = 27,    // CTA1: final row statistics written by CTA0 (one cluster-scope arrive)
    B_COUNT = 28
};
constexpr int OFF_TMEM = 256;
constexpr int OFF_ABORT = 260;
constexpr int OFF_REQ = 264;       // u32 request word (CTA1)
constexpr int OFF_FLAGS = 288;     // u32 [4]: per P buffer "some row moved its max" (CTA1)
constexpr int OFF_ALPHA = 512;     // f32 [4][128]: per P buffer, per head rescale factor (CTA1)
constexpr int OFF_STAT_M = 2560;   // f32 [128]: final running max, log2 units (CTA1)
constexpr int OFF_STAT_L = 3072;   // f32 [128]: row sum of the bf16-rounded P (normalises O)
constexpr int OFF_STAT_LT = 3584;  // f32 [128]: row sum of the unrounded P (gives the LSE)
constexpr int OFF_DATA = kCtrlBytes;
constexpr int OFF_P = OFF_DATA + kVStages * kVStageBytes;  // CTA1

// request word: bit 0 rescale, bit 1 zero tail, bit 2 end (epilogue), bit 3 "O holds data",
// bits 4-7 P buffer, bits 8-11 V stage, bits 12-19 valid rows, bit 20 OSTEP parity (end)
constexpr uint32_t REQ_FIX = 1u, REQ_TAIL = 2u, REQ_END = 4u, REQ_HAS_O = 8u;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kQCol = 0;    // CTA0: Q, 288 columns (576 bf16 per lane)
constexpr uint32_t kSCol = 384;  // CTA0: S buffer b at 384 + 64 b
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 64, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, false, true);
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kSoftmaxBar = 1;        // named barrier of the 128 softmax threads

struct RowGeom {
    int r, s, b, t, j0, j1, npages, page0;
};

__device__ __forceinline__ RowGeom row_geometry(const DecodeArgs& p, int unit, bool report) {
    RowGeom g;
    g.r = unit / p.num_splits;
    g.s = unit % p.num_splits;
    g.b = g.r / p.Sq;
    g.t = g.r % p.Sq;
    int seq = p.seq_lens[g.b];
    const int cap = p.max_blocks * kPage;
    if (seq > cap || seq > p.max_seq_len || seq < 0) {
        if (report && p.dev_status) atomicOr(p.dev_status, MLA_DEV_SEQ_TOO_LONG);
        seq = seq < 0 ? 0 : (seq > cap ? cap : seq);
    }
    int n = seq - (p.Sq - 1 - g.t);
    if (n < 0) n = 0;
    split_range(n, p.num_splits, g.s, &g.j0, &g.j1);
    g.npages = (g.j1 - g.j0 + kPage - 1) / kPage;
    g.page0 = g.j0 / kPage;
    return g;
}

// Physical first row of page `pg` of request b, or one past the cache (the TMA then fills
// zeros) if the block-table entry is out of range.
__device__ __forceinline__ int page_row(const DecodeArgs& p, int b, int pg) {
    int32_t blk = p.block_table[(size_t)b * p.max_blocks + pg];
    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
        if (p.dev_status) atomicOr(p.dev_status, MLA_DEV_BAD_BLOCK_ID);
        return (int)(p.num_blocks * kPage);
    }
    return blk * kPage;
}

template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* ds) {
    bool ok = wait_bar<kCluster>(bar, parity, abort, ds);
    return __all_sync(0xffffffffu, ok);
}

// CTA 0's K ring: Q first occupies stages 0 and 1, so page i goes to stage (i + 2) % 3 and is
// that stage's `kload`-th page.
__device__ __forceinline__ void k_slot(int i, int& st, int& kload) {
    st = (i + 2) % kKStages;
    kload = (i + 2) / kKStages - (st < 2 ? 1 : 0);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_sm103_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
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
    const RowGeom g = row_geometry(p, unit, tid == 0 && rank == 0);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
    int32_t* ds = p.dev_status;
    auto bar = [&](int i) -> uint32_t { return sbase + 8u * (uint32_t)i; };

    if (tid == 0) {
        *abort = 0;
        for (int i = 0; i < B_COUNT; ++i) {
            const bool many = (i >= B_SEMPTY && i < B_SEMPTY + 2) || i == B_QREADY || i == B_DONE;
            bar_init(bar(i), many ? 128u : 1u);
        }
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(sbase + OFF_TMEM, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // both CTAs' barriers exist before any remote arrive
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);
    const int npages = g.npages;

    if (rank == 0) {
        // ============================== scores CTA ==============================
        if (warp == 0) {
            if (lane == 0 && npages > 0) {
                tma_prefetch_desc(&q_map);
                tma_prefetch_desc(&kv_map);
                bar_arrive_expect_tx(bar(B_QFULL), 9 * kQPanelBytes);
#pragma unroll
                for (int pn = 0; pn < 9; ++pn)
                    tma_load_2d(sbase + OFF_DATA + pn * kQPanelBytes, &q_map, bar(B_QFULL), pn * 64, g.r * p.H);
                int issued = 0;
                for (int i = 0; i < npages; ++i) {
                    int st, kload;
                    k_slot(i, st, kload);
                    if (kload == 0 && st < 2) {
                        if (!wait_bar(bar(B_QREADY), 0, abort, ds)) break;  // Q region released
                    } else if (kload > 0 && !wait_bar(bar(B_KEMPTY + st), (kload - 1) & 1, abort, ds)) {
                        break;
                    }
                    const uint32_t full = bar(B_KFULL + st);
                    bar_arrive_expect_tx(full, kKStageBytes);
                    const int y = page_row(p, g.b, g.page0 + i);
                    const uint32_t dst = sbase + OFF_DATA + st * kKStageBytes;
#pragma unroll
                    for (int pn = 0; pn < 9; ++pn) tma_load_2d(dst + pn * kPanelBytes, &kv_map, full, pn * 64, y);
                    issued = i + 1;
                }
                if (*abort) {  // let the copies in flight land before the CTA can exit
                    volatile int dummy = 0;
                    wait_bar(bar(B_QFULL), 0, &dummy, nullptr);
                    for (int i = (issued > kKStages ? issued - kKStages : 0); i < issued; ++i) {
                        int st, kload;
                        k_slot(i, st, kload);
                        dummy = 0;
                        wait_bar(bar(B_KFULL + st), kload & 1, &dummy, nullptr);
                    }
                }
            }
        } else if (warp == 1) {
            if (lane == 0 && npages > 0) {
                int done = 0;
                if (wait_bar(bar(B_QREADY), 0, abort, ds)) {
                    tc_fence_after();
                    for (int i = 0; i < npages; ++i) {
                        int st, kload;
                        k_slot(i, st, kload);
                        const int sb = i & 1, us = i >> 1;
                        if (!wait_bar(bar(B_KFULL + st), kload & 1, abort, ds)) break;
                        if (us > 0 && !wait_bar(bar(B_SEMPTY + sb), (us - 1) & 1, abort, ds)) break;
                        tc_fence_after();
                        const uint32_t d = tmem + kSCol + 64u * sb;
                        const uint32_t kb = sbase + OFF_DATA + st * kKStageBytes;
#pragma unroll 4
                        for (int kk = 0; kk < kD / 16; ++kk) {
                            const uint64_t bd = smem_desc_sw128(kb + (kk >> 2) * kPanelBytes + (kk & 3) * 32, 16, 1024);
                            mma_ts(d, tmem + kQCol + 8u * kk, bd, kIdescQK, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(bar(B_SFULL + sb));
                        mma_commit(bar(B_KEMPTY + st));
                        done = i + 1;
                    }
                }
                volatile int dummy = 0;  // drain: the last commits have landed before teardown
                for (int i = (done > kKStages ? done - kKStages : 0); i < done; ++i) {
                    int st, kload;
                    k_slot(i, st, kload);
                    dummy = 0;
                    wait_bar(bar(B_KEMPTY + st), kload & 1, &dummy, nullptr);
                }
            }
        } else {
            // ------------------------------ softmax warps ------------------------------
            const int row = 32 * (warp & 3) + lane;  // head
            const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
            const bool live = row < p.H;
            if (npages > 0) {
                // Q row from the TMA tile (swizzled 16-byte chunks) into TMEM; zeros past H
                const bool okq = warp_wait(bar(B_QFULL), 0, abort, ds);
#pragma unroll 1
                for (int pn = 0; pn < 9; ++pn) {
                    uint32_t v[32];
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 x = make_uint4(0, 0, 0, 0);
                        if (live && okq)
                            x = *reinterpret_cast<const uint4*>(smem + OFF_DATA + pn * kQPanelBytes + row * 128 +
                                                                ((c ^ (row & 7)) << 4));
                        v[4 * c] = x.x;
                        v[4 * c + 1] = x.y;
                        v[4 * c + 2] = x.z;
                        v[4 * c + 3] = x.w;
                    }
                    tmem_st32(tmem + lane_base + kQCol + 32u * pn, v);
                }
                tmem_wait_st();
                tc_fence_before();
                bar_arrive(bar(B_QREADY));
            }
            const float sl2 = p.scale * 1.4426950408889634f;  // exp2 domain
            // l_run sums P exactly as the PV MMA sees it (bf16) so that o = P V / l_run stays
            // consistent when one token dominates; lt_run sums the unrounded P for the LSE.
            float m_run = -CUDART_INF_F, l_run = 0.f, lt_run = 0.f;
            const uint32_t p_remote = map_to_rank(sbase + OFF_P, 1);
            const uint32_t alpha_remote = map_to_rank(sbase + OFF_ALPHA, 1);
            const uint32_t flags_remote = map_to_rank(sbase + OFF_FLAGS, 1);
            for (int i = 0; i < npages; ++i) {
                const int sb = i & 1, us = i >> 1, pb = i % kPBufs, up = i / kPBufs;
                if (!warp_wait(bar(B_SFULL + sb), us & 1, abort, ds)) break;
                tc_fence_after();
                uint32_t s0[32], s1[32];
                tmem_ld32(tmem + lane_base + kSCol + 64u * sb, s0);
                tmem_ld32(tmem + lane_base + kSCol + 64u * sb + 32u, s1);
                tmem_wait_ld();
                tc_fence_before();
                bar_arrive(bar(B_SEMPTY + sb));
                const int valid = min(kPage, g.j1 - (g.j0 + kPage * i));
                float mt = -CUDART_INF_F;
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    if (c >= valid) s0[c] = __float_as_uint(-CUDART_INF_F);
                    if (c + 32 >= valid) s1[c] = __float_as_uint(-CUDART_INF_F);
                    mt = fmaxf(mt, fmaxf(__uint_as_float(s0[c]), __uint_as_float(s1[c])));
                }
                mt *= sl2;  // scale > 0: the max commutes with the scaling
                const bool resc = mt > m_run + kRescaleThreshold;
                float alpha = 1.f;
                if (resc) {
                    alpha = fast_exp2(m_run - mt);  // 0 on the first page (m_run = -inf)
                    m_run = mt;
                }
                uint32_t pk[32];
                float sum = 0.f, sum_t = 0.f;
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    const float a0 = fast_exp2(fmaf(__uint_as_float(s0[2 * c]), sl2, -m_run));
                    const float a1 = fast_exp2(fmaf(__uint_as_float(s0[2 * c + 1]), sl2, -m_run));
                    const float b0 = fast_exp2(fmaf(__uint_as_float(s1[2 * c]), sl2, -m_run));
                    const float b1 = fast_exp2(fmaf(__uint_as_float(s1[2 * c + 1]), sl2, -m_run));
                    pk[c] = pack_bf16x2(a0, a1);
                    pk[16 + c] = pack_bf16x2(b0, b1);
                    sum_t += (a0 + a1) + (b0 + b1);
                    sum += (bf16_lo_f(pk[c]) + bf16_hi_f(pk[c])) + (bf16_lo_f(pk[16 + c]) + bf16_hi_f(pk[16 + c]));
                }
                l_run = l_run * alpha + sum;
                lt_run = lt_run * alpha + sum_t;
                if (up > 0 && !warp_wait<true>(bar(B_PEMPTY + pb), (up - 1) & 1, abort, ds)) break;
                const uint32_t pdst = p_remote + pb * kPBytes + row * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    st_cluster_v4(pdst + ((uint32_t)(c ^ (row & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                                  pk[4 * c + 3]);
                st_cluster_u32(alpha_remote + 4u * (pb * 128 + row), __float_as_uint(alpha));
                fence_proxy_async_cluster();
                const bool any = named_bar_or(kSoftmaxBar, 128, resc && i > 0);
                if (tid == 64) {  // one cluster-scope release covers the whole group's writes
                    st_cluster_u32(flags_remote + 4u * pb, any ? 1u : 0u);
                    bar_arrive_remote(bar(B_PFULL + pb), 1);
                }
            }
            st_cluster_u32(map_to_rank(sbase + OFF_STAT_M, 1) + 4u * row, __float_as_uint(m_run));
            st_cluster_u32(map_to_rank(sbase + OFF_STAT_L, 1) + 4u * row, __float_as_uint(l_run));
            st_cluster_u32(map_to_rank(sbase + OFF_STAT_LT, 1) + 4u * row, __float_as_uint(lt_run));
            named_bar(kSoftmaxBar, 128);
            if (tid == 64) bar_arrive_remote(bar(B_STATS), 1);
            // no multicast commit may still be on its way to this CTA when it exits
            for (int i = (npages > kPBufs ? npages - kPBufs : 0); i < npages; ++i) {
                volatile int dummy = 0;
                wait_bar<true>(bar(B_PEMPTY + i % kPBufs), (i / kPBufs) & 1, *abort ? &dummy : abort, ds);
            }
        }
    } else {
        // ============================== output CTA ==============================
        if (warp == 0) {
            if (lane == 0 && npages > 0) {
                tma_prefetch_desc(&kv_map);
                int issued = 0;
                for (int i = 0; i < npages; ++i) {
                    const int st = i % kVStages, kv = i / kVStages;
                    if (kv > 0 && !wait_bar(bar(B_VEMPTY + st), (kv - 1) & 1, abort, ds)) break;
                    const uint32_t full = bar(B_VFULL + st);
                    bar_arrive_expect_tx(full, kVStageBytes);
                    const int y = page_row(p, g.b, g.page0 + i);
                    const uint32_t dst = sbase + OFF_DATA + st * kVStageBytes;
#pragma unroll
                    for (int pn = 0; pn < 8; ++pn) tma_load_2d(dst + pn * kPanelBytes, &kv_map, full, pn * 64, y);
                    issued = i + 1;
                }
                if (*abort) {
                    for (int i = (issued > kVStages ? issued - kVStages : 0); i < issued; ++i) {
                        volatile int dummy = 0;
                        wait_bar(bar(B_VFULL + i % kVStages), (i / kVStages) & 1, &dummy, nullptr);
                    }
                }
            }
        } else if (warp == 1) {
            if (lane == 0) {
                uint32_t* req_word = reinterpret_cast<uint32_t*>(smem + OFF_REQ);
                int n_req = 0, n_ostep = 0, done = 0;
                bool ok = true;
                for (int i = 0; i < npages && ok; ++i) {
                    const int st = i % kVStages, kv = i / kVStages, pb = i % kPBufs, up = i / kPBufs;
                    ok = wait_bar(bar(B_VFULL + st), kv & 1, abort, ds) &&
                         wait_bar<true>(bar(B_PFULL + pb), up & 1, abort, ds);
                    if (!ok) break;
                    const bool fix = i > 0 && reinterpret_cast<volatile uint32_t*>(smem + OFF_FLAGS)[pb] != 0;
                    const int valid = min(kPage, g.j1 - (g.j0 + kPage * i));
                    if (fix || valid < kPage) {
                        if (fix) {  // the rescale must see every earlier PV product in O
                            mma_commit(bar(B_OSTEP));
                            ok = wait_bar(bar(B_OSTEP), n_ostep & 1, abort, ds);
                            ++n_ostep;
                            if (!ok) break;
                        }
                        *reinterpret_cast<volatile uint32_t*>(req_word) =
                            (fix ? REQ_FIX : 0u) | (valid < kPage ? REQ_TAIL : 0u) | ((uint32_t)pb << 4) |
                            ((uint32_t)st << 8) | ((uint32_t)valid << 12);
                        bar_arrive(bar(B_REQ));
                        ok = wait_bar(bar(B_DONE), n_req & 1, abort, ds);
                        ++n_req;
                        if (!ok) break;
                    }
                    tc_fence_after();
                    const uint32_t vb = sbase + OFF_DATA + st * kVStageBytes;
                    const uint32_t pbuf = sbase + OFF_P + pb * kPBytes;
#pragma unroll
                    for (int kk = 0; kk < kPage / 16; ++kk) {
                        const uint64_t ad = smem_desc_sw128(pbuf + kk * 32, 16, 1024);
#pragma unroll
                        for (int nh = 0; nh < 2; ++nh) {
                            const uint64_t bd = smem_desc_sw128(vb + nh * 4 * kPanelBytes + kk * 2048, kPanelBytes, 1024);
                            mma_ss(tmem + 256u * nh, ad, bd, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    mma_commit(bar(B_VEMPTY + st));
                    mma_commit_multicast(bar(B_PEMPTY + pb), (uint16_t)0x1);
                    done = i + 1;
                }
                uint32_t end = REQ_END;
                if (done > 0) {
                    mma_commit(bar(B_OSTEP));  // completes when the last PV product is in O
                    end |= ((uint32_t)(n_ostep & 1) << 20) | (ok && done == npages ? REQ_HAS_O : 0u);
                    ++n_ostep;
                }
                *reinterpret_cast<volatile uint32_t*>(req_word) = end;
                bar_arrive(bar(B_REQ));
                volatile int dummy = 0;  // drain the V-ring commits before teardown
                for (int i = (done > kVStages ? done - kVStages : 0); i < done; ++i) {
                    dummy = 0;
                    wait_bar(bar(B_VEMPTY + i % kVStages), (i / kVStages) & 1, &dummy, nullptr);
                }
            }
        } else {
            // ------------------ helper warps: rescale, tail zeroing, epilogue ------------------
            const int row = 32 * (warp & 3) + lane;
            const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
            const int ctid = tid - 64;  // 0..127
            uint32_t req = REQ_END;
            for (int k = 0;; ++k) {
                if (!warp_wait(bar(B_REQ), k & 1, abort, ds)) {
                    req = REQ_END;
                    break;
                }
                req = *reinterpret_cast<volatile uint32_t*>(smem + OFF_REQ);
                if (req & REQ_END) break;
                const int pb = (req >> 4) & 15, st = (req >> 8) & 15, valid = (req >> 12) & 255;
                if (req & REQ_FIX) {
                    tc_fence_after();
                    const float a = reinterpret_cast<volatile float*>(smem + OFF_ALPHA)[pb * 128 + row];
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
                if (req & REQ_TAIL) {  // zero V rows [valid, 64) of all 8 panels of the stage
                    const uint32_t vb = OFF_DATA + st * kVStageBytes;
                    const int chunks = (kPage - valid) * 8 * 8;
                    for (int q = ctid; q < chunks; q += 128) {
                        const int rr = valid + q / 64, pn = (q / 8) % 8, cc = q % 8;
                        *reinterpret_cast<uint4*>(smem + vb + pn * kPanelBytes + rr * 128 + cc * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_cta();
                }
                tc_fence_before();
                bar_arrive(bar(B_DONE));
            }
            // epilogue
            const bool has_o = (req & REQ_HAS_O) != 0;
            wait_bar<true>(bar(B_STATS), 0, abort, ds);
            if (has_o) wait_bar(bar(B_OSTEP), (req >> 20) & 1, abort, ds);
            tc_fence_after();
            const float m = reinterpret_cast<volatile float*>(smem + OFF_STAT_M)[row];
            const float l = reinterpret_cast<volatile float*>(smem + OFF_STAT_L)[row];
            const float lt = reinterpret_cast<volatile float*>(smem + OFF_STAT_LT)[row];
            const bool empty = !has_o || !(l > 0.f);
            const float inv = empty ? 0.f : 1.f / l;
            const float lse_v = empty ? -CUDART_INF_F : (m + log2f(lt)) * 0.6931471805599453f;
            const bool live = row < p.H;
            float* of = nullptr;
            __nv_bfloat16* ob = nullptr;
            if (p.num_splits > 1) {
                of = p.part_o + (((size_t)g.r * p.num_splits + g.s) * p.H + row) * kL;
                if (live) p.part_lse[((size_t)g.r * p.num_splits + g.s) * p.H + row] = lse_v;
            } else {
                if (p.o_dtype == MLA_DT_F32)
                    of = (float*)p.o_latent + ((size_t)g.r * p.H + row) * kL;
                else
                    ob = (__nv_bfloat16*)p.o_latent + ((size_t)g.r * p.H + row) * kL;
                if (live && p.lse) p.lse[(size_t)g.r * p.H + row] = lse_v;
            }
#pragma unroll 1
            for (int c = 0; c < kL / 32; ++c) {
                uint32_t v[32];
                if (has_o) {
                    tmem_ld32(tmem + lane_base + 32u * c, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0u;
                }
                if (!live) continue;
                if (of) {
                    float4* dst = reinterpret_cast<float4*>(of + 32 * c);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        dst[j] = make_float4(__uint_as_float(v[4 * j]) * inv, __uint_as_float(v[4 * j + 1]) * inv,
                                             __uint_as_float(v[4 * j + 2]) * inv, __uint_as_float(v[4 * j + 3]) * inv);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(ob + 32 * c);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        dst[j] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * j]) * inv, __uint_as_float(v[8 * j + 1]) * inv),
                                            pack_bf16x2(__uint_as_float(v[8 * j + 2]) * inv, __uint_as_float(v[8 * j + 3]) * inv),
                                            pack_bf16x2(__uint_as_float(v[8 * j + 4]) * inv, __uint_as_float(v[8 * j + 5]) * inv),
                                            pack_bf16x2(__uint_as_float(v[8 * j + 6]) * inv, __uint_as_float(v[8 * j + 7]) * inv));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    cluster_sync();
}

int g_attr_done[64] = {0};

}  // namespace

cudaError_t launch_decode_sm103(const DecodeArgs& a, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !g_attr_done[dev]) {
        e = cudaFuncSetAttribute(decode_sm103_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        g_attr_done[dev] = 1;
    }
    CUtensorMap kv_map, q_map;
    memset(&kv_map, 0, sizeof kv_map);
    memset(&q_map, 0, sizeof q_map);
    if (a.num_blocks > 0 && a.max_seq_len > 0) {
        const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)a.num_blocks * kPage};
        const uint64_t strides[1] = {(uint64_t)kBf16RowBytes};
        const uint32_t box[2] = {64, 64};
        e = encode_tmap(&kv_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.cache, dims, strides, box, true);
        if (e != cudaSuccess) return e;
        const uint64_t qdims[2] = {(uint64_t)kD, (uint64_t)a.B * a.Sq * a.H};
        const uint32_t qbox[2] = {64, 128};
        e = encode_tmap(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, qdims, strides, qbox, true);
        if (e != cudaSuccess) return e;
    }
    const int64_t units = (int64_t)a.B * a.Sq * a.num_splits;
    decode_sm103_kernel<<<(unsigned)(2 * units), kThreads, kSmemBytes, s>>>(kv_map, q_map, a);
    return cudaGetLastError();
}

}  // namespace mla
