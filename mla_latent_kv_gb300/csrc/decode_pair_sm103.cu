// decode_pair_sm103.cu -- paged MLA decode over the latent cache with the tensor cores of two SMs
// working as one pair (tcgen05 cta_group::2).
//
// What it computes ([vLLM-MLA, two-algorithms section]; [vLLM-MLA, FlashMLA section]): for one
// query row (request b, query position t) and all H <= 128 heads, MQA attention over the row's
// visible tokens [j0, j1) (one split of it), every head reading the same 576-element cached row:
// S = scale * Q K^T, P = softmax(S), O = P V with V = the row's first 512 dims, plus the LSE.
//
// One thread-block cluster of two CTAs per (query row, split) unit; the pair works through the
// unit's pages four at a time (a "block" of 256 tokens, 128 per CTA). Both CTAs run the same
// program; the even CTA also issues the pair's MMAs.
//
//   Scores, transposed:  S^T[token][head] = K Q^T  as pair MMAs of M = 256 tokens (each CTA's
//                        rows are its own two pages), N = 128 heads (each CTA holds 64 heads of Q
//                        in shared memory), K = 576 in 36 steps. Each CTA's tensor memory receives
//                        its 128 tokens x all 128 heads, double-buffered.
//   Softmax:             eight warps per CTA; thread = one token x 64 heads. Block maxima and row
//                        sums are reduced across lanes (shuffles), across the four lane quarters
//                        (shared memory) and across the pair (one 512-byte exchange per block), so
//                        that both CTAs use the same running max for every head. Lazy rescale:
//                        the running max moves only when a head's max grows by more than 2^8.
//   P hand-off:          P (bf16) is written where the output MMA reads it: as the B operand
//                        P^T[token][head] of the CTA that holds the head (heads 0-63 in the even
//                        CTA, 64-127 in the odd one) -- half of each thread's row locally, half
//                        into the other CTA with st.async.
//   Output, transposed:  O^T[dim][head] += V^T P^T as pair MMAs of M = 256 dims (each CTA holds
//                        128 dims of each 256-dim half of V, streamed from L2), N = 128 heads,
//                        K = 16 tokens. Two accumulators (dims 0-255 and 256-511) of 128 columns.
//
// Tensor memory per SM: two S^T buffers (2 x 128 columns) and the two O^T accumulators (2 x 128):
// all 512 columns. Shared memory per CTA: Q half 72 KB, K ring 4 x 16 KB, V ring 3 x 16 KB,
// P^T 32 KB, control 11 KB.
//
// Per block the pair issues exactly the algorithm's 2 * 128 * 256 * (576 + 512) flops (fewer for
// a partial last page: K steps past the last visible token are skipped). Rows past the unit's
// last visible token are masked by index (S = -inf) and, in the last partial page, zeroed in the
// V tiles, so that stale or NaN bytes cannot leak through 0 * NaN. All waits are bounded (see
// sm103_ptx.cuh); on a timeout the kernel winds down and reports MLA_DEV_WAIT_TIMEOUT.
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

constexpr int kThreads = 384;  // 12 warps: 0 K/Q loads, 1 V loads, 2 QK MMAs (even CTA) or P relay
                               // (odd CTA), 3 PV MMAs and the even CTA's V tails (even CTA) or the odd
                               // CTA's V tails, 4-11 softmax + epilogue (3 warps per SM sub-partition,
                               // so up to 168 registers a thread)
constexpr int kWarpSoftmax0 = 4;
constexpr int kPPB = 4;                    // pages per block (2 per CTA)
constexpr int kBox = 64 * 128;             // one TMA box: 64 rows x 64 bf16 (8 KB)
constexpr int kKSlots = 5;                 // K ring: one 64-dim panel of this CTA's 128 tokens (16 KB)
                                           // and the same panel of this CTA's 64 heads of Q (8 KB)
constexpr int kKSlotBytes = 3 * kBox;
constexpr int kVStages = 4;                // V ring: 64 tokens x this CTA's 128 dims of one half
constexpr int kVStageBytes = 2 * kBox;
constexpr int kQPanels = 9;                // 576 dims in 64-dim panels
constexpr int kPBufs = 1;                  // P^T buffers (the PV MMAs of block b - kPBufs free one)
constexpr int kPBytes = 256 * 128;         // P^T: 256 tokens x 64 heads bf16
constexpr int kPHalfBytes = kPBytes / 2;   // the part the other CTA writes

// shared memory (the same layout in both CTAs: pair MMAs read the same offsets in each)
constexpr int OFF_TMEM = 320;
constexpr int OFF_ABORT = 324;
constexpr int OFF_FLAG = 328;      // u32 [2]: a head moved its max in this block (even CTA's PV issuer)
constexpr int OFF_INVL = 512;      // f32 [128]: 1 / l for the epilogue
constexpr int OFF_REDMAX = 1024;   // f32 [4][128]: block maxima of each lane quarter
constexpr int OFF_REDSUM = 3072;   // f32 [4][128][2]: block sums (bf16-rounded P, unrounded P)
constexpr int OFF_MUSE = 7168;     // f32 [128]: running max (log2 units) the block's P uses
constexpr int OFF_ALPHA = 7680;    // f32 [128]: rescale factor of the block
constexpr int OFF_MAXIN = 8192;    // f32 [4][128]: the other CTA's block maxima (st.async)
constexpr int OFF_LIN = 10240;     // f32 [128][2]: the other CTA's final sums (st.async)
constexpr int OFF_K = 11264;
constexpr int OFF_V = OFF_K + kKSlots * kKSlotBytes;
constexpr int OFF_P = OFF_V + kVStages * kVStageBytes;
constexpr int kSmemBytes = OFF_P + kPBufs * kPBytes;
static_assert(kSmemBytes <= 232448, "over the per-CTA shared memory limit");
static_assert(OFF_LIN + 128 * 8 <= OFF_K && OFF_INVL + 512 <= OFF_REDMAX, "control area");
static_assert(OFF_K % 1024 == 0 && OFF_V % 1024 == 0 && OFF_P % 1024 == 0,
              "128-byte-swizzled tiles need 1024-byte alignment");

enum : int {
    B_KFULL = 0,                     // [kKSlots] even CTA: both CTAs' K and Q panels of a slot landed
    B_KEMPTY = B_KFULL + kKSlots,    // [kKSlots] both: the slot's QK MMAs completed (pair commit)
    B_SFULL = B_KEMPTY + kKSlots,    // [2] both: S^T buffer written
    B_SFREE = B_SFULL + 2,           // [2] even CTA: S^T buffer read by the 16 softmax warps of the pair
    B_VFULL = B_SFREE + 2,           // [kVStages] each CTA: its V stage landed (TMA tx)
    B_VREADY = B_VFULL + kVStages,   // [kVStages] even CTA: the odd CTA's V stage ready (tail rows zeroed)
    B_VEMPTY = B_VREADY + kVStages,  // [kVStages] both: the stage's PV MMAs completed
    B_PREADY = B_VEMPTY + kVStages,  // [kPBufs] each CTA: its P^T buffer complete (local writers + st.async bytes)
    B_PVDONE = B_PREADY + kPBufs,    // [kPBufs] both: the PV MMAs of the block that used P^T buffer i completed
    B_MAXFULL = B_PVDONE + kPBufs,   // [4] each CTA: the other CTA's block maxima landed (st.async)
    B_CORR = B_MAXFULL + 4,          // even CTA: O^T rescaled by the 16 softmax warps of the pair
    B_LFULL = B_CORR + 1,            // each CTA: the other CTA's final sums landed
    B_COUNT = B_LFULL + 1
};
static_assert(8 * B_COUNT <= OFF_TMEM, "barriers");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;  // O^T accumulators at columns [256, 384) and [384, 512)
constexpr uint32_t kIdescQK = idesc_bf16_f32(256, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(256, 128, true, true);
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kBarA = 1, kBarB = 2, kBarC = 3;  // named barriers of the 256 softmax threads

struct UnitGeom {
    int r, b, t, j0, j1, npages, page0;
    int slot;  // partial-output slot, or -1: this unit writes the row's final output
};

__device__ __forceinline__ UnitGeom unit_geometry(const DecodeArgs& p, int unit, bool report) {
    UnitGeom g;
    if (p.plan_units) {  // device-built schedule
        const int4 u = p.plan_units[unit];
        g.r = u.x;
        g.j0 = u.y;
        g.j1 = u.z;
        g.slot = u.w;
    } else {  // uniform splits: unit = row * S + split
        const int S = p.num_splits;
        g.r = unit / S;
        split_range(visible_tokens(p, g.r, report), S, unit % S, &g.j0, &g.j1);
        g.slot = S > 1 ? unit : -1;
    }
    int q_len;
    row_request(p, g.r, &g.b, &g.t, &q_len);
    g.npages = (g.j1 - g.j0 + kPage - 1) / kPage;
    g.page0 = g.j0 / kPage;
    return g;
}

// First cache row of page `pg` of request b, or one past the cache (the TMA then fills zeros)
// if the block-table entry is out of range.
__device__ __forceinline__ int page_row(const DecodeArgs& p, int b, int pg) {
    int32_t blk = p.block_table[(size_t)b * p.max_blocks + pg];
    if (blk < 0 || (int64_t)blk >= p.num_blocks) {
        if (p.dev_status) atomicOr(p.dev_status, MLA_DEV_BAD_BLOCK_ID);
        return (int)(p.num_blocks * kPage);
    }
    return blk * kPage;
}

__device__ __forceinline__ int valid_rows(const UnitGeom& g, int page) {
    return page < g.npages ? min(kPage, g.j1 - (g.j0 + kPage * page)) : 0;
}

template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* ds) {
    bool ok = wait_bar<kCluster>(bar, parity, abort, ds);
    return __all_sync(0xffffffffu, ok);
}

struct AddOp {
    __device__ __forceinline__ float operator()(float a, float b) const { return a + b; }
};

// One step of the lane-transposing reduction: v[0 .. 2n) holds n index pairs (i, i + n); after
// the step v[0 .. n) holds index i + n (lanes with `bit` set) or i (the others), each combined
// with the partner lane's value of the same index.
template <int n, class Op>
__device__ __forceinline__ void xstep(float* v, int lane, int bit, Op op) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < n; ++i) {
        const float send = up ? v[i] : v[i + n];
        const float keep = up ? v[i + n] : v[i];
        v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, bit));
    }
}

// v[0 .. 32) of every lane (32 indices) reduced over the warp's 32 lanes: lane l ends with
// index l in v[0].
template <class Op>
__device__ __forceinline__ void xreduce32(float (&v)[32], int lane, Op op) {
    xstep<16>(v, lane, 16, op);
    xstep<8>(v, lane, 8, op);
    xstep<4>(v, lane, 4, op);
    xstep<2>(v, lane, 2, op);
    xstep<1>(v, lane, 1, op);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_pair_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                       const DecodeArgs p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const bool lead = rank == 0;
    if (sbase & 1023u) {  // the swizzled layouts need 1024-byte aligned tiles; never expected
        if (tid == 0 && p.dev_status) atomicOr(p.dev_status, MLA_DEV_WAIT_TIMEOUT);
        return;  // both CTAs of the cluster see the same alignment and leave together
    }
    const int unit = (int)(blockIdx.x >> 1);
    if (p.plan_units) {
        // the schedule is the preceding kernel's output; clusters past its unit count leave
        // together (both CTAs read the same count) before touching anything
        griddep_wait();
        if (unit >= *p.plan_count) return;
    }
    const UnitGeom g = unit_geometry(p, unit, tid == 0 && lead);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + OFF_ABORT);
    int32_t* ds = p.dev_status;
    auto bar = [&](int i) -> uint32_t { return sbase + 8u * (uint32_t)i; };
    const int npages = g.npages;
    const int nblocks = (npages + kPPB - 1) / kPPB;
    const int ntok = g.j1 - g.j0;

    if (tid == 0) {
        *abort = 0;
        for (int i = 0; i < B_COUNT; ++i) {
            uint32_t cnt = 1;
            if (i == B_SFREE || i == B_SFREE + 1 || i == B_CORR) cnt = 16;
            if (i >= B_PREADY && i < B_PREADY + kPBufs) cnt = lead ? 130 : 129;
            bar_init(bar(i), cnt);
        }
        // first phases of the barriers that count the other CTA's st.async bytes
        for (int i = 0; i < kPBufs; ++i) bar_arrive_expect_tx(bar(B_PREADY + i), kPHalfBytes);
        for (int i = 0; i < 4; ++i) bar_arrive_expect_tx(bar(B_MAXFULL + i), 128 * 4);
        bar_arrive_expect_tx(bar(B_LFULL), 128 * 8);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc_pair(sbase + OFF_TMEM, kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync();  // both CTAs' barriers exist before any remote arrive, store or copy
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + OFF_TMEM);
    if (tid == 0) griddep_launch_dependents();

    if (warp == 0) {
        // ---------------- K and Q panels (both CTAs; completion counted in the even CTA) ----------------
        // Every ring slot takes one 64-dim panel of this CTA's two pages (K) and the same panel of
        // this CTA's 64 heads of Q. Q is re-read for every block: it is small and stays in L2,
        // and not keeping it resident leaves shared memory for deeper rings.
        if (lane == 0 && npages > 0) {
            tma_prefetch_desc(&q_map);
            tma_prefetch_desc(&kv_map);
            const uint32_t kfull = map_to_rank(bar(B_KFULL), 0);
            const int oob = (int)(p.num_blocks * kPage);
            const int qy = g.r * p.H + 64 * (int)rank;
            bool ok = true;
            int issued = 0;
            for (int b = 0; b < nblocks && ok; ++b) {
                int y[2];
                for (int i = 0; i < 2; ++i) {
                    const int pg = kPPB * b + 2 * (int)rank + i;
                    y[i] = pg < npages ? page_row(p, g.b, g.page0 + pg) : oob;
                }
                for (int pn = 0; pn < kQPanels; ++pn) {
                    const int m = kQPanels * b + pn, slot = m % kKSlots, k = m / kKSlots;
                    if (k > 0 && !(ok = wait_bar<true>(bar(B_KEMPTY + slot), (k - 1) & 1, abort, ds))) break;
                    if (lead) bar_arrive_expect_tx(bar(B_KFULL + slot), 2 * kKSlotBytes);
                    const uint32_t dst = sbase + OFF_K + slot * kKSlotBytes;
                    for (int i = 0; i < 2; ++i) tma_load_2d_pair(dst + i * kBox, &kv_map, kfull + 8u * slot, pn * 64, y[i]);
                    if (m == kKSlots - 1) {
                        // Q is the preceding kernel's output: the first slots' K panels went out
                        // before the wait, their Q panels after it
                        griddep_wait();
                        for (int mm = 0; mm < kKSlots; ++mm)
                            tma_load_2d_pair(sbase + OFF_K + mm * kKSlotBytes + 2 * kBox, &q_map, kfull + 8u * mm, mm * 64, qy);
                    } else if (m >= kKSlots) {
                        tma_load_2d_pair(dst + 2 * kBox, &q_map, kfull + 8u * slot, pn * 64, qy);
                    }
                    ++issued;
                }
            }
            if (*abort && lead) {  // let the copies in flight land before the pair can exit
                for (int m = (issued > kKSlots ? issued - kKSlots : 0); m < issued; ++m) {
                    volatile int dummy = 0;
                    wait_bar<true>(bar(B_KFULL + m % kKSlots), (m / kKSlots) & 1, &dummy, nullptr);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- V loads: this CTA's 128 dims of each 256-dim half, every page ----------------
        if (lane == 0 && npages > 0) {
            int vi = 0;
            bool ok = true;
            for (int pg = 0; pg < npages && ok; ++pg) {
                const int y = page_row(p, g.b, g.page0 + pg);
                for (int a = 0; a < 2; ++a) {
                    const int st = vi % kVStages, k = vi / kVStages;
                    if (k > 0 && !(ok = wait_bar<true>(bar(B_VEMPTY + st), (k - 1) & 1, abort, ds))) break;
                    const uint32_t full = bar(B_VFULL + st);
                    bar_arrive_expect_tx(full, kVStageBytes);
                    const uint32_t dst = sbase + OFF_V + st * kVStageBytes;
                    for (int h = 0; h < 2; ++h) tma_load_2d(dst + h * kBox, &kv_map, full, 256 * a + 128 * (int)rank + 64 * h, y);
                    ++vi;
                }
            }
            if (*abort) {
                for (int i = (vi > kVStages ? vi - kVStages : 0); i < vi; ++i) {
                    volatile int dummy = 0;
                    wait_bar(bar(B_VFULL + i % kVStages), (i / kVStages) & 1, &dummy, nullptr);
                }
            }
        }
    } else if (warp == 2) {
        if (lead) {
            // ---------------- QK^T MMAs: S^T[token][head] per block, double-buffered ----------------
            if (lane == 0 && npages > 0) {
                int done = 0;
                bool ok = true;
                for (int b = 0; b < nblocks && ok; ++b) {
                    const int sb = b & 1;
                    if (b >= 2) {  // the 16 softmax warps of the pair have read S^T of block b - 2
                        if (!(ok = wait_bar<true>(bar(B_SFREE + sb), ((b - 2) >> 1) & 1, abort, ds))) break;
                        tc_fence_after();
                    }
                    const uint32_t d = tmem + 128u * sb;
                    for (int pn = 0; pn < kQPanels; ++pn) {
                        const int m = kQPanels * b + pn, slot = m % kKSlots;
                        if (!(ok = wait_bar<true>(bar(B_KFULL + slot), (m / kKSlots) & 1, abort, ds))) break;
                        const uint32_t kb = sbase + OFF_K + slot * kKSlotBytes;
                        const uint32_t qb = kb + 2 * kBox;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            mma_pair_ss(d, smem_desc_sw128(kb + 32 * j, 16, 1024), smem_desc_sw128(qb + 32 * j, 16, 1024),
                                        kIdescQK, (pn | j) ? 1u : 0u);
                        mma_pair_commit(bar(B_KEMPTY + slot));
                        ++done;
                    }
                    if (ok) mma_pair_commit(bar(B_SFULL + sb));
                }
                volatile int dummy = 0;  // the last commits have landed before teardown
                for (int m = (done > kKSlots ? done - kKSlots : 0); m < done; ++m) {
                    dummy = 0;
                    wait_bar<true>(bar(B_KEMPTY + m % kKSlots), (m / kKSlots) & 1, &dummy, nullptr);
                }
            }
        } else if (lane == 0 && npages > 0) {
            // ---------------- odd CTA: its P^T buffer is complete -> tell the even CTA ----------------
            for (int b = 0; b < nblocks; ++b) {
                const int pbi = b % kPBufs;
                if (!wait_bar<true>(bar(B_PREADY + pbi), (b / kPBufs) & 1, abort, ds)) break;
                bar_arrive_remote(bar(B_PREADY + pbi), 0);
                if (b + kPBufs < nblocks) bar_arrive_expect_tx(bar(B_PREADY + pbi), kPHalfBytes);
            }
        }
    } else if (warp == 3) {
        // zero V rows [valid, 64) of a stage that holds the unit's last, partial page (whole warp)
        auto zero_tail = [&](int st, int valid) {
            const int chunks = (kPage - valid) * 8;  // 16-byte chunks per box
            for (int q = lane; q < 2 * chunks; q += 32) {
                const int h = q / chunks, c = q % chunks;
                *reinterpret_cast<uint4*>(smem + OFF_V + st * kVStageBytes + h * kBox + valid * 128 + c * 16) =
                    make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_cta();
            __syncwarp();
        };
        if (!lead && npages > 0) {
            // ---------------- odd CTA: its V stages -> the even CTA's PV issuer ----------------
            int vi = 0;
            for (int pg = 0; pg < npages; ++pg) {
                const int valid = valid_rows(g, pg);
                for (int a = 0; a < 2; ++a, ++vi) {
                    const int st = vi % kVStages;
                    if (!warp_wait(bar(B_VFULL + st), (vi / kVStages) & 1, abort, ds)) continue;
                    if (valid < kPage) zero_tail(st, valid);
                    if (lane == 0) bar_arrive_remote(bar(B_VREADY + st), 0);
                }
            }
        } else if (lead && npages > 0) {
            // ---------------- PV MMAs: O^T[dim][head] += V^T P^T (lane 0 issues) ----------------
            int vi = 0, ncorr = 0;
            bool ok = true;
            for (int b = 0; b < nblocks && ok; ++b) {
                const int pbi = b % kPBufs;
                if (!(ok = warp_wait<true>(bar(B_PREADY + pbi), (b / kPBufs) & 1, abort, ds))) break;
                if (lane == 0 && b + kPBufs < nblocks) bar_arrive_expect_tx(bar(B_PREADY + pbi), kPHalfBytes);
                if (*reinterpret_cast<volatile uint32_t*>(smem + OFF_FLAG + 4 * (b & 1))) {
                    if (!(ok = warp_wait<true>(bar(B_CORR), ncorr & 1, abort, ds))) break;
                    ++ncorr;
                }
                const int np = min(kPPB, npages - kPPB * b);
                for (int pg = 0; pg < np && ok; ++pg) {
                    const int valid = valid_rows(g, kPPB * b + pg);
                    const int nk = (valid + 15) / 16;
                    for (int a = 0; a < 2; ++a) {
                        const int st = vi % kVStages;
                        if (!(ok = warp_wait(bar(B_VFULL + st), (vi / kVStages) & 1, abort, ds))) break;
                        if (valid < kPage) zero_tail(st, valid);
                        if (!(ok = warp_wait<true>(bar(B_VREADY + st), (vi / kVStages) & 1, abort, ds))) break;
                        if (lane == 0) {
                            tc_fence_after();
                            const uint32_t vb = sbase + OFF_V + st * kVStageBytes;
                            const uint32_t pb = sbase + OFF_P + pbi * kPBytes + pg * 64 * 128;
                            for (int kk = 0; kk < nk; ++kk)
                                mma_pair_ss(tmem + kColO + 128u * a, smem_desc_sw128(vb + kk * 2048, kBox, 1024),
                                            smem_desc_sw128(pb + kk * 2048, kBox, 1024), kIdescPV,
                                            (b | pg | kk) ? 1u : 0u);
                            mma_pair_commit(bar(B_VEMPTY + st));
                        }
                        __syncwarp();
                        ++vi;
                    }
                }
                if (ok && lane == 0) mma_pair_commit(bar(B_PVDONE + pbi));
                __syncwarp();
            }
            if (lane == 0) {
                volatile int dummy = 0;  // drain the V-ring commits before teardown
                for (int i = (vi > kVStages ? vi - kVStages : 0); i < vi; ++i) {
                    dummy = 0;
                    wait_bar<true>(bar(B_VEMPTY + i % kVStages), (i / kVStages) & 1, &dummy, nullptr);
                }
            }
        }
    } else {
        // ---------------- softmax warps 4-11 and the epilogue ----------------
        const int sw = warp - kWarpSoftmax0;       // 0..7
        const int wq = warp & 3;                   // TMEM lane quarter (tokens 32 wq .. 32 wq + 31)
        const int ch = sw >> 2;                    // heads 64 ch .. 64 ch + 63
        const int stid = tid - 32 * kWarpSoftmax0;  // 0..255
        const int tl = 32 * wq + lane;             // token of this CTA's half of the block
        const int prow = 128 * (int)rank + tl;     // its row in the P^T buffers
        const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
        const bool head_thr = stid < 128;          // owns head `stid`'s running statistics
        const int hh = stid;
        float* redmax = reinterpret_cast<float*>(smem + OFF_REDMAX);
        float* redsum = reinterpret_cast<float*>(smem + OFF_REDSUM);
        float* muse = reinterpret_cast<float*>(smem + OFF_MUSE);
        float* alpha_s = reinterpret_cast<float*>(smem + OFF_ALPHA);
        const float sl2 = p.scale * 1.4426950408889634f;  // exp2 domain
        float m_run = -CUDART_INF_F, L = 0.f, Lt = 0.f;   // head threads: max (log2 units), sums
        const uint32_t peer_maxin = map_to_rank(sbase + OFF_MAXIN, peer);
        const uint32_t peer_maxfull = map_to_rank(bar(B_MAXFULL), peer);
        const bool p_local = ch == (int)rank;  // this thread's 64 heads are held by this CTA
        const uint32_t p_row = p_local ? sbase + OFF_P + prow * 128 : map_to_rank(sbase + OFF_P + prow * 128, peer);
        const uint32_t peer_pready = map_to_rank(bar(B_PREADY), peer);

        for (int b = 0; b < nblocks; ++b) {
            // No early exit from this loop: all 256 threads must pass the same named barriers
            // (which cannot time out); after an abort the waits return at once and the work is
            // skipped. S^T stays in tensor memory for the whole block: each 32-head half is read
            // twice (for the max, then for P), which keeps 32 scores per thread in registers.
            const int sb = b & 1;
            const bool okS = warp_wait<true>(bar(B_SFULL + sb), (b >> 1) & 1, abort, ds);
            if (okS) tc_fence_after();
            const bool tvalid = kPPB * kPage * b + tl + 128 * (int)rank < ntok;
            // masking is needed only in a unit's last, partial block and when H < 128
            const bool masked = kPPB * kPage * (b + 1) > ntok || p.H < 128 || !okS;
            // scores of heads 64 ch + 32 k .. + 31: -inf past the unit's last token, 0 past H
            auto load_half = [&](int k, float (&x)[32]) {
                uint32_t v[32];
                if (okS) {
                    tmem_ld32(tmem + lane_base + 128u * sb + 64u * ch + 32u * k, v);
                    tmem_wait_ld();
                }
                if (!masked) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(v[j]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        float f = okS ? __uint_as_float(v[j]) : -CUDART_INF_F;
                        if (64 * ch + 32 * k + j >= p.H) f = 0.f;
                        x[j] = tvalid ? f : -CUDART_INF_F;
                    }
                }
            };
            // block max of each head over this CTA's 128 tokens; lane l ends with head 64 ch + 32 k + l
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                float x[32];
                load_half(k, x);
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = redux_max(x[j]);  // the same in every lane
                if (lane == 0) {
                    float4* dst = reinterpret_cast<float4*>(redmax + wq * 128 + 64 * ch + 32 * k);
#pragma unroll
                    for (int j = 0; j < 8; ++j) dst[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
                }
            }
            named_bar(kBarA, 256);
            bool moved = false;
            if (head_thr) {
                const int q4 = b & 3;
                float bm = fmaxf(fmaxf(redmax[hh], redmax[128 + hh]), fmaxf(redmax[256 + hh], redmax[384 + hh]));
                st_async_b32(peer_maxin + 4u * (128 * q4 + hh), __float_as_uint(bm), peer_maxfull + 8u * q4);
                if (wait_bar<true>(bar(B_MAXFULL + q4), (b >> 2) & 1, abort, ds))
                    bm = fmaxf(bm, reinterpret_cast<volatile float*>(smem + OFF_MAXIN)[128 * q4 + hh]);
                if (hh == 0 && b + 4 < nblocks) bar_arrive_expect_tx(bar(B_MAXFULL + q4), 128 * 4);
                const float mt = bm * sl2;  // scale > 0
                float a = 1.f;
                if (mt > m_run + kRescaleThreshold) {
                    a = fast_exp2(m_run - mt);  // 0 on the first block (m_run = -inf)
                    m_run = mt;
                    moved = b > 0;
                    L *= a;
                    Lt *= a;
                }
                muse[hh] = m_run;
                alpha_s[hh] = a;
            }
            const bool any = named_bar_or(kBarB, 256, moved);
            if (stid == 0 && lead) *reinterpret_cast<volatile uint32_t*>(smem + OFF_FLAG + 4 * (b & 1)) = any ? 1u : 0u;
            // P = exp2(S * scale * log2e - m), rounded once to bf16 for the MMA and written 16 bytes
            // (8 heads) at a time as this token's P^T row in the CTA that holds the heads; the
            // block's two sums per head (bf16-rounded P, unrounded P) reduced over the lanes
            const int pbi = b % kPBufs;
            if (b >= kPBufs)  // P^T buffer free again: the PV MMAs of block b - 2 completed
                warp_wait<true>(bar(B_PVDONE + pbi), ((b - kPBufs) / kPBufs) & 1, abort, ds);
            const bool wr = okS && !*abort;
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                float x[32];
                uint32_t pw[16];  // the bf16 P of the 32 heads, two to a word
                load_half(k, x);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float4 ma = *reinterpret_cast<const float4*>(muse + 64 * ch + 32 * k + 8 * c);
                    const float4 mb = *reinterpret_cast<const float4*>(muse + 64 * ch + 32 * k + 8 * c + 4);
                    float* y = x + 8 * c;
                    y[0] = fast_exp2(fmaf(y[0], sl2, -ma.x));
                    y[1] = fast_exp2(fmaf(y[1], sl2, -ma.y));
                    y[2] = fast_exp2(fmaf(y[2], sl2, -ma.z));
                    y[3] = fast_exp2(fmaf(y[3], sl2, -ma.w));
                    y[4] = fast_exp2(fmaf(y[4], sl2, -mb.x));
                    y[5] = fast_exp2(fmaf(y[5], sl2, -mb.y));
                    y[6] = fast_exp2(fmaf(y[6], sl2, -mb.z));
                    y[7] = fast_exp2(fmaf(y[7], sl2, -mb.w));
                    pw[4 * c] = pack_bf16x2(y[0], y[1]);
                    pw[4 * c + 1] = pack_bf16x2(y[2], y[3]);
                    pw[4 * c + 2] = pack_bf16x2(y[4], y[5]);
                    pw[4 * c + 3] = pack_bf16x2(y[6], y[7]);
                    const uint4 w = make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
                    const int cc = 4 * k + c;
                    const uint32_t off = (uint32_t)((cc ^ (prow & 7)) << 4);
                    if (wr) {
                        if (p_local)
                            *reinterpret_cast<uint4*>(smem + OFF_P + pbi * kPBytes + prow * 128 + off) = w;
                        else
                            st_async_v4(p_row + pbi * kPBytes + off, w, peer_pready + 8u * pbi);
                    }
                }
                // rounded sum: the first step moves two bf16 values per shuffle
                float r[16];
                {
                    const bool up = (lane & 16) != 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t send = up ? pw[i] : pw[i + 8];
                        const uint32_t keep = up ? pw[i + 8] : pw[i];
                        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 16);
                        r[2 * i] = bf16_lo_f(keep) + bf16_lo_f(recv);
                        r[2 * i + 1] = bf16_hi_f(keep) + bf16_hi_f(recv);
                    }
                }
                xstep<8>(r, lane, 8, AddOp());
                xstep<4>(r, lane, 4, AddOp());
                xstep<2>(r, lane, 2, AddOp());
                xstep<1>(r, lane, 1, AddOp());
                xreduce32(x, lane, AddOp());
                *reinterpret_cast<float2*>(redsum + 2 * (wq * 128 + 64 * ch + 32 * k + lane)) = make_float2(r[0], x[0]);
            }
            // S^T of this block has been read for the last time
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && okS) {
                if (lead)
                    bar_arrive(bar(B_SFREE + sb));
                else
                    bar_arrive_remote(bar(B_SFREE + sb), 0);
            }
            if (wr && p_local) {
                fence_proxy_async_cta();
                bar_arrive(bar(B_PREADY + pbi));
            }
            // a head moved its max: scale its O^T column (this warp's quarter of the lanes, its
            // accumulator) before the block's PV MMAs
            if (any && okS && !*abort) {
                warp_wait<true>(bar(B_PVDONE + (b - 1) % kPBufs), ((b - 1) / kPBufs) & 1, abort, ds);
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t v[32];
                    const uint32_t col = tmem + lane_base + kColO + 128u * ch + 32u * c;
                    tmem_ld32(col, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha_s[32 * c + j]);
                    tmem_st32(col, v);
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (lead)
                        bar_arrive(bar(B_CORR));
                    else
                        bar_arrive_remote(bar(B_CORR), 0);
                }
            }
            named_bar(kBarC, 256);
            if (head_thr) {
                const float2 s0 = *reinterpret_cast<const float2*>(redsum + 2 * hh);
                const float2 s1 = *reinterpret_cast<const float2*>(redsum + 2 * (128 + hh));
                const float2 s2 = *reinterpret_cast<const float2*>(redsum + 2 * (256 + hh));
                const float2 s3 = *reinterpret_cast<const float2*>(redsum + 2 * (384 + hh));
                L += (s0.x + s1.x) + (s2.x + s3.x);
                Lt += (s0.y + s1.y) + (s2.y + s3.y);
            }
        }

        // ---------------- epilogue ----------------
        // the pair's sums: own half + the other CTA's (the same two additions in both CTAs)
        float* inv_l = reinterpret_cast<float*>(smem + OFF_INVL);
        if (head_thr) {
            float l = 0.f, lt = 0.f;
            if (nblocks > 0) {
                st_async_v2(map_to_rank(sbase + OFF_LIN + 8u * hh, peer), __float_as_uint(L), __float_as_uint(Lt),
                            map_to_rank(bar(B_LFULL), peer));
                if (wait_bar<true>(bar(B_LFULL), 0, abort, ds)) {
                    const volatile float* o = reinterpret_cast<volatile float*>(smem + OFF_LIN) + 2 * hh;
                    l = L + o[0];
                    lt = Lt + o[1];
                }
            }
            const bool empty = !(l > 0.f) || *abort;
            inv_l[hh] = empty ? 0.f : 1.f / l;
            if (lead && hh < p.H) {
                griddep_wait();  // outputs may still be read by the preceding kernel until it completes
                const float lse_v = empty ? -CUDART_INF_F : (m_run + log2f(lt)) * 0.6931471805599453f;
                if (g.slot >= 0)
                    p.part_lse[(size_t)g.slot * p.H + hh] = lse_v;
                else if (p.lse)
                    p.lse[(size_t)g.r * p.H + hh] = lse_v;
            }
        }
        named_bar(kBarA, 256);
        bool use_o = nblocks > 0 &&
                     warp_wait<true>(bar(B_PVDONE + (nblocks - 1) % kPBufs), ((nblocks - 1) / kPBufs) & 1, abort, ds);
        use_o = use_o && !*abort;
        tc_fence_after();
        griddep_wait();
        // this warp's accumulator (dims 256 ch + 128 rank + 32 wq + lane), every head
        const int dim = 256 * ch + 128 * (int)rank + 32 * wq + lane;
        const bool out_f32 = g.slot >= 0 || p.o_dtype == MLA_DT_F32;
        const size_t zr = (size_t)(g.slot >= 0 ? g.slot : g.r) * p.H;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
            uint32_t v[32];
            if (use_o) {
                tmem_ld32(tmem + lane_base + kColO + 128u * ch + 32u * c, v);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0u;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int h = 32 * c + j;
                if (h < p.H) {
                    const float o = __uint_as_float(v[j]) * inv_l[h];
                    if (g.slot >= 0)
                        p.part_o[(zr + h) * kL + dim] = o;
                    else if (out_f32)
                        reinterpret_cast<float*>(p.o_latent)[(zr + h) * kL + dim] = o;
                    else
                        reinterpret_cast<__nv_bfloat16*>(p.o_latent)[(zr + h) * kL + dim] = __float2bfloat16_rn(o);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 0) tmem_dealloc_pair(tmem, kTmemCols);
}

int g_attr_done[64] = {};

}  // namespace

cudaError_t launch_decode_pair_sm103(const DecodeArgs& a, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 64 && !g_attr_done[dev]) {
        e = cudaFuncSetAttribute(decode_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return e;
        g_attr_done[dev] = 1;
    }
    CUtensorMap kv_map, q_map;
    memset(&kv_map, 0, sizeof kv_map);
    memset(&q_map, 0, sizeof q_map);
    const int64_t units = a.plan_units ? a.plan_max_units : (int64_t)a.rows * a.num_splits;
    if (a.num_blocks > 0 && a.max_seq_len > 0) {
        const uint64_t dims[2] = {(uint64_t)kD, (uint64_t)a.num_blocks * kPage};
        const uint64_t strides[1] = {(uint64_t)kBf16RowBytes};
        const uint32_t box[2] = {64, 64};
        e = encode_tmap(&kv_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.cache, dims, strides, box, true);
        if (e != cudaSuccess) return e;
        const uint64_t qdims[2] = {(uint64_t)kD, (uint64_t)a.rows * a.H};
        e = encode_tmap(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.q, qdims, strides, box, true);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(decode_pair_kernel, dim3((unsigned)(2 * units)), dim3(kThreads), kSmemBytes, s, kv_map, q_map, a);
}

}  // namespace mla
