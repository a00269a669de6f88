// prefill_sm103.cu -- the prefill ("compute-friendly") route of MLA on the 5th-generation tensor
// cores ([vLLM-MLA, Prefill section]).
//
// A prefill request b has ctx_b tokens in the paged cache and q_b new tokens. Keys and values are
// not absorbed: every latent row c_j is up-projected per head, k_j = [c_j W_UK (128) || k_pe_j
// (64)], v_j = c_j W_UV (128), and attention is standard MHA with a 192-dim q.k and a 128-dim
// output. The route runs as segments, each one gather -> two up-projection GEMMs (gemm_sm103.cu)
// -> attention (this file):
//   1. the new tokens, attending causally among themselves; the result is written;
//   2. the context, in chunks of at most chunk_rows gathered rows; each chunk's result is merged
//      into the running one by LSE in the attention kernel's epilogue (merge_attn_states).
//
// Attention kernel: one CTA per (128-query tile, request, head), 384 threads, 1 CTA per SM.
//   warp 8 lane 0   TMA: the q tile (three 64-dim panels); per 128-key tile the K panels (k_nope
//                   dims 0-63 and 64-127 of this head, k_pe shared by all heads) into a 2-stage ring
//   warp 10 lane 0  TMA: per 128-key tile the two V panels into another 2-stage ring
//   warp 9 lane 0   tcgen05.mma: S_j = Q K_j^T (M = 128 queries, N = 128 keys, K = 192, both
//                   operands in shared memory) into one of three 128-column TMEM buffers
//   warp 11 lane 0  tcgen05.mma: O += P_j V_j (P read from TMEM over S, V an MN-major operand in
//                   shared memory); two issuing threads, so that one's waits leave the pipe busy
//                   with the other's MMAs
//   warps 0-7       softmax, two warps per TMEM lane quarter (one query row per lane, 64 key
//                   columns per warp): fp32 online softmax in the exp2 domain with a lazily moved
//                   running max (O and l are rescaled only when a row's max grows by more than
//                   2^8); P goes back over S as bf16; at the end O / l and the LSE, merged with
//                   the result of the earlier segments
// FP8 cache: the gathered rows hold the e4m3 values unscaled; k_scale multiplies the key's logit
// column and v_scale its P column, which is exact because the up-projection is linear.
// TMEM: S buffers at columns 0, 128 and 256, O at 384..511. Every wait is bounded.
#include <cuda.h>
#include <math_constants.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mla {

cudaError_t encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                        bool swizzle128);

namespace {

using namespace ptx;

// ---------------------------------------------------------------- context prefix sums
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kScanThreads)
    cu_ctx_kernel(const int32_t* __restrict__ ctx_lens, int B, int32_t cap, int32_t* __restrict__ cu,
                  int32_t* dev_status) {
    if (threadIdx.x == 0) griddep_launch_dependents();
    griddep_wait();
    __shared__ int32_t part[kScanThreads];
    const int per = (B + kScanThreads - 1) / kScanThreads;
    const int b0 = threadIdx.x * per;
    auto len = [&](int b) {
        int32_t n = ctx_lens[b];
        if (n < 0 || n > cap) {
            if (dev_status) atomicOr(dev_status, MLA_DEV_SEQ_TOO_LONG);
            n = n < 0 ? 0 : cap;
        }
        return n;
    };
    int32_t sum = 0;
    for (int b = b0; b < b0 + per && b < B; ++b) sum += len(b);
    part[threadIdx.x] = sum;
    __syncthreads();
    for (int off = 1; off < kScanThreads; off <<= 1) {  // inclusive scan
        const int32_t v = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
        __syncthreads();
        part[threadIdx.x] += v;
        __syncthreads();
    }
    int32_t run = threadIdx.x > 0 ? part[threadIdx.x - 1] : 0;
    for (int b = b0; b < b0 + per && b < B; ++b) {
        cu[b] = run;
        run += len(b);
    }
    if (threadIdx.x == kScanThreads - 1) cu[B] = part[kScanThreads - 1];
}

// ---------------------------------------------------------------- gather
// One warp per row: 64 16-byte chunks of latent and 8 of rope (bf16), or 72 8-byte chunks of e4m3
// widened to bf16 plus the row's two scales.
constexpr int kGatherWarps = 8;

__global__ void __launch_bounds__(kGatherWarps * 32) gather_kernel(PrefillGather g) {
    if (threadIdx.x == 0) griddep_launch_dependents();
    griddep_wait();  // the workspace may still be read by the previous segment's kernels
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * kGatherWarps + warp;
    if (i >= g.rows) return;
    uint4* const xd = reinterpret_cast<uint4*>(g.x + (int64_t)i * kL);
    uint4* const pd = reinterpret_cast<uint4*>(g.kpe + (int64_t)i * kR);
    // workspace row -> a new token's row of kv_c / k_pe, or (request, position) in the cache
    int64_t new_row = -1, pos = 0;
    int lo = 0;
    if (g.mode == kPrefillNew) {
        new_row = i;
    } else {
        // the last request whose first row is <= this row
        const int64_t gr = g.mode == kPrefillAll ? (int64_t)i : g.c0 + i;
        int hi = g.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            const int64_t first = (int64_t)g.cu_ctx[mid] + (g.mode == kPrefillAll ? g.qsl[mid] : 0);
            if (first <= gr)
                lo = mid;
            else
                hi = mid - 1;
        }
        pos = gr - g.cu_ctx[lo] - (g.mode == kPrefillAll ? g.qsl[lo] : 0);
        const int64_t ctx = g.cu_ctx[lo + 1] - g.cu_ctx[lo];
        if (g.mode == kPrefillAll && pos >= ctx) new_row = g.qsl[lo] + (pos - ctx);
    }
    if (new_row >= 0) {  // a new token's own row, unscaled
        const uint4* xs = reinterpret_cast<const uint4*>(g.kv_c + new_row * g.st_c);
        const uint4* ps = reinterpret_cast<const uint4*>(g.k_pe + new_row * g.st_pe);
        const uint4 a = xs[lane], b = xs[lane + 32];
        xd[lane] = a;
        xd[lane + 32] = b;
        if (lane < 8) pd[lane] = ps[lane];
        if (lane == 0 && g.scales) g.scales[i] = make_float2(1.f, 1.f);
        return;
    }
    const int64_t blk = g.block_table[(int64_t)lo * g.max_blocks + pos / kPage];
    if (blk < 0 || blk >= g.num_blocks) {
        if (lane == 0 && g.dev_status) atomicOr(g.dev_status, MLA_DEV_BAD_BLOCK_ID);
        xd[lane] = make_uint4(0, 0, 0, 0);
        xd[lane + 32] = make_uint4(0, 0, 0, 0);
        if (lane < 8) pd[lane] = make_uint4(0, 0, 0, 0);
        if (lane == 0 && g.scales) g.scales[i] = make_float2(0.f, 0.f);
        return;
    }
    const int64_t slot = blk * kPage + pos % kPage;
    if (g.kv_dtype == MLA_KV_BF16) {
        const uint4* src = reinterpret_cast<const uint4*>(g.cache + slot * kBf16RowBytes);
        const uint4 a = src[lane], b = src[lane + 32];
        uint4 c = make_uint4(0, 0, 0, 0);
        if (lane < 8) c = src[64 + lane];
        xd[lane] = a;
        xd[lane + 32] = b;
        if (lane < 8) pd[lane] = c;
    } else {
        const uint8_t* row = g.cache + slot * kFp8RowBytes;  // 584-byte rows are 8-byte aligned
        uint2 v[3];
#pragma unroll
        for (int k = 0; k < 3; ++k)
            if (lane + 32 * k < 72) v[k] = *reinterpret_cast<const uint2*>(row + 8 * (lane + 32 * k));
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            const int c = lane + 32 * k;
            if (c >= 72) continue;
            const uint4 o = make_uint4(e4m3x2_to_bf16x2(v[k].x & 0xffffu), e4m3x2_to_bf16x2(v[k].x >> 16),
                                       e4m3x2_to_bf16x2(v[k].y & 0xffffu), e4m3x2_to_bf16x2(v[k].y >> 16));
            if (c < 64)
                xd[c] = o;
            else
                pd[c - 64] = o;
        }
        if (lane == 0) g.scales[i] = *reinterpret_cast<const float2*>(row + kD);
    }
}

// ---------------------------------------------------------------- attention
constexpr int kAttnThreads = 384;       // warps 0-7 softmax, 8 TMA (q, K) + TMEM, 9 QK MMAs, 10 TMA (V), 11 PV MMAs
constexpr int kPanel = 128 * 128;       // 128 rows x 64 bf16 (128-byte swizzle): 16 KB
constexpr int OFF_Q = 0;                // 3 panels (the A operand of QK)
constexpr int OFF_K = 3 * kPanel;       // 2 stages x 3 panels (k_nope 0-63, 64-127, k_pe)
constexpr int OFF_V = 9 * kPanel;       // 2 stages x 2 panels
constexpr int OFF_SC = 13 * kPanel;     // FP8: 2 x 128 (k_scale, v_scale)
// row maxima of the two column halves per tile parity (2 x 2 x 128), then the row sums (2 x 128)
constexpr int OFF_MX = OFF_SC + 2 * 128 * 8;
constexpr int kAttnSmem = OFF_MX + 6 * 128 * 4 + 1024;  // + 1024-byte alignment slack
constexpr int kSBufs = 3;               // TMEM: S buffers at 0, 128, 256; O at 384
constexpr uint32_t kOCol = 384;
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 128, false, true);
constexpr uint32_t kBarScales = 1;      // named barrier of the eight softmax warps
constexpr uint32_t kBarPair0 = 2;       // 2 + q: the two softmax warps of TMEM lane quarter q
enum {
    B_Q = 0,        // q tile landed in shared memory
    B_KFULL = 1,    // 2
    B_KEMPTY = 3,   // 2
    B_VFULL = 5,    // 2
    B_VEMPTY = 7,   // 2
    B_SFULL = 9,    // 3
    B_PREADY = 12,  // 3 (256 arrivals)
    B_PVDONE = 15,  // 3
    B_FINAL = 18,     // the PV thread's MMAs have completed
    B_FINAL_QK = 19,  // the QK thread's MMAs have completed
    kNumBars = 20
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* ds) {
    const bool ok = wait_bar(bar, parity, abort, ds);
    return __all_sync(0xffffffffu, ok);
}

template <bool kFp8>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap kn_map,
                const __grid_constant__ CUtensorMap kpe_map, const __grid_constant__ CUtensorMap v_map,
                const PrefillAttn p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[kNumBars];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    if (threadIdx.x == 0) griddep_launch_dependents();
    griddep_wait();  // q, the up-projected keys and the running o / lse come from earlier kernels

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.y, h = blockIdx.z;
    const int q_begin = p.qsl[b];
    const int q_len = p.qsl[b + 1] - q_begin;
    const int r0 = blockIdx.x * 128;  // first query row of the tile, within the request
    if (r0 >= q_len) return;
    int64_t key0;  // first key row in the segment's workspace
    int n_keys;
    int shift = 0;  // causal segments: query row t sees keys [0, shift + t]
    if (p.mode == kPrefillNew) {
        key0 = q_begin;
        n_keys = min(q_len, r0 + 128);  // the tile's last row sees new tokens 0 .. r0 + 127
    } else if (p.mode == kPrefillAll) {
        shift = p.cu_ctx[b + 1] - p.cu_ctx[b];  // the request's context precedes its new tokens
        key0 = (int64_t)p.cu_ctx[b] + q_begin;
        n_keys = shift + min(q_len, r0 + 128);
    } else {
        const int64_t g0 = max(p.c0, (int64_t)p.cu_ctx[b]);
        const int64_t g1 = min(p.c1, (int64_t)p.cu_ctx[b + 1]);
        if (g1 <= g0) return;  // no context of this request in the chunk: nothing to merge
        key0 = g0 - p.c0;
        n_keys = (int)(g1 - g0);
    }
    const int n_tiles = (n_keys + 127) / 128;

    const uint32_t sbase = (smem_addr(smem_raw) + 1023u) & ~1023u;
    uint8_t* const sgen = smem_raw + (sbase - smem_addr(smem_raw));
    const uint32_t bar0 = smem_addr(&bars[0]);
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    int32_t* const ds = p.dev_status;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        bar_init(bar(B_Q), 1);
        for (int i = 0; i < 2; ++i) {
            bar_init(bar(B_KFULL + i), 1);
            bar_init(bar(B_KEMPTY + i), 1);
            bar_init(bar(B_VFULL + i), 1);
            bar_init(bar(B_VEMPTY + i), 1);
        }
        for (int i = 0; i < kSBufs; ++i) {
            bar_init(bar(B_SFULL + i), 1);
            bar_init(bar(B_PREADY + i), 256);
            bar_init(bar(B_PVDONE + i), 1);
        }
        bar_init(bar(B_FINAL), 1);
        bar_init(bar(B_FINAL_QK), 1);
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc(smem_addr(&tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int* abort = &abort_flag;

    if (warp == 8) {
        // ------------------------------------------------------------ TMA producer: q and K
        if (lane == 0) {
            tma_prefetch_desc(&q_map);
            tma_prefetch_desc(&kn_map);
            tma_prefetch_desc(&kpe_map);
            bar_arrive_expect_tx(bar(B_Q), 3 * kPanel);
            for (int pn = 0; pn < 3; ++pn)
                tma_load_3d(sbase + OFF_Q + pn * kPanel, &q_map, bar(B_Q), 64 * pn, h, q_begin + r0);
            int klast[2] = {-1, -1};
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j & 1;
                if (j >= 2 && !wait_bar(bar(B_KEMPTY + st), ((j >> 1) - 1) & 1, abort, ds)) break;
                const uint32_t dst = sbase + OFF_K + st * 3 * kPanel;
                const int z = (int)(key0 + 128 * j);
                bar_arrive_expect_tx(bar(B_KFULL + st), 3 * kPanel);
                tma_load_3d(dst, &kn_map, bar(B_KFULL + st), 0, z, h);
                tma_load_3d(dst + kPanel, &kn_map, bar(B_KFULL + st), 64, z, h);
                tma_load_2d(dst + 2 * kPanel, &kpe_map, bar(B_KFULL + st), 0, z);
                klast[st] = j;
            }
            // every copy issued has landed before the CTA can leave
            int ignore = 0;
            wait_bar(bar(B_Q), 0, &ignore, nullptr);
            for (int st = 0; st < 2; ++st) {
                ignore = 0;
                if (klast[st] >= 0) wait_bar(bar(B_KFULL + st), (klast[st] >> 1) & 1, &ignore, nullptr);
            }
        }
    } else if (warp == 10) {
        // ------------------------------------------------------------ TMA producer: V
        // A thread of its own, so that a V stage still in use never holds back the next K tile.
        if (lane == 0) {
            tma_prefetch_desc(&v_map);
            int vlast[2] = {-1, -1};
            for (int j = 0; j < n_tiles; ++j) {
                const int st = j & 1;
                if (j >= 2 && !wait_bar(bar(B_VEMPTY + st), ((j >> 1) - 1) & 1, abort, ds)) break;
                const uint32_t dst = sbase + OFF_V + st * 2 * kPanel;
                const int z = (int)(key0 + 128 * j);
                bar_arrive_expect_tx(bar(B_VFULL + st), 2 * kPanel);
                tma_load_3d(dst, &v_map, bar(B_VFULL + st), 0, z, h);
                tma_load_3d(dst + kPanel, &v_map, bar(B_VFULL + st), 64, z, h);
                vlast[st] = j;
            }
            int ignore = 0;
            for (int st = 0; st < 2; ++st) {
                ignore = 0;
                if (vlast[st] >= 0) wait_bar(bar(B_VFULL + st), (vlast[st] >> 1) & 1, &ignore, nullptr);
            }
        }
    } else if (warp == 9 || warp == 11) {
        // ------------------------------------------------------------ MMA issuers
        // Two threads issue: warp 9 the QK MMAs, warp 11 the PV MMAs. The tensor pipe queues
        // only about two MMAs behind an issuing thread, so a wait in a single issuer left the
        // pipe idle; with two, one thread's waits are covered by the other's MMAs. Each thread's
        // commits track its own MMAs, and every hazard between the two goes through a barrier:
        // PV_j needs P_j (B_PREADY, after S_j and the softmax), QK_j reuses the S buffer of tile
        // j - 3 only after PV_{j-3} (B_PVDONE), and the softmax rescales O only after PV_{j-1}.
        // QK runs up to two tiles ahead of PV, as far as the K ring and the S buffers allow.
        if (lane == 0) {
            bool ok = wait_bar(bar(B_Q), 0, abort, ds);
            if (warp == 9) {
                for (int j = 0; j < n_tiles && ok; ++j) {
                    const int st = j & 1, sb = j % kSBufs;
                    if (!(ok = wait_bar(bar(B_KFULL + st), (j >> 1) & 1, abort, ds))) break;
                    if (j >= kSBufs &&
                        !(ok = wait_bar(bar(B_PVDONE + sb), ((j - kSBufs) / kSBufs) & 1, abort, ds)))
                        break;
                    tc_fence_after();
                    const uint32_t kb = sbase + OFF_K + st * 3 * kPanel;
#pragma unroll
                    for (int pn = 0; pn < 3; ++pn)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            mma_ss(tmem + 128u * sb, smem_desc_sw128(sbase + OFF_Q + pn * kPanel + kk * 32, 16, 1024),
                                   smem_desc_sw128(kb + pn * kPanel + kk * 32, 16, 1024), kIdescQK,
                                   (pn | kk) ? 1u : 0u);
                    mma_commit(bar(B_KEMPTY + st));
                    mma_commit(bar(B_SFULL + sb));
                }
                mma_commit(bar(B_FINAL_QK));  // lands when every QK MMA issued above has completed
                int ignore = 0;
                wait_bar(bar(B_FINAL_QK), 0, &ignore, nullptr);
            } else {
                for (int i = 0; i < n_tiles && ok; ++i) {
                    const int st = i & 1, sb = i % kSBufs;
                    if (!(ok = wait_bar(bar(B_VFULL + st), (i >> 1) & 1, abort, ds))) break;
                    if (!(ok = wait_bar(bar(B_PREADY + sb), (i / kSBufs) & 1, abort, ds))) break;
                    tc_fence_after();  // P was written by the softmax warps' tcgen05.st
                    const uint32_t vb = sbase + OFF_V + st * 2 * kPanel;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // 16 keys per step: 16 rows of V, 8 columns of P
                        mma_ts(tmem + kOCol, tmem + 128u * sb + 8u * kk, smem_desc_sw128(vb + kk * 2048, kPanel, 1024),
                               kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(bar(B_VEMPTY + st));
                    mma_commit(bar(B_PVDONE + sb));
                }
                mma_commit(bar(B_FINAL));  // lands when every PV MMA issued above has completed
                int ignore = 0;
                wait_bar(bar(B_FINAL), 0, &ignore, nullptr);
            }
        }
    } else {
        // ------------------------------------------------------------ softmax (warps 0-7)
        // Warp w owns TMEM lane quarter w % 4 (32 query rows) and key columns [64 hf, 64 hf + 64)
        // of each tile, hf = w / 4; the two warps of a quarter agree on each row's max through
        // shared memory. Every named barrier below runs on every tile whatever the waits
        // returned, so that a wait that gives up cannot leave the partner warp stuck.
        const int quarter = warp & 3, hf = warp >> 2;
        const int row = 32 * quarter + lane;  // TMEM lane = query row of the tile
        const int t = r0 + row;               // query row within the request
        const uint32_t lane_base = (uint32_t)(32 * quarter) << 16;
        const uint32_t pair_bar = kBarPair0 + (uint32_t)quarter;
        const float sl2 = p.scale * 1.4426950408889634f;
        const int limit = p.mode != kPrefillChunk ? min(n_keys, shift + t + 1) : n_keys;  // keys [0, limit) visible
        float2* const sc = reinterpret_cast<float2*>(sgen + OFF_SC);
        float* const mx = reinterpret_cast<float*>(sgen + OFF_MX);  // [tile parity][hf][row]
        // running max m (exp2 domain) and the sum of this half's P relative to it
        float m = -CUDART_INF_F, lt = 0.f;
        bool alive = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int sb = j % kSBufs;
            if (kFp8) {  // the tile's key scales, staged once for the eight warps
                if (threadIdx.x < 128) {
                    const int kr = 128 * j + threadIdx.x;
                    sc[(j & 1) * 128 + threadIdx.x] = kr < n_keys ? p.scales[key0 + kr] : make_float2(0.f, 0.f);
                }
                named_bar(kBarScales, 256);
            }
            const bool ok_s = alive && warp_wait(bar(B_SFULL + sb), (j / kSBufs) & 1, abort, ds);
            uint32_t s[2][32];
            float mt = -CUDART_INF_F;
            const int kb = 128 * j + 64 * hf;  // first key of this warp's columns
            if (ok_s) {
                tc_fence_after();
                tmem_ld32(tmem + lane_base + 128u * sb + 64u * hf, s[0]);
                tmem_ld32(tmem + lane_base + 128u * sb + 64u * hf + 32u, s[1]);
                tmem_wait_ld();
                const bool masked = __any_sync(0xffffffffu, kb + 64 > limit);
                float m4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
                if (kFp8) {
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            s[c][i] = __float_as_uint(__uint_as_float(s[c][i]) * (sl2 * sc[(j & 1) * 128 + 64 * hf + 32 * c + i].x));
                }
                if (masked) {  // a tile that reaches past a row's last visible key
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (kb + 32 * c + i >= limit) s[c][i] = __float_as_uint(-CUDART_INF_F);
                }
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int i = 0; i < 32; ++i) m4[i & 3] = fmaxf(m4[i & 3], __uint_as_float(s[c][i]));
                mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                if (!kFp8) mt *= sl2;  // bf16: the scale is applied with the exponent below
            }
            mx[((j & 1) * 2 + hf) * 128 + row] = mt;
            named_bar(pair_bar, 64);
            mt = fmaxf(mt, mx[((j & 1) * 2 + (hf ^ 1)) * 128 + row]);
            alive = ok_s;
            if (!alive) continue;
            const float m_new = fmaxf(m, mt);
            const bool need = m_new > m + 8.f;  // also true when m is still -inf
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                // O holds P_0 .. P_{j-1} V: once PV_{j-1} is done, rescale this warp's half of
                // the rows that move
                alive = warp_wait(bar(B_PVDONE + (j - 1) % kSBufs), ((j - 1) / kSBufs) & 1, abort, ds);
                if (!alive) continue;
                tc_fence_after();
                const float f = need ? fast_exp2(m - m_new) : 1.f;
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    uint32_t o[32];
                    const uint32_t col = tmem + lane_base + kOCol + 64u * hf + 32u * c;
                    tmem_ld32(col, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
                    tmem_st32(col, o);
                }
                tmem_wait_st();
            }
            if (need) {
                lt *= fast_exp2(m - m_new);  // 0 while m is -inf
                m = m_new;
            }
            const float mu = m == -CUDART_INF_F ? 0.f : m;  // a row with nothing visible yet
            uint32_t pk[32];
            float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    float p0, p1;
                    if (kFp8) {
                        p0 = fast_exp2(__uint_as_float(s[c][i]) - mu);
                        p1 = fast_exp2(__uint_as_float(s[c][i + 1]) - mu);
                    } else {
                        p0 = fast_exp2(fmaf(__uint_as_float(s[c][i]), sl2, -mu));
                        p1 = fast_exp2(fmaf(__uint_as_float(s[c][i + 1]), sl2, -mu));
                    }
                    l4[(i >> 1) & 3] += p0 + p1;
                    if (kFp8) {
                        const int k = 64 * hf + 32 * c + i;
                        pk[16 * c + i / 2] = pack_bf16x2(p0 * sc[(j & 1) * 128 + k].y, p1 * sc[(j & 1) * 128 + k + 1].y);
                    } else {
                        pk[16 * c + i / 2] = pack_bf16x2(p0, p1);
                    }
                }
            lt += (l4[0] + l4[1]) + (l4[2] + l4[3]);
            tmem_st32(tmem + lane_base + 128u * sb + 32u * hf, pk);  // P over S: keys 64 hf .. at 32 hf
            tmem_wait_st();
            tc_fence_before();
            bar_arrive(bar(B_PREADY + sb));
        }
        // ------------------------------------------------------------ epilogue
        // Rows of o are 64 KB apart in global memory (one head of a token), so each warp passes its
        // 32 rows x 64 columns through a shared-memory slab in the freed K ring and moves them
        // with whole 256-byte rows per instruction. The earlier segments' result is read first,
        // while the last PV is still running.
        constexpr int kSlabStride = 68;  // floats per slab row (padding keeps 16-byte accesses conflict-free)
        float* const slab = reinterpret_cast<float*>(sgen + OFF_K) + warp * 32 * kSlabStride;
        const bool live_row = t < q_len;
        const int64_t gi = (int64_t)(q_begin + (live_row ? t : 0)) * p.H + h;
        const float lse_old = (p.merge && live_row) ? p.lse[gi] : -CUDART_INF_F;  // read before either half writes
        const int sub = lane >> 4, c4 = lane & 15;  // coalesced phase: two rows per instruction
        if (p.merge) {
#pragma unroll 4
            for (int r2 = 0; r2 < 16; ++r2) {
                const int rl = 2 * r2 + sub, tq = r0 + 32 * quarter + rl;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (tq < q_len)
                    v = *reinterpret_cast<const float4*>(p.o + ((int64_t)(q_begin + tq) * p.H + h) * kV + 64 * hf + 4 * c4);
                *reinterpret_cast<float4*>(slab + rl * kSlabStride + 4 * c4) = v;
            }
        }
        const bool ok =
            alive && warp_wait(bar(B_PVDONE + (n_tiles - 1) % kSBufs), ((n_tiles - 1) / kSBufs) & 1, abort, ds);
        mx[(4 + hf) * 128 + row] = lt;  // the row's sum is the two halves' sums (same running max)
        named_bar(pair_bar, 64);
        const float l = lt + mx[(4 + (hf ^ 1)) * 128 + row];
        const float nan = __uint_as_float(0x7fc00000u);  // marks a CTA that gave up
        const float inv = ok ? 1.f / l : nan;
        float lse = ok ? (m + log2f(l)) * 0.6931471805599453f : nan;
        float wo = 0.f, wn = 1.f;
        if (p.merge) {  // merge_attn_states with the earlier segments' (o, lse)
            const float M = fmaxf(lse_old, lse);
            wo = lse_old == -CUDART_INF_F ? 0.f : expf(lse_old - M);
            wn = lse == -CUDART_INF_F ? 0.f : expf(lse - M);
            const float ws = wo + wn;
            lse = M + logf(ws);
            wo /= ws;
            wn /= ws;
        }
        const float fn = wn * inv;
        if (ok) tc_fence_after();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            uint32_t r[32];
            if (ok) {
                tmem_ld32(tmem + lane_base + kOCol + 64u * hf + 32u * c, r);
                tmem_wait_ld();
            }
            float* const srow = slab + lane * kSlabStride + 32 * c;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                float4 v = make_float4(__uint_as_float(r[i]) * fn, __uint_as_float(r[i + 1]) * fn,
                                       __uint_as_float(r[i + 2]) * fn, __uint_as_float(r[i + 3]) * fn);
                if (!ok) v = make_float4(nan, nan, nan, nan);
                if (p.merge) {
                    const float4 u = *reinterpret_cast<const float4*>(srow + i);
                    v.x = fmaf(wo, u.x, v.x);
                    v.y = fmaf(wo, u.y, v.y);
                    v.z = fmaf(wo, u.z, v.z);
                    v.w = fmaf(wo, u.w, v.w);
                }
                *reinterpret_cast<float4*>(srow + i) = v;
            }
        }
        __syncwarp();
#pragma unroll 4
        for (int r2 = 0; r2 < 16; ++r2) {
            const int rl = 2 * r2 + sub, tq = r0 + 32 * quarter + rl;
            if (tq < q_len)
                *reinterpret_cast<float4*>(p.o + ((int64_t)(q_begin + tq) * p.H + h) * kV + 64 * hf + 4 * c4) =
                    *reinterpret_cast<const float4*>(slab + rl * kSlabStride + 4 * c4);
        }
        if (hf == 0 && live_row) p.lse[gi] = lse;
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 8) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_prefill_cu_ctx(const int32_t* ctx_lens, int B, int32_t* cu_ctx, int32_t* dev_status,
                                  cudaStream_t s) {
    return launch_pdl(cu_ctx_kernel, dim3(1), dim3(kScanThreads), 0, s, ctx_lens, B, (int32_t)0x7fffffff, cu_ctx,
                      dev_status);
}

cudaError_t launch_prefill_gather(const PrefillGather& g, cudaStream_t s) {
    if (g.rows <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((g.rows + kGatherWarps - 1) / kGatherWarps);
    return launch_pdl(gather_kernel, dim3(blocks), dim3(kGatherWarps * 32), 0, s, g);
}

cudaError_t launch_prefill_attn(const PrefillAttn& a, cudaStream_t s) {
    if (a.T <= 0 || a.key_rows <= 0 || a.max_q_len <= 0) return cudaSuccess;
    CUtensorMap qm, knm, kpm, vm;
    cudaError_t e;
    {
        const uint64_t dims[3] = {192, (uint64_t)a.H, (uint64_t)a.T};
        const uint64_t strides[2] = {192 * 2, (uint64_t)a.H * 192 * 2};
        const uint32_t box[3] = {64, 1, 128};
        if ((e = encode_tmap(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.q, dims, strides, box, true)) != cudaSuccess)
            return e;
    }
    {
        // head-major [H][key_rows][128]: one head's keys are contiguous 256-byte rows
        const uint64_t dims[3] = {128, (uint64_t)a.key_rows, (uint64_t)a.H};
        const uint64_t strides[2] = {128 * 2, (uint64_t)a.key_rows * 128 * 2};
        const uint32_t box[3] = {64, 128, 1};
        if ((e = encode_tmap(&knm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.kn, dims, strides, box, true)) != cudaSuccess)
            return e;
        if ((e = encode_tmap(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.v, dims, strides, box, true)) != cudaSuccess)
            return e;
    }
    {
        const uint64_t dims[2] = {64, (uint64_t)a.key_rows};
        const uint64_t strides[1] = {64 * 2};
        const uint32_t box[2] = {64, 128};
        if ((e = encode_tmap(&kpm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.kpe, dims, strides, box, true)) != cudaSuccess)
            return e;
    }
    const dim3 grid((unsigned)((a.max_q_len + 127) / 128), (unsigned)a.B, (unsigned)a.H);
    if (a.scales != nullptr) {
        if ((e = cudaFuncSetAttribute(attn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem)) !=
            cudaSuccess)
            return e;
        return launch_pdl(attn_kernel<true>, grid, dim3(kAttnThreads), (size_t)kAttnSmem, s, qm, knm, kpm, vm, a);
    }
    if ((e = cudaFuncSetAttribute(attn_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kAttnSmem)) !=
        cudaSuccess)
        return e;
    return launch_pdl(attn_kernel<false>, grid, dim3(kAttnThreads), (size_t)kAttnSmem, s, qm, knm, kpm, vm, a);
}

}  // namespace mla
