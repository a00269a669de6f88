// plan.cu -- device-built decode schedule ("scheduler metadata"; [vLLM-MLA, metadata section]:
// FlashMLA's decode metadata carries a scheduler plan, and the lengths that shape a batch are
// not synchronised back to the host).
//
// One CTA reads seq_lens and cuts every query row into page-aligned units of about c pages,
// choosing c from a short ladder by a model of the hardware's cluster scheduling:
//     time(c) ~ max(longest unit + o, ceil(units / pairs) * (mean unit + o))      [pages]
// where o is the fixed cost of a unit (start-up and tail of one cluster pair, in page-times)
// and pairs is the number of 2-SM clusters that run at once. Only c >= total / (2 pairs) is
// considered, so the unit count stays within rows + 2 pairs. A row that gets one unit writes its
// final output directly; the units of a split row write fp32 partials that the merge combines.
// The split points follow the same page-aligned rule as uniform splits (split_range).
#include <algorithm>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kMaxThreads = 1024;  // one CTA; the block size follows the row count (128..1024)
constexpr int kCands = 13;
constexpr int kSmemRows = 12288;  // rows whose page counts are kept in shared memory
constexpr float kUnitCost = 6.f;  // fixed cost of one unit, in page-times

__device__ __forceinline__ int pages_of(int n) { return (n + kPage - 1) / kPage; }

// Block scan of one value per thread; returns the exclusive prefix (and the block total).
__device__ __forceinline__ long long block_exclusive_scan(long long v, long long* warp_tot, long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    long long x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long w = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const long long before = (warp > 0 ? warp_tot[warp - 1] : 0) + x - v;
    if (total) *total = warp_tot[nwarps - 1];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kMaxThreads) plan_kernel(DecodeArgs p, int pairs) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();  // the schedule overwrites workspace an earlier kernel may still read
    __shared__ long long s_warp[32];
    __shared__ int s_pages[kSmemRows];
    __shared__ int s_cand[kCands];
    __shared__ float s_cost[kCands];
    __shared__ int s_best;
    const int R = p.rows;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int per = (R + (int)blockDim.x - 1) / (int)blockDim.x;
    const int r0 = min(R, tid * per), r1 = min(R, r0 + per);

    // total and longest row, in pages
    long long tot = 0;
    int mx = 0;
    for (int r = r0; r < r1; ++r) {
        const int pg = pages_of(visible_tokens(p, r, true));
        if (r < kSmemRows) s_pages[r] = pg;
        tot += pg;
        mx = max(mx, pg);
    }
    auto pages = [&](int r) { return r < kSmemRows ? s_pages[r] : pages_of(visible_tokens(p, r, false)); };
    long long total_pages = 0;
    block_exclusive_scan(tot, s_warp, &total_pages);
    int mxw = mx;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mxw = max(mxw, __shfl_xor_sync(0xffffffffu, mxw, off));
    __shared__ int s_mx[32];
    if (lane == 0) s_mx[warp] = mxw;
    __syncthreads();
    if (tid == 0) {
        int m = 0;
        for (int w = 0; w < nwarps; ++w) m = max(m, s_mx[w]);
        const int longest = max(m, 1);
        const long long cmin = max(1LL, (total_pages + 2LL * pairs - 1) / (2LL * pairs));
        const float mult[kCands - 1] = {1.f, 1.25f, 1.5f, 2.f, 2.5f, 3.f, 4.f, 6.f, 8.f, 12.f, 16.f, 32.f};
        for (int k = 0; k < kCands - 1; ++k) {
            long long c = (long long)ceilf((float)cmin * mult[k]);
            c = (c + 3) / 4 * 4;  // whole 4-page groups
            if (c < cmin) c = cmin;
            if (c > longest) c = longest;
            s_cand[k] = (int)c;
        }
        s_cand[kCands - 1] = longest;  // one unit per row
    }
    __syncthreads();

    // cost of each candidate (one warp each)
    for (int k = warp; k < kCands; k += nwarps) {
        const int c = s_cand[k];
        long long units = 0;
        int longest_unit = 0;
        for (int r = lane; r < R; r += 32) {
            const int pg = pages(r);
            const int S = pg <= c ? 1 : (pg + c - 1) / c;
            units += S;
            longest_unit = max(longest_unit, (pg + S - 1) / S);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            units += __shfl_xor_sync(0xffffffffu, units, off);
            longest_unit = max(longest_unit, __shfl_xor_sync(0xffffffffu, longest_unit, off));
        }
        if (lane == 0) {
            float cost = 3.0e38f;
            if (units <= p.plan_max_units) {
                const float waves = (float)((units + pairs - 1) / pairs);
                cost = fmaxf((float)longest_unit + kUnitCost,
                             waves * ((float)total_pages / (float)units + kUnitCost));
            }
            s_cost[k] = cost;
        }
    }
    __syncthreads();
    if (tid == 0) {
        int best = kCands - 1;
        for (int k = 0; k < kCands; ++k)
            if (s_cost[k] < s_cost[best] || (s_cost[k] == s_cost[best] && s_cand[k] > s_cand[best])) best = k;
        s_best = s_cand[best];
    }
    __syncthreads();

    // The list, longest units first (the hardware hands clusters out in list order, so this is
    // greedy longest-first scheduling): bucket 0 holds the units of split rows (about c pages
    // each), buckets 1-4 the unsplit rows by length (>= c/2, >= c/4, >= c/16, shorter).
    const int c = s_best;
    auto bucket_of = [&](int pg) {
        if (pg > c) return 0;
        if (2 * pg >= c) return 1;
        if (4 * pg >= c) return 2;
        if (16 * pg >= c) return 3;
        return 4;
    };
    int4* units = const_cast<int4*>(p.plan_units);
    int2* rows = const_cast<int2*>(p.plan_rows);
    long long ubase_all = 0;
    long long pbase = 0;
    for (int bk = 0; bk < 5; ++bk) {
        long long nu = 0;
        for (int r = r0; r < r1; ++r) {
            const int pg = pages(r);
            if (bucket_of(pg) == bk) nu += pg <= c ? 1 : (pg + c - 1) / c;
        }
        long long bucket_units = 0;
        long long ub = ubase_all + block_exclusive_scan(nu, s_warp, &bucket_units);
        long long pb = bk == 0 ? ub : 0;  // partial slots: bucket 0 comes first (ubase_all = 0)
        for (int r = r0; r < r1; ++r) {
            const int pg = pages(r);
            if (bucket_of(pg) != bk) continue;
            const int n = visible_tokens(p, r, false);
            const int S = pg <= c ? 1 : (pg + c - 1) / c;
            for (int k = 0; k < S; ++k) {
                int j0, j1;
                split_range(n, S, k, &j0, &j1);
                units[ub + k] = make_int4(r, j0, j1, S > 1 ? (int)(pb + k) : -1);
            }
            rows[r] = make_int2(S > 1 ? (int)pb : -1, S);
            ub += S;
            if (S > 1) pb += S;
        }
        ubase_all += bucket_units;
        if (bk == 0) pbase = bucket_units;
    }
    const long long total_units = ubase_all;
    (void)pbase;
    if (tid == 0) *const_cast<int*>(p.plan_count) = (int)total_units;
}

}  // namespace

cudaError_t launch_plan(const DecodeArgs& a, int pairs, cudaStream_t s) {
    // one row per thread where the batch allows it, so that few threads wait at each barrier
    const int threads = (int)std::min<int64_t>(kMaxThreads, std::max<int64_t>(128, (a.rows + 31) / 32 * 32));
    return launch_pdl(plan_kernel, dim3(1), dim3(threads), 0, s, a, pairs);
}

}  // namespace mla
