// plan.cu -- device-built decode schedule ("scheduler metadata"; [vLLM-MLA, metadata section]:
// FlashMLA's decode metadata carries a scheduler plan, and the lengths that shape a batch are
// not synchronised back to the host).
//
// One CTA reads seq_lens and cuts every query row into page-aligned units of about c pages,
// choosing c from a ladder of candidates by a model of the hardware's cluster scheduling:
//     time(c) ~ max(longest unit + o, ceil(units / pairs) * (mean unit + o))      [pages]
// where o is the fixed cost of a unit (start-up and tail of one cluster pair, in page-times)
// and pairs is the number of 2-SM clusters that run at once. The candidates are multiples of
// total / (2 pairs) and the even splits of the longest row (longest / k); a candidate whose
// unit count exceeds rows + 2 pairs (the grid's size) is not taken. A row that gets one unit
// writes its final output directly; the units of a split row write fp32 partials that the merge
// combines. The split points follow the same page-aligned rule as uniform splits (split_range).
//
// The kernel is a chain of dependent steps on one SM, so it is written for short chains: one
// warp per candidate walks the rows, one lane per candidate picks the winner, and the per-warp
// sums of the bucket counters are scanned by one lane per warp. Five block barriers in all.
#include "internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 1024;     // one CTA: a warp per candidate, up to a row per thread
constexpr int kWarps = kThreads / 32;
constexpr int kLadder = 12;        // multiples of total / (2 pairs)
constexpr int kEven = 16;          // longest / k, k = 1..kEven
constexpr int kCands = kLadder + kEven;
static_assert(kCands <= 32 && kCands <= kThreads / 32, "a warp per candidate, a lane per candidate in warp 0");
constexpr int kSmemRows = 8192;    // rows whose visible token counts are kept in shared memory
constexpr int kBuckets = 5;        // longest first: split rows, then unsplit rows by length
constexpr float kUnitCostBf16 = 8.f;  // fixed cost of one unit, in page-times of the bf16 kernel
constexpr float kUnitCostFp8 = 4.f;   // the FP8 kernel's pages take about twice as long

__device__ __forceinline__ int pages_of(int n) { return (n + kPage - 1) / kPage; }
__device__ __forceinline__ int units_of(int pg, int c) { return pg <= c ? 1 : (pg + c - 1) / c; }
// longest first: bucket 0 holds the units of split rows (about c pages each), buckets 1-4 the
// unsplit rows by length (>= c/2, >= c/4, >= c/16, shorter)
__device__ __forceinline__ int bucket_of(int pg, int c) {
    if (pg > c) return 0;
    if (2 * pg >= c) return 1;
    if (4 * pg >= c) return 2;
    if (16 * pg >= c) return 3;
    return 4;
}

__global__ void __launch_bounds__(kThreads) plan_kernel(DecodeArgs p, int pairs) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();  // the schedule overwrites workspace an earlier kernel may still read
    __shared__ int s_n[kSmemRows];
    __shared__ unsigned long long s_tot[kWarps];
    __shared__ int s_mx[kWarps];
    __shared__ int s_cand[kCands];
    __shared__ unsigned long long s_units[kCands];
    __shared__ int s_lu[kCands];
    __shared__ int s_best;
    __shared__ unsigned long long s_total;
    __shared__ int s_wsum[kWarps][kBuckets + 1];  // per warp: units per bucket, split rows
    const int R = p.rows;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (R + kThreads - 1) / kThreads;
    const int r0 = min(R, tid * per), r1 = min(R, r0 + per);

    // visible tokens of this thread's rows; total and longest row, in pages
    unsigned long long tot = 0;
    int mx = 0;
    for (int r = r0; r < r1; ++r) {
        const int n = visible_tokens(p, r, true);
        if (r < kSmemRows) s_n[r] = n;
        tot += (unsigned long long)pages_of(n);
        mx = max(mx, pages_of(n));
    }
    auto tokens = [&](int r) { return r < kSmemRows ? s_n[r] : visible_tokens(p, r, false); };
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    mx = (int)__reduce_max_sync(0xffffffffu, (unsigned)mx);
    if (lane == 0) {
        s_tot[warp] = tot;
        s_mx[warp] = mx;
    }
    __syncthreads();

    // warp k evaluates candidate k: its unit count and longest unit over all rows
    if (warp < kCands) {
        unsigned long long total_pages = 0;
        int longest = 1;
#pragma unroll 8
        for (int w = 0; w < kWarps; ++w) {
            total_pages += s_tot[w];
            longest = max(longest, s_mx[w]);
        }
        int c;
        if (warp < kLadder) {  // a multiple of total / (2 pairs), in whole 4-page groups
            const float mult[kLadder] = {1.f, 1.25f, 1.5f, 2.f, 2.5f, 3.f, 4.f, 6.f, 8.f, 12.f, 16.f, 32.f};
            // (float division: a candidate a page short of the bound is caught by the unit check)
            const int cmin = max(1, (int)ceilf((float)total_pages / (float)(2 * pairs)));
            int cc = (int)ceilf((float)cmin * mult[warp]);
            cc = (cc + 3) / 4 * 4;
            c = min(longest, max(cc, cmin));
        } else {  // the longest row cut into k even pieces
            const int k = warp - kLadder + 1;
            const int cc = (longest + k - 1) / k;
            c = min(longest, (cc + 3) / 4 * 4);
        }
        unsigned long long units = 0;
        int lu = 0;
        for (int r = lane; r < R; r += 32) {
            const int pg = pages_of(tokens(r));
            const int S = units_of(pg, c);
            units += (unsigned long long)S;
            lu = max(lu, (pg + S - 1) / S);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) units += __shfl_xor_sync(0xffffffffu, units, off);
        lu = (int)__reduce_max_sync(0xffffffffu, (unsigned)lu);
        if (lane == 0) {
            s_cand[warp] = c;
            s_units[warp] = units;
            s_lu[warp] = lu;
            if (warp == 0) s_total = total_pages;
        }
    }
    __syncthreads();

    // warp 0 picks the candidate with the least modelled time (ties: the longer units)
    if (warp == 0) {
        const float o = p.kv_dtype == MLA_KV_FP8_E4M3_SCALED ? kUnitCostFp8 : kUnitCostBf16;
        const float total_pages = (float)s_total;
        float cost = 3.0e38f;
        int c = 0;
        if (lane < kCands) {
            c = s_cand[lane];
            const unsigned long long units = s_units[lane];
            if (units > 0 && units <= (unsigned long long)p.plan_max_units) {
                const float waves = (float)(((unsigned)units + pairs - 1) / (unsigned)pairs);
                cost = fmaxf((float)s_lu[lane] + o, waves * (total_pages / (float)units + o));
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float oc = __shfl_xor_sync(0xffffffffu, cost, off);
            const int occ = __shfl_xor_sync(0xffffffffu, c, off);
            if (oc < cost || (oc == cost && occ > c)) {
                cost = oc;
                c = occ;
            }
        }
        if (lane == 0) s_best = cost < 3.0e38f ? c : s_cand[kCands - kEven];  // no fit: one unit per row
    }
    __syncthreads();

    // the list: per-bucket unit counters (and split rows) scanned over the block in row order
    const int c = s_best;
    int cnt[kBuckets + 1] = {0, 0, 0, 0, 0, 0};  // unit indices fit an int: at most plan_max_units
    for (int r = r0; r < r1; ++r) {
        const int pg = pages_of(tokens(r));
        const int b = bucket_of(pg, c);
        cnt[b] += units_of(pg, c);
        if (b == 0) cnt[kBuckets] += 1;
    }
    int incl[kBuckets + 1];
#pragma unroll
    for (int b = 0; b <= kBuckets; ++b) {
        int x = cnt[b];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        incl[b] = x;
        if (lane == 31) s_wsum[warp][b] = x;
    }
    __syncthreads();
    if (warp == 0) {  // lane w: warp w's offset within each bucket, then the buckets' starts
        int bucket_start = 0;
#pragma unroll
        for (int b = 0; b <= kBuckets; ++b) {
            const int v = s_wsum[lane][b];
            int x = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            const int all = __shfl_sync(0xffffffffu, x, 31);
            s_wsum[lane][b] = (b < kBuckets ? bucket_start : 0) + x - v;
            if (b < kBuckets) bucket_start += all;
            if (lane == 0 && b == kBuckets - 1) *const_cast<int*>(p.plan_count) = bucket_start;
            if (lane == 0 && b == kBuckets) const_cast<int*>(p.plan_count)[1] = all;
        }
    }
    __syncthreads();
    int base[kBuckets + 1];  // this thread's first unit of each bucket (first split-row index)
#pragma unroll
    for (int b = 0; b <= kBuckets; ++b) base[b] = s_wsum[warp][b] + incl[b] - cnt[b];
    int4* units = const_cast<int4*>(p.plan_units);
    int2* rows = const_cast<int2*>(p.plan_rows);
    int* split_rows = const_cast<int*>(p.plan_split_rows);
    for (int r = r0; r < r1; ++r) {
        const int n = tokens(r);
        const int pg = pages_of(n);
        const int b = bucket_of(pg, c);
        const int S = units_of(pg, c);
        const int ub = base[b];
        // bucket 0 comes first, so a split row's units and its partial slots share indices
        for (int k = 0; k < S; ++k) {
            int j0, j1;
            split_range(n, S, k, &j0, &j1);
            units[ub + k] = make_int4(r, j0, j1, S > 1 ? ub + k : -1);
        }
        rows[r] = make_int2(S > 1 ? ub : -1, S);
        if (S > 1) split_rows[base[kBuckets]++] = r;
        base[b] += S;
    }
}

}  // namespace

cudaError_t launch_plan(const DecodeArgs& a, int pairs, cudaStream_t s) {
    return launch_pdl(plan_kernel, dim3(1), dim3(kThreads), 0, s, a, pairs);
}

}  // namespace mla
