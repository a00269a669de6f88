// plan.cu -- device-built decode schedule ("scheduler metadata"; [vLLM-MLA, metadata section]:
// FlashMLA's decode metadata carries a scheduler plan, and the lengths that shape a batch are
// not synchronised back to the host).
//
// One CTA reads seq_lens and cuts every query row into page-aligned units of about c pages,
// choosing c from a ladder of candidates by a model of the hardware's cluster scheduling:
//     time(c) ~ max(longest unit + o, ceil(units / pairs) * (mean unit + o))      [pages]
// where o is the fixed cost of a unit (start-up and tail of one cluster pair, in page-times)
// and pairs is the number of 2-SM clusters that run at once. The candidates are multiples of
// total / (2 pairs) and the even splits of the longest row (longest / k), both cutting a row into
// equal page-aligned pieces (split_range, the uniform splits' rule), and the sizes that fill
// W = 2, 3, 4 or 6 waves, which cut a row into units of c pages and a shorter last one (FP8
// cache only, whose pages take long enough next to a split unit's partials and merge); for
// those the model is the greedy list-scheduling bound max(longest + o, (total + units o) / pairs).
// A candidate whose unit count exceeds rows + 2 pairs (the grid's size) is not taken. A row that
// gets one unit writes its final output directly; the units of a split row write fp32 partials
// that the merge combines.
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
constexpr int kRem = 4;            // total / (W pairs) for W = 2, 3, 4, 6, cut with a remainder
constexpr int kCands = kLadder + kEven + kRem;
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
    __shared__ int s_wsum[kWarps][kBuckets + 2];  // per warp: units per bucket, split rows, their units
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
        } else if (warp < kLadder + kEven) {  // the longest row cut into k even pieces
            const int k = warp - kLadder + 1;
            const int cc = (longest + k - 1) / k;
            c = min(longest, (cc + 3) / 4 * 4);
        } else {  // units of the size that fills W waves, a row's last unit taking the remainder
            const int W = warp - kLadder - kEven == 3 ? 6 : warp - kLadder - kEven + 2;
            const int cc = (int)ceilf((float)total_pages / (float)(W * pairs));
            c = min(longest, max(4, (cc + 3) / 4 * 4));
        }
        const bool rem = warp >= kLadder + kEven;
        unsigned long long units = 0;
        int lu = 0;
        for (int r = lane; r < R; r += 32) {
            const int pg = pages_of(tokens(r));
            const int S = units_of(pg, c);
            units += (unsigned long long)S;
            lu = max(lu, rem ? min(pg, c) : (pg + S - 1) / S);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) units += __shfl_xor_sync(0xffffffffu, units, off);
        lu = (int)__reduce_max_sync(0xffffffffu, (unsigned)lu);
        if (lane == 0) {
            s_cand[warp] = rem ? -c : c;  // negative: cut with a remainder
            s_units[warp] = units;
            s_lu[warp] = lu;
            if (warp == 0) s_total = total_pages;
        }
    }
    __syncthreads();

    // warp 0 picks the candidate with the least modelled time (ties: the longer units)
    if (warp == 0) {
        const bool fp8 = p.kv_dtype == MLA_KV_FP8_E4M3_SCALED;
        const float o = fp8 ? kUnitCostFp8 : kUnitCostBf16;
        const float total_pages = (float)s_total;
        float cost = 3.0e38f;
        int c = 0;
        if (lane < kCands) {
            c = s_cand[lane];
            const unsigned long long units = s_units[lane];
            if (units > 0 && units <= (unsigned long long)p.plan_max_units) {
                if (c > 0) {  // equal pieces: whole waves of units of about the mean size
                    const float waves = (float)(((unsigned)units + pairs - 1) / (unsigned)pairs);
                    cost = fmaxf((float)s_lu[lane] + o, waves * (total_pages / (float)units + o));
                } else if (fp8) {  // full units and remainders, longest first: the greedy bound
                    // (bf16 pages are cheap next to a split unit's partials and merge: measured
                    // slower at ragged, 202.5 against 193.1 us, so the cut is for FP8 only)
                    cost = fmaxf((float)s_lu[lane] + o, (total_pages + (float)units * o) / (float)pairs);
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float oc = __shfl_xor_sync(0xffffffffu, cost, off);
            const int occ = __shfl_xor_sync(0xffffffffu, c, off);
            if (oc < cost || (oc == cost && abs(occ) > abs(c))) {
                cost = oc;
                c = occ;
            }
        }
        if (lane == 0) s_best = cost < 3.0e38f ? c : s_cand[kLadder];  // no fit: one unit per row
    }
    __syncthreads();

    // the list: per-bucket unit counters (and split rows) scanned over the block in row order
    const bool rem = s_best < 0;
    const int c = rem ? -s_best : s_best;
    // counters: units per bucket, then split rows (list index) and their units (partial slots)
    constexpr int kC = kBuckets + 2;
    int cnt[kC] = {0, 0, 0, 0, 0, 0, 0};  // unit indices fit an int: at most plan_max_units
    for (int r = r0; r < r1; ++r) {
        const int pg = pages_of(tokens(r));
        const int S = units_of(pg, c);
        if (S == 1) {
            cnt[bucket_of(pg, c)] += 1;
        } else {
            cnt[0] += rem ? S - 1 : S;  // full-size units
            if (rem) cnt[bucket_of(pg - (S - 1) * c, c)] += 1;
            cnt[kBuckets] += 1;
            cnt[kBuckets + 1] += S;
        }
    }
    int incl[kC];
#pragma unroll
    for (int b = 0; b < kC; ++b) {
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
        for (int b = 0; b < kC; ++b) {
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
            if (lane == 0 && b == kBuckets) const_cast<int*>(p.plan_count)[1] = all;  // split rows
        }
    }
    __syncthreads();
    // this thread's first unit of each bucket, first split-row index, first partial slot
    int base[kC];
#pragma unroll
    for (int b = 0; b < kC; ++b) base[b] = s_wsum[warp][b] + incl[b] - cnt[b];
    int4* units = const_cast<int4*>(p.plan_units);
    int2* rows = const_cast<int2*>(p.plan_rows);
    int* split_rows = const_cast<int*>(p.plan_split_rows);
    for (int r = r0; r < r1; ++r) {
        const int n = tokens(r);
        const int pg = pages_of(n);
        const int S = units_of(pg, c);
        if (S == 1) {
            units[base[bucket_of(pg, c)]++] = make_int4(r, 0, n, -1);
            rows[r] = make_int2(-1, 1);
            continue;
        }
        const int slot0 = base[kBuckets + 1];
        for (int k = 0; k < S; ++k) {
            int j0, j1;
            if (rem) {  // c pages per unit, the last one the rest
                j0 = k * c * kPage;
                j1 = min(n, j0 + c * kPage);
            } else {
                split_range(n, S, k, &j0, &j1);
            }
            const int b = rem && k == S - 1 ? bucket_of(pg - (S - 1) * c, c) : 0;
            units[base[b]++] = make_int4(r, j0, j1, slot0 + k);
        }
        rows[r] = make_int2(slot0, S);
        split_rows[base[kBuckets]++] = r;
        base[kBuckets + 1] += S;
    }
}

}  // namespace

cudaError_t launch_plan(const DecodeArgs& a, int pairs, cudaStream_t s) {
    return launch_pdl(plan_kernel, dim3(1), dim3(kThreads), 0, s, a, pairs);
}

}  // namespace mla
