// merge.cu -- split-KV stage 2: combine the per-split partial states of every (row, head).
//
// [vLLM-MLA, Triton MLA section]: stage 1 writes a partial output and LSE per split into an
// fp32 buffer (B, N, splits, 512 + 1); stage 2 reduces them by LSE. [vLLM-MLA, Prefill
// section], merge_attn_states: partials are re-weighted by exp(lse - max_lse); an empty partial
// (o = 0, lse = -inf) has no weight.
//     M = max_s lse_s,  w_s = exp(lse_s - M),  lse = M + ln sum_s w_s,  o = sum_s w_s o_s / sum_s w_s
// One warp per (row, head, half of the latent dims); lane i owns 8 dims of its half. The partial
// states are read once, coalesced, four splits at a time so that each lane has eight 16-byte
// loads in flight, and the result is written once.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;
constexpr int kBatch = 4;  // splits whose partials are loaded together

__device__ __forceinline__ void merge_item(const DecodeArgs& p, int64_t r, int h, int half, int lane);

__global__ void __launch_bounds__(kWarps * 32) merge_kernel(DecodeArgs p) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();  // the partials are the preceding kernel's output
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    // grid-stride over (row, head, half) of the rows with partials: every row with uniform
    // splits, the listed split rows with a device-built schedule (none: the kernel ends here)
    const int64_t n_rows = p.plan_rows ? (int64_t)p.plan_count[1] : (int64_t)p.rows;
    const int64_t n_tasks = n_rows * p.H * 2;
    for (int64_t t = (int64_t)blockIdx.x * kWarps + warp; t < n_tasks; t += (int64_t)gridDim.x * kWarps) {
        const int64_t item = t >> 1;
        const int64_t i = item / p.H;
        const int64_t r = p.plan_rows ? (int64_t)p.plan_split_rows[i] : i;
        merge_item(p, r, (int)(item % p.H), (int)(t & 1), lane);
    }
}

__device__ __forceinline__ void merge_item(const DecodeArgs& p, int64_t r, int h, int half, int lane) {
    // the row's partials are slots [slot0, slot0 + S): uniform splits put row r at r * S; a
    // device-built schedule lists them per row (a row with one unit already wrote its output)
    int S, slot0;
    if (p.plan_rows) {
        const int2 ri = p.plan_rows[r];
        S = ri.y;
        slot0 = ri.x;
        if (S <= 1) return;
    } else {
        S = p.num_splits;
        slot0 = (int)(r * S);
    }
    const float* lse_p = p.part_lse + (size_t)slot0 * p.H + h;  // stride H between splits

    float M = -CUDART_INF_F;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, lse_p[(size_t)s * p.H]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    float wsum = 0.f;
    if (M != -CUDART_INF_F) {
        const size_t split_stride = (size_t)p.H * kL;
        const float* src0 = p.part_o + ((size_t)slot0 * p.H + h) * kL + half * (kL / 2) + lane * 8;
        for (int s0 = 0; s0 < S; s0 += kBatch) {
            // all loads of the batch first, then the arithmetic in split order
            float ls[kBatch];
            float4 v[kBatch][2];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                ls[u] = -CUDART_INF_F;
                v[u][0] = v[u][1] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (s0 + u < S) {
                    ls[u] = lse_p[(size_t)(s0 + u) * p.H];
                    const float4* src = reinterpret_cast<const float4*>(src0 + (size_t)(s0 + u) * split_stride);
                    v[u][0] = src[0];
                    v[u][1] = src[1];
                }
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (ls[u] == -CUDART_INF_F) continue;  // an empty split has no weight
                const float w = __expf(ls[u] - M);
                wsum += w;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    acc[4 * i + 0] = fmaf(w, v[u][i].x, acc[4 * i + 0]);
                    acc[4 * i + 1] = fmaf(w, v[u][i].y, acc[4 * i + 1]);
                    acc[4 * i + 2] = fmaf(w, v[u][i].z, acc[4 * i + 2]);
                    acc[4 * i + 3] = fmaf(w, v[u][i].w, acc[4 * i + 3]);
                }
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const size_t base = ((size_t)r * p.H + h) * kL + half * (kL / 2) + lane * 8;
    if (p.o_dtype == MLA_DT_F32) {
        float4* dst = reinterpret_cast<float4*>((float*)p.o_latent + base);
#pragma unroll
        for (int i = 0; i < 2; ++i)
            dst[i] = make_float4(acc[4 * i] * inv, acc[4 * i + 1] * inv, acc[4 * i + 2] * inv, acc[4 * i + 3] * inv);
    } else {
        __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>((__nv_bfloat16*)p.o_latent + base);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = __floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
    }
    if (half == 0 && lane == 0 && p.lse) p.lse[(size_t)r * p.H + h] = wsum > 0.f ? M + __logf(wsum) : -CUDART_INF_F;
}

}  // namespace

cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t s) {
    const int64_t n_tasks = (int64_t)a.rows * a.H * 2;
    int64_t blocks = (n_tasks + kWarps - 1) / kWarps;
    // grid-stride over the split rows: enough warps that each takes about one (row, head, half),
    // since a task is a chain of dependent loads; with no split row every block ends at once
    if (a.plan_rows && blocks > 1216) blocks = 1216;
    return launch_pdl(merge_kernel, dim3((unsigned)blocks), dim3(kWarps * 32), 0, s, a);
}

}  // namespace mla
