// gemm_simt.cu -- first, plain CUDA-core versions of the two per-head batched GEMMs.
//
// absorb:   q[t, h, 0:512] = q_nope[t, h, :] . W_UK_T[h]   and  q[t, h, 512:576] = q_pe[t, h, :]
//           ([vLLM-MLA, two-algorithms section]: torch.bmm(q_nope^T, W_UK_T) then concat q_pe)
// out_proj: o[t, h, :] = o_latent[t, h, :] . W_UV[h]        ([vLLM-MLA], _v_up_proj)
// One CTA per (head, group of 8 tokens); each thread owns one output column for the 8 tokens
// and streams the head's weight matrix once, coalesced along that column index.
#include <cuda_bf16.h>

#include "internal.h"

namespace mla {
namespace {

constexpr int kTok = 8;

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__global__ void __launch_bounds__(kL) absorb_simt_kernel(const uint16_t* __restrict__ q_nope, int64_t snt,
                                                         int64_t snh, const uint16_t* __restrict__ q_pe,
                                                         int64_t spt, int64_t sph,
                                                         const uint16_t* __restrict__ w_uk_t,
                                                         uint16_t* __restrict__ q_out, int T, int H) {
    __shared__ float qn[kTok][kP];
    const int h = blockIdx.x, t0 = blockIdx.y * kTok, l = threadIdx.x;
    for (int i = threadIdx.x; i < kTok * kP; i += blockDim.x) {
        int tt = i / kP, pp = i % kP;
        qn[tt][pp] = (t0 + tt < T) ? bf(q_nope[(int64_t)(t0 + tt) * snt + (int64_t)h * snh + pp]) : 0.f;
    }
    __syncthreads();
    float acc[kTok];
#pragma unroll
    for (int i = 0; i < kTok; ++i) acc[i] = 0.f;
    const uint16_t* w = w_uk_t + (size_t)h * kP * kL + l;
    for (int pp = 0; pp < kP; ++pp) {
        const float wv = bf(w[(size_t)pp * kL]);
#pragma unroll
        for (int i = 0; i < kTok; ++i) acc[i] = fmaf(qn[i][pp], wv, acc[i]);
    }
    for (int i = 0; i < kTok && t0 + i < T; ++i) {
        uint16_t* out = q_out + ((size_t)(t0 + i) * H + h) * kD;
        __nv_bfloat16 v = __float2bfloat16_rn(acc[i]);
        out[l] = *reinterpret_cast<uint16_t*>(&v);
        if (q_pe && l < kR) out[kL + l] = q_pe[(int64_t)(t0 + i) * spt + (int64_t)h * sph + l];
    }
}

__global__ void __launch_bounds__(kV) out_proj_simt_kernel(const void* __restrict__ o_latent, int in_dtype,
                                                           const uint16_t* __restrict__ w_uv, void* __restrict__ o,
                                                           int out_dtype, int T, int H) {
    __shared__ float x[kTok][kL];
    const int h = blockIdx.x, t0 = blockIdx.y * kTok, v = threadIdx.x;
    for (int i = threadIdx.x; i < kTok * kL; i += blockDim.x) {
        int tt = i / kL, ll = i % kL;
        float val = 0.f;
        if (t0 + tt < T) {
            size_t idx = ((size_t)(t0 + tt) * H + h) * kL + ll;
            val = in_dtype == MLA_DT_F32 ? ((const float*)o_latent)[idx] : bf(((const uint16_t*)o_latent)[idx]);
        }
        x[tt][ll] = val;
    }
    __syncthreads();
    float acc[kTok];
#pragma unroll
    for (int i = 0; i < kTok; ++i) acc[i] = 0.f;
    const uint16_t* w = w_uv + (size_t)h * kL * kV + v;
    for (int ll = 0; ll < kL; ++ll) {
        const float wv = bf(w[(size_t)ll * kV]);
#pragma unroll
        for (int i = 0; i < kTok; ++i) acc[i] = fmaf(x[i][ll], wv, acc[i]);
    }
    for (int i = 0; i < kTok && t0 + i < T; ++i) {
        size_t idx = ((size_t)(t0 + i) * H + h) * kV + v;
        if (out_dtype == MLA_DT_F32)
            ((float*)o)[idx] = acc[i];
        else
            ((__nv_bfloat16*)o)[idx] = __float2bfloat16_rn(acc[i]);
    }
}

}  // namespace

cudaError_t launch_absorb_simt(const uint16_t* q_nope, int64_t snt, int64_t snh, const uint16_t* q_pe, int64_t spt,
                               int64_t sph, const uint16_t* w_uk_t, uint16_t* q_out, int T, int H, cudaStream_t s) {
    dim3 grid(H, (T + kTok - 1) / kTok);
    absorb_simt_kernel<<<grid, kL, 0, s>>>(q_nope, snt, snh, q_pe, spt, sph, w_uk_t, q_out, T, H);
    return cudaGetLastError();
}

cudaError_t launch_out_proj_simt(const void* o_latent, int in_dtype, const uint16_t* w_uv, void* o, int out_dtype,
                                 int T, int H, cudaStream_t s) {
    dim3 grid(H, (T + kTok - 1) / kTok);
    out_proj_simt_kernel<<<grid, kV, 0, s>>>(o_latent, in_dtype, w_uv, o, out_dtype, T, H);
    return cudaGetLastError();
}

}  // namespace mla
