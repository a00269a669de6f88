// decode_simt.cu -- first, plain CUDA-core version of the paged latent decode.
//
// One CTA handles 16 heads of one query row and one split: it walks the split's tokens in tiles
// of 32 rows gathered through the block table, keeps an online softmax per head and accumulates
// the 512-dim latent output in registers ([vLLM-MLA, two-algorithms section]: decode is MQA over
// the 576-dim rows; V is the first 512 dims of the same row).
#include <cuda_bf16.h>
#include <math_constants.h>

#include "internal.h"

namespace mla {
namespace {

constexpr int kHG = 16;          // heads per CTA
constexpr int kTT = 16;          // tokens per tile
constexpr int kThreads = 256;
constexpr int kRowWords = kD / 2 + 1;  // 289 32-bit words per smem row: odd stride, no bank clashes
static_assert(kHG * 16 == kThreads && kTT == 16, "one score per thread");

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kThreads) decode_simt_kernel(DecodeArgs p) {
    __shared__ uint32_t qs[kHG][kRowWords];  // bf16 pairs
    __shared__ uint32_t ks[kTT][kRowWords];
    __shared__ float ps[kHG][kTT];
    __shared__ float m_s[kHG], l_s[kHG], alpha_s[kHG];

    const int tid = threadIdx.x;
    const int hg = blockIdx.x, s = blockIdx.y, r = blockIdx.z;
    const int b = r / p.Sq, t = r % p.Sq;
    const int h0 = hg * kHG;

    int seq = p.seq_lens[b];
    const int cap = p.max_blocks * kPage;
    if (seq > cap || seq > p.max_seq_len) {
        if (tid == 0 && p.dev_status) atomicOr(p.dev_status, MLA_DEV_SEQ_TOO_LONG);
        seq = min(seq, cap);
    }
    int n = seq - (p.Sq - 1 - t);
    if (n < 0) n = 0;
    int j0, j1;
    split_range(n, p.num_splits, s, &j0, &j1);

    for (int i = tid; i < kHG * (kD / 2); i += kThreads) {
        int hh = i / (kD / 2), w = i % (kD / 2);
        uint32_t v = 0u;
        if (h0 + hh < p.H)
            v = reinterpret_cast<const uint32_t*>(p.q + ((size_t)r * p.H + h0 + hh) * kD)[w];
        qs[hh][w] = v;
    }
    if (tid < kHG) {
        m_s[tid] = -CUDART_INF_F;
        l_s[tid] = 0.f;
    }

    const int hh = tid / 16;         // head owned in the PV update
    const int d0 = (tid % 16) * 32;  // 32 latent dims owned
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    const float sl2 = p.scale * 1.4426950408889634f;  // scale * log2(e): exp2 domain
    const int32_t* bt = p.block_table + (size_t)b * p.max_blocks;
    __syncthreads();

    for (int j = j0; j < j1; j += kTT) {
        const int nt = min(kTT, j1 - j);
        // gather nt rows (1152 bytes each = 72 x 16 bytes)
        for (int i = tid; i < nt * 72; i += kThreads) {
            int row = i / 72, c = i % 72;
            int tok = j + row;
            int64_t blk = bt[tok / kPage];
            uint4 v = make_uint4(0, 0, 0, 0);
            if (blk < 0 || blk >= p.num_blocks) {
                if (c == 0 && p.dev_status) atomicOr(p.dev_status, MLA_DEV_BAD_BLOCK_ID);
            } else {
                const uint4* src = reinterpret_cast<const uint4*>(
                    p.cache + ((size_t)blk * kPage + tok % kPage) * kBf16RowBytes);
                v = __ldg(src + c);
            }
            uint32_t* dst = &ks[row][c * 4];
            dst[0] = v.x;
            dst[1] = v.y;
            dst[2] = v.z;
            dst[3] = v.w;
        }
        __syncthreads();
        // scores: thread (head tid / 16, token tid % 16)
        {
            const int sh = tid / 16, jj = tid % 16;
            float sc = -CUDART_INF_F;
            if (jj < nt) {
                float a0 = 0.f, a1 = 0.f;
                const uint32_t* qq = qs[sh];
                const uint32_t* kk = ks[jj];
#pragma unroll 8
                for (int w = 0; w < kD / 2; ++w) {
                    uint32_t kw = kk[w], qw = qq[w];
                    a0 = fmaf(bf16_lo(qw), bf16_lo(kw), a0);
                    a1 = fmaf(bf16_hi(qw), bf16_hi(kw), a1);
                }
                sc = (a0 + a1) * sl2;
            }
            ps[sh][jj] = sc;
        }
        __syncthreads();
        if (tid < kHG) {
            float mt = -CUDART_INF_F;
            for (int jj = 0; jj < nt; ++jj) mt = fmaxf(mt, ps[tid][jj]);
            float m_old = m_s[tid];
            float m_new = fmaxf(m_old, mt);
            float alpha = exp2f(m_old - m_new);  // 0 on the first tile (m_old = -inf)
            float sum = 0.f;
            for (int jj = 0; jj < nt; ++jj) {
                float pv = exp2f(ps[tid][jj] - m_new);
                ps[tid][jj] = pv;
                sum += pv;
            }
            l_s[tid] = l_s[tid] * alpha + sum;
            m_s[tid] = m_new;
            alpha_s[tid] = alpha;
        }
        __syncthreads();
        {
            const float alpha = alpha_s[hh];
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] *= alpha;
            for (int jj = 0; jj < nt; ++jj) {
                const float pv = ps[hh][jj];
                const uint32_t* kk = &ks[jj][d0 / 2];
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    uint32_t kw = kk[w];
                    acc[2 * w] = fmaf(pv, bf16_lo(kw), acc[2 * w]);
                    acc[2 * w + 1] = fmaf(pv, bf16_hi(kw), acc[2 * w + 1]);
                }
            }
        }
        __syncthreads();
    }

    const int h = h0 + hh;
    if (h >= p.H) return;
    const float l = l_s[hh];
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = l > 0.f ? (m_s[hh] + log2f(l)) * 0.6931471805599453f : -CUDART_INF_F;
    if (p.num_splits > 1) {
        float* dst = p.part_o + (((size_t)r * p.num_splits + s) * p.H + h) * kL + d0;
#pragma unroll
        for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) =
                make_float4(acc[i] * inv, acc[i + 1] * inv, acc[i + 2] * inv, acc[i + 3] * inv);
        if ((tid % 16) == 0) p.part_lse[((size_t)r * p.num_splits + s) * p.H + h] = lse_v;
    } else {
        size_t base = ((size_t)r * p.H + h) * kL + d0;
        if (p.o_dtype == MLA_DT_F32) {
            float* dst = (float*)p.o_latent + base;
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4*>(dst + i) =
                    make_float4(acc[i] * inv, acc[i + 1] * inv, acc[i + 2] * inv, acc[i + 3] * inv);
        } else {
            __nv_bfloat16* dst = (__nv_bfloat16*)p.o_latent + base;
#pragma unroll
            for (int i = 0; i < 32; ++i) dst[i] = __float2bfloat16_rn(acc[i] * inv);
        }
        if ((tid % 16) == 0 && p.lse) p.lse[(size_t)r * p.H + h] = lse_v;
    }
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t s) {
    dim3 grid((a.H + kHG - 1) / kHG, a.num_splits, a.B * a.Sq);
    decode_simt_kernel<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace mla
