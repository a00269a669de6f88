// cache_write.cu -- the KV cache write that precedes decode: each new token's row
// [kv_c (512) || k_pe (64)] is stored at its slot (block * 64 + in-page offset), copied as bf16 or
// quantised on the fly to the 584-byte FP8 row ([vLLM-MLA, cache write section]: latent and
// k_pe land in one kernel, at slot_mapping; [vLLM-MLA, cache shape and numbers sections]: 576
// e4m3 bytes, then k_scale and v_scale as fp32).
//
// One warp per four tokens, all their loads issued first. FP8: the row's scale is the static
// kv_scale, or amax(|row|) / 448 (a warp max over the 576 values; 1 for an all-zero row); each
// value is multiplied by the correctly rounded reciprocal of the scale and converted with
// round-to-nearest-even and saturation at +-448, so the stored bytes are exactly those of the
// definition. HBM-bound: 1152 bytes read and 584 (or 1152) written per token.
#include "internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;
constexpr int kTok = 4;  // tokens per warp: all their loads are in flight before any is used

// Two binary32 values -> two OCP E4M3 bytes (lo at the lower address), nearest even, saturating.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(kWarps * 32)
    cache_write_kernel(const uint16_t* __restrict__ kv_c, int64_t st_c, const uint16_t* __restrict__ k_pe,
                       int64_t st_pe, const int64_t* __restrict__ slots, int T, uint8_t* __restrict__ cache,
                       int fp8, int64_t num_blocks, float kv_scale, int32_t* dev_status) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();  // the rows come from, and the cache may still be read by, earlier kernels
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = ((int64_t)blockIdx.x * kWarps + warp) * kTok;
    // the row as 72 chunks of 8 bf16: chunks 0-63 from kv_c, 64-71 from k_pe; lane takes
    // chunks lane, lane + 32, lane + 64
    int64_t slot[kTok];
    uint4 v[kTok][3];
#pragma unroll
    for (int u = 0; u < kTok; ++u) {
        const int64_t t = t0 + u;
        slot[u] = t < T ? slots[t] : -1;
        if (slot[u] >= num_blocks * kPage) {
            if (lane == 0 && dev_status) atomicOr(dev_status, MLA_DEV_BAD_SLOT);
            slot[u] = -1;
        }
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int k = lane + 32 * i;
            v[u][i] = make_uint4(0, 0, 0, 0);
            if (slot[u] >= 0 && k < 72)
                v[u][i] = k < 64 ? *reinterpret_cast<const uint4*>(kv_c + t * st_c + 8 * k)
                                 : *reinterpret_cast<const uint4*>(k_pe + t * st_pe + 8 * (k - 64));
        }
    }
#pragma unroll
    for (int u = 0; u < kTok; ++u) {
        if (slot[u] < 0) continue;  // padding, past T, or beyond the cache (warp-uniform)
        if (!fp8) {
            uint4* dst = reinterpret_cast<uint4*>(cache + slot[u] * kBf16RowBytes);
#pragma unroll
            for (int i = 0; i < 3; ++i)
                if (lane + 32 * i < 72) dst[lane + 32 * i] = v[u][i];
            continue;
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const uint32_t w[4] = {v[u][i].x, v[u][i].y, v[u][i].z, v[u][i].w};
#pragma unroll
            for (int j = 0; j < 4; ++j)
                amax = fmaxf(amax, fmaxf(fabsf(ptx::bf16_lo_f(w[j])), fabsf(ptx::bf16_hi_f(w[j]))));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float scale = kv_scale > 0.f ? kv_scale : (amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f);
        const float inv = __frcp_rn(scale);
        uint8_t* dst = cache + slot[u] * kFp8RowBytes;  // 584-byte rows are 8-byte aligned
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int k = lane + 32 * i;
            if (k >= 72) continue;
            const uint32_t w[4] = {v[u][i].x, v[u][i].y, v[u][i].z, v[u][i].w};
            uint32_t b[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                b[j] = f32x2_to_e4m3x2(__fmul_rn(ptx::bf16_lo_f(w[j]), inv), __fmul_rn(ptx::bf16_hi_f(w[j]), inv));
            reinterpret_cast<uint2*>(dst)[k] = make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
        }
        if (lane == 0) *reinterpret_cast<float2*>(dst + kD) = make_float2(scale, scale);
    }
}

}  // namespace

cudaError_t launch_cache_write(const uint16_t* kv_c, int64_t st_c, const uint16_t* k_pe, int64_t st_pe,
                               const int64_t* slots, int T, uint8_t* cache, int kv_dtype, int64_t num_blocks,
                               float kv_scale, int32_t* dev_status, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((T + kWarps * kTok - 1) / (kWarps * kTok));
    return launch_pdl(cache_write_kernel, dim3(blocks), dim3(kWarps * 32), 0, s, kv_c, st_c, k_pe, st_pe, slots, T,
                      cache, kv_dtype == MLA_KV_FP8_E4M3_SCALED ? 1 : 0, num_blocks, kv_scale, dev_status);
}

}  // namespace mla
