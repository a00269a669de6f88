// gemm_sm103.cu -- the two per-head batched GEMMs of the absorbed MLA path on the 5th-generation
// tensor cores (tcgen05 + TMEM accumulators, weights staged by TMA).
//
//   absorb:   q[t, h, 0:512]   = q_nope[t, h, :] . W_UK_T[h]      (K = 128, M = 512)
//             q[t, h, 512:576] = q_pe[t, h, :]                      (copied, fused concat)
//             ([vLLM-MLA, two-algorithms section]: bmm of q_nope with W_UK_T, then concat q_pe;
//              [TRT-TP, absorption section]: fused_q = [q_nope W_kb^T || q_pe])
//   out_proj: o[t, h, :]        = o_latent[t, h, :] . W_UV[h]       (K = 512, M = 128)
//             ([vLLM-MLA, two-algorithms section]: the V up-projection after the latent kernel)
//
// Both are D[t, h, m] = sum_k W[h][k][m] * X[t, h, k] with the weights stored [H][K][M] (m
// fastest) and few tokens T (decode batches). The kernel runs them "swap-AB": the MMA's M side is
// the weight's m (128 rows per CTA, the full tensor-core height) and its N side is the token
// count, so a batch of a handful of tokens does not waste a 128-row MMA. A = W[h]^T is read
// MN-major straight from the weight layout; B = X^T is K-major.
//
// Work split: one CTA per (128-row m tile, head, tile of up to 128 tokens). K is walked in
// 64-deep chunks through a ring of shared-memory stages:
//   warp 4 lane 0  TMA of the weight chunk (two 64 x 64 boxes, 128-byte swizzle) per stage
//   warps 0-3      load the activation chunk with plain 16-byte loads, convert it to bf16 and
//                  write it in the swizzled K-major layout the MMA reads; an fp32 activation
//                  (out_proj's o_latent) is split into bf16 hi + lo parts, x = hi + lo to ~2^-17
//                  relative, and both are multiplied (two MMAs per K step), so the fp32 input is
//                  not truncated to bf16
//   warp 5 lane 0  issues the tcgen05.mma (M = 128, N = token tile, K = 16 per instruction),
//                  commits each stage back to its producers and, at the end, the accumulator
//   warps 0-3      epilogue: tcgen05.ld of the fp32 accumulator (lane = m, column = token) and
//                  the stores to the output (rounded once to bf16 where the output is bf16)
// The weights (16.8 MB per GEMM at H = 128) are read from HBM once per token tile; the kernel is
// bound by that stream, not by the tensor cores.
#include <cuda.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mla {

cudaError_t encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                        bool swizzle128);

namespace {

using namespace ptx;

constexpr int kThreads = 192;      // warps 0-3 loaders + epilogue, warp 4 TMA + TMEM, warp 5 MMA
constexpr int kKChunk = 64;        // K rows per stage
constexpr int kMaxStages = 4;
constexpr int kWBox = 64 * 64 * 2; // one 64 (m) x 64 (k) bf16 box = 8 KB
constexpr int kWStage = 2 * kWBox; // 128 m rows per CTA

struct HeadGemmArgs {
    int T, H, K;
    int n_tile;          // tokens per CTA: multiple of 16, <= 128
    int stages;          // ring depth, <= kMaxStages
    const void* x;       // activations, element (t, h, k) at x[t * x_st + h * x_sh + k]
    int x_f32;           // 1: fp32 (split into bf16 hi + lo), 0: bf16
    int64_t x_st, x_sh;
    void* out;           // element (t, h, m) at out[t * out_st + h * out_sh + m]
    int out_f32;
    int64_t out_st, out_sh;
    const uint16_t* q_pe; // absorb only (may be null): copied to out[t, h, 512:576] by m tile 0
    int64_t pe_st, pe_sh;
};

__device__ __forceinline__ uint32_t bf16_bits_rn(float x) { return pack_bf16x2(x, 0.f) & 0xffffu; }

__device__ __forceinline__ void store_out(const HeadGemmArgs& p, int t, int m, float v) {
    const int64_t off = (int64_t)t * p.out_st + (int64_t)blockIdx.y * p.out_sh + m;
    if (p.out_f32)
        static_cast<float*>(p.out)[off] = v;
    else
        static_cast<uint16_t*>(p.out)[off] = (uint16_t)bf16_bits_rn(v);
}

__global__ void __launch_bounds__(kThreads, 1)
    head_gemm_kernel(const __grid_constant__ CUtensorMap w_map, const HeadGemmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[3 * kMaxStages + 1];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y;
    const int m0 = blockIdx.x * 128;
    const int n0 = blockIdx.z * p.n_tile;
    const int NT = p.n_tile;
    const int ST = p.stages;
    const int nchunks = p.K / kKChunk;
    const uint32_t x_panel = (uint32_t)NT * 128u;  // one 64-deep K-major panel of NT rows
    const uint32_t stage_bytes = kWStage + (p.x_f32 ? 2u : 1u) * x_panel;

    const uint32_t sbase = (smem_addr(smem_raw) + 1023u) & ~1023u;
    uint8_t* const sgen = smem_raw + (sbase - smem_addr(smem_raw));
    const uint32_t bar0 = smem_addr(&bars[0]);
    auto FULL_W = [&](int s) { return bar0 + 8u * s; };
    auto FULL_X = [&](int s) { return bar0 + 8u * (kMaxStages + s); };
    auto EMPTY = [&](int s) { return bar0 + 8u * (2 * kMaxStages + s); };
    const uint32_t DONE = bar0 + 8u * (3 * kMaxStages);

    const uint32_t tmem_cols = NT <= 32 ? 32u : (NT <= 64 ? 64u : 128u);
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < kMaxStages; ++s) {
            bar_init(FULL_W(s), 1);
            bar_init(FULL_X(s), 128);
            bar_init(EMPTY(s), 1);
        }
        bar_init(DONE, 1);
        fence_barrier_init();
    }
    if (warp == 4) {
        tmem_alloc(smem_addr(&tmem_slot), tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int* abort_p = &abort_flag;

    if (warp == 4) {
        // ---- weight producer ------------------------------------------------------------
        if (lane == 0) {
            tma_prefetch_desc(&w_map);
            int last_issued[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) last_issued[s] = -1;
            for (int c = 0; c < nchunks; ++c) {
                const int s = c % ST;
                if (c >= ST && !wait_bar(EMPTY(s), ((c / ST) - 1) & 1, abort_p, nullptr)) break;
                const uint32_t dst = sbase + s * stage_bytes;
                bar_arrive_expect_tx(FULL_W(s), kWStage);
                const int y = h * p.K + c * kKChunk;
                tma_load_2d(dst, &w_map, FULL_W(s), m0, y);
                tma_load_2d(dst + kWBox, &w_map, FULL_W(s), m0 + 64, y);
                last_issued[s] = c;
            }
            // Wind-down after an abort: let the copies still in flight land before the CTA
            // leaves (bounded as well).
            if (*abort_p) {
                int dummy = 0;
                for (int s = 0; s < kMaxStages; ++s)
                    if (last_issued[s] >= 0) wait_bar(FULL_W(s), (last_issued[s] / ST) & 1, &dummy, nullptr);
            }
        }
    } else if (warp == 5) {
        // ---- MMA issuer -----------------------------------------------------------------
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, NT, true, false);
            bool ok = true;
            for (int c = 0; c < nchunks && ok; ++c) {
                const int s = c % ST;
                const uint32_t par = (c / ST) & 1;
                ok = wait_bar(FULL_W(s), par, abort_p, nullptr) && wait_bar(FULL_X(s), par, abort_p, nullptr);
                if (!ok) break;
                tc_fence_after();
                const uint32_t wb = sbase + s * stage_bytes;
                const uint32_t xb = wb + kWStage;
#pragma unroll
                for (int kk = 0; kk < kKChunk / 16; ++kk) {
                    const uint64_t ad = smem_desc_sw128(wb + kk * 2048, kWBox, 1024);
                    const uint64_t bd = smem_desc_sw128(xb + kk * 32, 16, 1024);
                    mma_ss(tmem, ad, bd, idesc, (c | kk) != 0);
                }
                if (p.x_f32) {
#pragma unroll
                    for (int kk = 0; kk < kKChunk / 16; ++kk) {
                        const uint64_t ad = smem_desc_sw128(wb + kk * 2048, kWBox, 1024);
                        const uint64_t bd = smem_desc_sw128(xb + x_panel + kk * 32, 16, 1024);
                        mma_ss(tmem, ad, bd, idesc, 1u);
                    }
                }
                mma_commit(EMPTY(s));
            }
            if (ok) mma_commit(DONE);
        }
    } else {
        // ---- activation loaders (warps 0-3) ---------------------------------------------
        const int tid = threadIdx.x;  // 0..127
        const int items = NT * 8;     // (row, 16-byte chunk) pairs of one 64-deep panel
        for (int c = 0; c < nchunks; ++c) {
            const int s = c % ST;
            if (c >= ST && !wait_bar(EMPTY(s), ((c / ST) - 1) & 1, abort_p, nullptr)) break;
            uint8_t* const xg = sgen + s * stage_bytes + kWStage;
            const int k0 = c * kKChunk;
            for (int i = tid; i < items; i += 128) {
                const int r = i >> 3, c16 = i & 7;
                const int t = n0 + r;
                uint4 hi = make_uint4(0, 0, 0, 0), lo = make_uint4(0, 0, 0, 0);
                if (t < p.T) {
                    const int64_t off = (int64_t)t * p.x_st + (int64_t)h * p.x_sh + k0 + 8 * c16;
                    if (p.x_f32) {
                        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + off);
                        const float4 a = src[0], b = src[1];
                        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            hw[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
                            lw[j] = pack_bf16x2(v[2 * j] - bf16_lo_f(hw[j]), v[2 * j + 1] - bf16_hi_f(hw[j]));
                        }
                        hi = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        lo = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    } else {
                        hi = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) + off);
                    }
                }
                const uint32_t so = (uint32_t)r * 128u + (uint32_t)((c16 ^ (r & 7)) * 16);
                *reinterpret_cast<uint4*>(xg + so) = hi;
                if (p.x_f32) *reinterpret_cast<uint4*>(xg + x_panel + so) = lo;
            }
            fence_proxy_async_cta();
            bar_arrive(FULL_X(s));
        }
        // Fused concat of the rope part (absorb only): q[t, h, 512:576] = q_pe[t, h, :].
        if (p.q_pe != nullptr && blockIdx.x == 0) {
            for (int i = tid; i < NT * 8; i += 128) {
                const int r = i >> 3, c16 = i & 7;
                const int t = n0 + r;
                if (t >= p.T) continue;
                const uint4 v = *reinterpret_cast<const uint4*>(p.q_pe + (int64_t)t * p.pe_st + (int64_t)h * p.pe_sh +
                                                                8 * c16);
                *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + (int64_t)t * p.out_st +
                                          (int64_t)h * p.out_sh + kL + 8 * c16) = v;
            }
        }
        // ---- epilogue: TMEM lane = m, column = token ------------------------------------
        const bool ok = wait_bar(DONE, 0, abort_p, nullptr);
        tc_fence_after();
        const int m = m0 + warp * 32 + lane;
        for (int j0 = 0; j0 < NT; j0 += 32) {
            uint32_t r[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)j0, r);
            tmem_wait_ld();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int t = n0 + j0 + jj;
                if (j0 + jj < NT && t < p.T)
                    store_out(p, t, m, ok ? __uint_as_float(r[jj]) : __int_as_float(0x7fc00000));
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 4) tmem_dealloc(tmem, tmem_cols);
}

int pick_n_tile(int T) {
    const int t16 = ((T + 15) / 16) * 16;
    return t16 < 128 ? t16 : 128;
}

cudaError_t launch_head_gemm(const HeadGemmArgs& a, const uint16_t* w, int M_total, cudaStream_t s) {
    CUtensorMap map;
    const uint64_t dims[2] = {(uint64_t)M_total, (uint64_t)a.H * a.K};
    const uint64_t strides[1] = {(uint64_t)M_total * 2};
    const uint32_t box[2] = {64, 64};
    cudaError_t e = encode_tmap(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, dims, strides, box, true);
    if (e != cudaSuccess) return e;
    const int stage_bytes = kWStage + (a.x_f32 ? 2 : 1) * a.n_tile * 128;
    const int smem = a.stages * stage_bytes + 1024;
    e = cudaFuncSetAttribute(head_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(M_total / 128, a.H, (a.T + a.n_tile - 1) / a.n_tile);
    head_gemm_kernel<<<grid, kThreads, smem, s>>>(map, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_absorb_sm103(const uint16_t* q_nope, int64_t snt, int64_t snh, const uint16_t* q_pe,
                                int64_t spt, int64_t sph, const uint16_t* w_uk_t, uint16_t* q_out, int T, int H,
                                cudaStream_t s) {
    HeadGemmArgs a{};
    a.T = T;
    a.H = H;
    a.K = kP;
    a.n_tile = pick_n_tile(T);
    a.stages = 2;
    a.x = q_nope;
    a.x_f32 = 0;
    a.x_st = snt;
    a.x_sh = snh;
    a.out = q_out;
    a.out_f32 = 0;
    a.out_st = (int64_t)H * kD;
    a.out_sh = kD;
    a.q_pe = q_pe;
    a.pe_st = spt;
    a.pe_sh = sph;
    return launch_head_gemm(a, w_uk_t, kL, s);
}

cudaError_t launch_out_proj_sm103(const void* o_latent, int in_dtype, const uint16_t* w_uv, void* o,
                                  int out_dtype, int T, int H, cudaStream_t s) {
    HeadGemmArgs a{};
    a.T = T;
    a.H = H;
    a.K = kL;
    a.n_tile = pick_n_tile(T);
    a.stages = kMaxStages;
    a.x = o_latent;
    a.x_f32 = in_dtype == MLA_DT_F32;
    a.x_st = (int64_t)H * kL;
    a.x_sh = kL;
    a.out = o;
    a.out_f32 = out_dtype == MLA_DT_F32;
    a.out_st = (int64_t)H * kV;
    a.out_sh = kV;
    a.q_pe = nullptr;
    return launch_head_gemm(a, w_uv, kV, s);
}

}  // namespace mla
