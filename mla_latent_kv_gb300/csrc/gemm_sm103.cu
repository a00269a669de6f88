// gemm_sm103.cu -- the two per-head batched GEMMs of the absorbed MLA path on the 5th-generation
// tensor cores (tcgen05 + TMEM accumulators, all operands staged by TMA).
//
//   absorb:   q[t, h, 0:512]   = q_nope[t, h, :] . W_UK_T[h]      (K = 128, M = 512)
//             q[t, h, 512:576] = q_pe[t, h, :]                      (copied, fused concat)
//             ([vLLM-MLA, two-algorithms section]: bmm of q_nope with W_UK_T, then concat q_pe;
//              [TRT-TP, absorption section]: fused_q = [q_nope W_kb^T || q_pe])
//   out_proj: o[t, h, :]        = o_latent[t, h, :] . W_UV[h]       (K = 512, M = 128)
//             ([vLLM-MLA, two-algorithms section]: the V up-projection after the latent kernel)
//   up_proj:  k_nope[j, h, :]   = c[j, :] . W_UK_T[h]^T, v[j, h, :] = c[j, :] . W_UV[h]
//             (K = 512, M = 128; [vLLM-MLA, Prefill section]: kv_b_proj of the gathered latent
//              rows; the activation row is shared by all heads, and W_UK_T[h] is read K-major)
//
// Both are D[t, h, m] = sum_k W[h][k][m] * X[t, h, k] with the weights stored [H][K][M] (m
// fastest) and few tokens T (decode batches). The kernel runs them "swap-AB": the MMA's M side is
// the weight's m (128 rows per work unit, the full tensor-core height) and its N side is the
// token count, so a batch of a handful of tokens does not waste a 128-row MMA. A = W[h]^T is read
// MN-major straight from the weight layout; B = X^T is K-major.
//
// A work unit is (128-row m tile, head, tile of up to 128 tokens). The kernel is persistent: one
// CTA per SM walks units u = blockIdx.x, + gridDim.x, ..., and every role streams across unit
// boundaries, so the weight stream (16.8 MB per GEMM at H = 128, read once per token tile) never
// waits for an epilogue:
//   warp 4 lane 0  TMA producer: per 64-deep K chunk, two 64 x 64 weight boxes and the
//                  activation box(es) into a ring stage (128-byte swizzle for bf16 operands)
//   warps 6-9      fp32 activations only (out_proj's o_latent): rewrite each staged fp32 chunk
//                  in place as bf16 hi + lo panels, x = hi + lo to ~2^-17 relative; both panels
//                  are multiplied (two MMAs per K step), so the fp32 input is not cut to bf16
//   warp 5 lane 0  tcgen05.mma (M = 128, N = token tile, K = 16 per instruction) into one of two
//                  TMEM accumulators, commits each ring stage back to the producer and each
//                  finished accumulator to the epilogue
//   warps 0-3      epilogue: tcgen05.ld of the fp32 accumulator (lane = m, column = token) in
//                  32-token slices, each written (rounded once where the output is bf16) to a
//                  double-buffered [32 tokens][128 m] shared tile that one thread sends out with
//                  a TMA store; then frees the accumulator for the unit after next
//   warps 6-9      bf16 activations (absorb): the fused q_pe copy, off the epilogue's path
// Every wait is bounded; a CTA that gives up writes NaN to the outputs it owns.
#include <cuda.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mla {

cudaError_t encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                        const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                        bool swizzle128);

namespace {

using namespace ptx;

constexpr int kThreads = 320;       // warps 0-3 epilogue, 4 TMA + TMEM, 5 MMA, 6-9 fp32 split
constexpr int kKChunk = 64;         // K rows per ring stage
constexpr int kStages = 4;          // ring depth (at most; see HeadGemmArgs::stages)
constexpr int kWBox = 64 * 64 * 2;  // one 64 (m) x 64 (k) bf16 box = 8 KB
constexpr int kWStage = 2 * kWBox;  // 128 m rows per unit
constexpr uint32_t kBarConvert = 1; // named barrier of the fp32-split warps
constexpr uint32_t kBarEpi = 2;     // named barrier of the epilogue warps
constexpr int kSlice = 32;          // tokens per epilogue slice (one tcgen05.ld 32x32b.x32)

struct HeadGemmArgs {
    int T, H, K, M_total;
    int n_tile;              // tokens per unit: multiple of 16, <= 128 (256 for bf16 activations
                             // without the q_pe copy: the up-projection of many rows)
    int stages;              // ring depth, <= kStages
    int x_f32;               // activations fp32 (split into bf16 hi + lo) or bf16
    void* out;               // element (t, h, m) at out[t * out_st + h * out_sh + m]
    int out_f32;
    int64_t out_st, out_sh;
    const uint16_t* q_pe;    // absorb only (may be null): copied to out[t, h, 512:576] by m tile 0
    int64_t pe_st, pe_sh;
    int x_shared;            // one activation row per token, used by every head (up_proj)
    int w_kmajor;            // weights stored [H][M][K] (k fastest) instead of [H][K][M]
    int64_t out_m_ext;       // extent of the output's m dimension (0: out_sh, m runs up to the head stride)
};

struct Unit {
    int mt, h, nt;
};

__device__ __forceinline__ Unit unit_of(int u, int n_tiles, int m_tiles) {
    Unit r;
    r.nt = u % n_tiles;
    const int rest = u / n_tiles;
    r.mt = rest % m_tiles;
    r.h = rest / m_tiles;
    return r;
}

__global__ void __launch_bounds__(kThreads, 2)
    head_gemm_kernel(const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap x_map,
                     const __grid_constant__ CUtensorMap o_map, const HeadGemmArgs p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[3 * kStages + 4];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NT = p.n_tile;
    const int ST = p.stages;
    const int n_tiles = (p.T + NT - 1) / NT;
    const int m_tiles = p.M_total / 128;
    const int units = n_tiles * m_tiles * p.H;
    const int nchunks = p.K / kKChunk;
    const uint32_t x_panel = (uint32_t)NT * 128u;  // one 64-deep bf16 K-major panel of NT rows
    const uint32_t x_bytes = (p.x_f32 ? 2u : 1u) * x_panel;
    const uint32_t stage_bytes = kWStage + x_bytes;
    const uint32_t acc_cols = NT <= 32 ? 32u : (NT <= 64 ? 64u : (NT <= 128 ? 128u : 256u));
    const uint32_t out_es = p.out_f32 ? 4u : 2u;
    const uint32_t slice_bytes = kSlice * 128u * out_es;  // [32 tokens][128 m] output tile

    const uint32_t sbase = (smem_addr(smem_raw) + 1023u) & ~1023u;
    uint8_t* const sgen = smem_raw + (sbase - smem_addr(smem_raw));
    const uint32_t bar0 = smem_addr(&bars[0]);
    auto FULL = [&](int s) { return bar0 + 8u * s; };
    auto CONV = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto EMPTY = [&](int s) { return bar0 + 8u * (2 * kStages + s); };
    auto TFULL = [&](int a) { return bar0 + 8u * (3 * kStages + a); };
    auto TEMPTY = [&](int a) { return bar0 + 8u * (3 * kStages + 2 + a); };

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < kStages; ++s) {
            bar_init(FULL(s), 1);
            bar_init(CONV(s), 128);
            bar_init(EMPTY(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            bar_init(TFULL(a), 1);
            bar_init(TEMPTY(a), 128);
        }
        fence_barrier_init();
    }
    if (warp == 4) {
        tmem_alloc(smem_addr(&tmem_slot), 2 * acc_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    volatile int* abort_p = &abort_flag;
    if (threadIdx.x == 0) griddep_launch_dependents();

    if (warp == 4) {
        // ---- TMA producer ---------------------------------------------------------------
        if (lane == 0) {
            tma_prefetch_desc(&w_map);
            tma_prefetch_desc(&x_map);
            // one 128 (m) x 64 (k) weight tile as two 64-row boxes: [K][M] layout boxes are
            // 64 m wide at k rows c*64.., [M][K] layout boxes are 64 k wide at m rows mt*128..
            auto load_w = [&](uint32_t dst, uint32_t bar, const Unit& u, int c) {
                if (p.w_kmajor) {
                    const int wy = u.h * p.M_total + u.mt * 128;
                    tma_load_2d(dst, &w_map, bar, c * kKChunk, wy);
                    tma_load_2d(dst + kWBox, &w_map, bar, c * kKChunk, wy + 64);
                } else {
                    const int wy = u.h * p.K + c * kKChunk;
                    tma_load_2d(dst, &w_map, bar, u.mt * 128, wy);
                    tma_load_2d(dst + kWBox, &w_map, bar, u.mt * 128 + 64, wy);
                }
            };
            // The weights of the first unit's first stages go out before the preceding kernel
            // (which may be writing the activations, or still reading this kernel's output)
            // has finished; everything else waits for it.
            const int pre = blockIdx.x < units ? (nchunks < ST ? nchunks : ST) : 0;
            int last[kStages] = {-1, -1, -1, -1};
            if (pre > 0) {
                const Unit w0 = unit_of(blockIdx.x, n_tiles, m_tiles);
                for (int c = 0; c < pre; ++c) {
                    const uint32_t dst = sbase + c * stage_bytes;
                    bar_arrive_expect_tx(FULL(c), stage_bytes);
                    load_w(dst, FULL(c), w0, c);
                    last[c] = c;
                }
            }
            griddep_wait();
            int g = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const Unit w = unit_of(u, n_tiles, m_tiles);
                for (int c = 0; c < nchunks; ++c, ++g) {
                    const int s = g % ST;
                    if (g >= ST && !wait_bar(EMPTY(s), ((g / ST) - 1) & 1, abort_p, nullptr)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = sbase + s * stage_bytes;
                    if (g >= pre) {  // the first `pre` stages' weights are already on their way
                        bar_arrive_expect_tx(FULL(s), stage_bytes);
                        load_w(dst, FULL(s), w, c);
                    }
                    const int xh = p.x_shared ? 0 : w.h;
                    if (p.x_f32) {
                        tma_load_3d(dst + kWStage, &x_map, FULL(s), c * kKChunk, xh, w.nt * NT);
                        tma_load_3d(dst + kWStage + x_panel, &x_map, FULL(s), c * kKChunk + 32, xh, w.nt * NT);
                    } else {
                        tma_load_3d(dst + kWStage, &x_map, FULL(s), c * kKChunk, xh, w.nt * NT);
                    }
                    last[s] = g;
                }
            }
            if (!ok) {  // let the copies still in flight land before the CTA leaves
                int ignore = 0;
                for (int s = 0; s < kStages; ++s)
                    if (last[s] >= 0) wait_bar(FULL(s), (last[s] / ST) & 1, &ignore, nullptr);
            }
        }
    } else if (warp == 5) {
        // ---- MMA issuer -----------------------------------------------------------------
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, NT, !p.w_kmajor, false);
            int g = 0, i = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++i) {
                const int acc = i & 1;
                if (i >= 2 && !wait_bar(TEMPTY(acc), ((i >> 1) - 1) & 1, abort_p, nullptr)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)acc * acc_cols;
                for (int c = 0; c < nchunks; ++c, ++g) {
                    const int s = g % ST;
                    const uint32_t par = (g / ST) & 1;
                    if (!wait_bar(p.x_f32 ? CONV(s) : FULL(s), par, abort_p, nullptr)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t wb = sbase + s * stage_bytes;
                    const uint32_t xb = wb + kWStage;
#pragma unroll
                    for (int kk = 0; kk < kKChunk / 16; ++kk) {
                        // A = W^T: MN-major (two 64-m boxes, 16 k rows per step) or K-major
                        // (128 m rows of 128 bytes, 32 bytes per step)
                        const uint64_t ad = p.w_kmajor ? smem_desc_sw128(wb + kk * 32, 16, 1024)
                                                       : smem_desc_sw128(wb + kk * 2048, kWBox, 1024);
                        mma_ss(d, ad, smem_desc_sw128(xb + kk * 32, 16, 1024), idesc, (c | kk) != 0);
                        if (p.x_f32) mma_ss(d, ad, smem_desc_sw128(xb + x_panel + kk * 32, 16, 1024), idesc, 1u);
                    }
                    mma_commit(EMPTY(s));
                }
                if (ok) mma_commit(TFULL(acc));
            }
        }
    } else if (warp >= 6) {
        if (!p.x_f32 && p.q_pe != nullptr) {
            // ---- fused concat of the rope part (absorb): q[t, h, 512:576] = q_pe[t, h, :] --
            // The m tiles of a head share its copy (tile mt takes 16-byte items it with
            // it % m_tiles == mt); every load of a unit is issued before its stores, so a unit
            // costs one memory latency.
            const int tid = threadIdx.x - 192;
            griddep_wait();
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                const Unit w = unit_of(u, n_tiles, m_tiles);
                constexpr int kMaxItems = 8;  // NT * 8 items / (128 threads) with NT <= 128
                uint4 v[kMaxItems];
                int64_t dst[kMaxItems];
#pragma unroll
                for (int k = 0; k < kMaxItems; ++k) {
                    const int it = tid + 128 * k;
                    const int rr = it >> 3, c8 = it & 7;
                    const int t = w.nt * NT + rr;
                    dst[k] = -1;
                    if (it < NT * 8 && (it % m_tiles) == w.mt && t < p.T) {
                        v[k] = *reinterpret_cast<const uint4*>(p.q_pe + (int64_t)t * p.pe_st + (int64_t)w.h * p.pe_sh +
                                                               8 * c8);
                        dst[k] = (int64_t)t * p.out_st + (int64_t)w.h * p.out_sh + kL + 8 * c8;
                    }
                }
#pragma unroll
                for (int k = 0; k < kMaxItems; ++k)
                    if (dst[k] >= 0) *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + dst[k]) = v[k];
            }
        }
        // ---- fp32 activations -> bf16 hi / lo panels, in place --------------------------
        if (p.x_f32) {
            const int tid = threadIdx.x - 192;  // 0..127
            const int per = NT / 16;            // (row, 8-value group) items per thread
            int g = 0;
            for (int u = blockIdx.x; u < units; u += gridDim.x) {
                for (int c = 0; c < nchunks; ++c, ++g) {
                    const int s = g % ST;
                    // After an abort the wait returns at once; the loop still runs every named
                    // barrier so that no thread of the group is left waiting on another.
                    wait_bar(FULL(s), (g / ST) & 1, abort_p, nullptr);
                    uint8_t* const xg = sgen + s * stage_bytes + kWStage;
                    // staged layout: two unswizzled boxes [NT][32] fp32 (k 0-31, k 32-63)
                    uint32_t hw[8][4], lw[8][4];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (j < per) {
                            const int it = tid + 128 * j;
                            const int r = it >> 3, c8 = it & 7;
                            const float4* src =
                                reinterpret_cast<const float4*>(xg + (c8 >> 2) * x_panel + r * 128 + (c8 & 3) * 32);
                            const float4 a = src[0], b = src[1];
                            const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                hw[j][q] = pack_bf16x2(v[2 * q], v[2 * q + 1]);
                                lw[j][q] = pack_bf16x2(v[2 * q] - bf16_lo_f(hw[j][q]),
                                                       v[2 * q + 1] - bf16_hi_f(hw[j][q]));
                            }
                        }
                    }
                    named_bar(kBarConvert, 128);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (j < per) {
                            const int it = tid + 128 * j;
                            const int r = it >> 3, c8 = it & 7;
                            const uint32_t so = (uint32_t)r * 128u + (uint32_t)((c8 ^ (r & 7)) * 16);
                            *reinterpret_cast<uint4*>(xg + so) = make_uint4(hw[j][0], hw[j][1], hw[j][2], hw[j][3]);
                            *reinterpret_cast<uint4*>(xg + x_panel + so) =
                                make_uint4(lw[j][0], lw[j][1], lw[j][2], lw[j][3]);
                        }
                    }
                    fence_proxy_async_cta();
                    bar_arrive(CONV(s));
                }
            }
        }
    } else {
        // ---- epilogue (warps 0-3): TMEM lane = m, column = token ------------------------
        const int tid = threadIdx.x;
        griddep_wait();
        const uint32_t stage_base = sbase + ST * stage_bytes;  // two slice tiles
        uint8_t* const stage_gen = sgen + ST * stage_bytes;
        int i = 0, sc = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++i) {
            const Unit w = unit_of(u, n_tiles, m_tiles);
            const int acc = i & 1;
            const bool ok = wait_bar(TFULL(acc), (i >> 1) & 1, abort_p, nullptr);
            tc_fence_after();
            for (int j0 = 0; j0 < NT; j0 += kSlice, ++sc) {
                const int b = sc & 1;
                if (sc >= 2) {  // the TMA store that last read tile b has finished reading it
                    if (tid == 0) bulk_wait_group_read<1>();
                    named_bar(kBarEpi, 128);
                }
                uint32_t r[32];
                if (ok) {
                    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)acc * acc_cols + (uint32_t)j0, r);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) r[jj] = 0x7fc00000u;  // NaN marks a CTA that gave up
                }
                uint8_t* const tile = stage_gen + b * slice_bytes;
                if (p.out_f32) {
                    float* const row = reinterpret_cast<float*>(tile) + tid;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) row[jj * 128] = __uint_as_float(r[jj]);
                } else {
                    uint16_t* const row = reinterpret_cast<uint16_t*>(tile) + tid;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj)
                        row[jj * 128] = (uint16_t)(pack_bf16x2(__uint_as_float(r[jj]), 0.f) & 0xffffu);
                }
                fence_proxy_async_cta();
                named_bar(kBarEpi, 128);
                if (tid == 0) {
                    tma_store_3d(&o_map, stage_base + b * slice_bytes, w.mt * 128, w.h, w.nt * NT + j0);
                    bulk_commit_group();
                }
            }
            tc_fence_before();
            bar_arrive(TEMPTY(acc));
        }
        if (tid == 0) bulk_wait_group<0>();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 4) tmem_dealloc(tmem, 2 * acc_cols);
}

int pick_n_tile(int T) {
    const int t16 = ((T + 15) / 16) * 16;
    return t16 < 128 ? t16 : 128;
}

// x: element (t, h, k) at x[t * x_st + h * x_sh + k], K values per (t, h) row.
cudaError_t launch_head_gemm(HeadGemmArgs a, const uint16_t* w, const void* x, int64_t x_st, int64_t x_sh,
                             cudaStream_t s) {
    CUtensorMap wmap, xmap;
    {
        const uint64_t dims[2] = {a.w_kmajor ? (uint64_t)a.K : (uint64_t)a.M_total,
                                  a.w_kmajor ? (uint64_t)a.H * a.M_total : (uint64_t)a.H * a.K};
        const uint64_t strides[1] = {dims[0] * 2};
        const uint32_t box[2] = {64, 64};
        cudaError_t e = encode_tmap(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w, dims, strides, box, true);
        if (e != cudaSuccess) return e;
    }
    {
        const uint64_t es = a.x_f32 ? 4 : 2;
        const int xh = a.x_shared ? 1 : a.H;
        // A stride of a dimension of extent 1 is never used; give it a harmless legal value.
        if (xh == 1) x_sh = a.K;
        if (a.T == 1) x_st = x_sh * xh;
        const uint64_t dims[3] = {(uint64_t)a.K, (uint64_t)xh, (uint64_t)a.T};
        const uint64_t strides[2] = {(uint64_t)x_sh * es, (uint64_t)x_st * es};
        const uint32_t box[3] = {a.x_f32 ? 32u : 64u, 1u, (uint32_t)a.n_tile};
        cudaError_t e = encode_tmap(&xmap, a.x_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                    3, x, dims, strides, box, !a.x_f32);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap omap;
    {
        const uint64_t es = a.out_f32 ? 4 : 2;
        const int64_t ost = a.T == 1 ? a.out_sh * a.H : a.out_st;
        const uint64_t dims[3] = {(uint64_t)(a.out_m_ext > 0 ? a.out_m_ext : a.out_sh), (uint64_t)a.H, (uint64_t)a.T};
        const uint64_t strides[2] = {(uint64_t)a.out_sh * es, (uint64_t)ost * es};
        const uint32_t box[3] = {128u, 1u, (uint32_t)kSlice};
        cudaError_t e = encode_tmap(&omap, a.out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                    3, a.out, dims, strides, box, false);
        if (e != cudaSuccess) return e;
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int stage_bytes = kWStage + (a.x_f32 ? 2 : 1) * a.n_tile * 128;
    const int smem = a.stages * stage_bytes + 2 * kSlice * 128 * (a.out_f32 ? 4 : 2) + 1024;
    e = cudaFuncSetAttribute(head_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int units = ((a.T + a.n_tile - 1) / a.n_tile) * (a.M_total / 128) * a.H;
    // persistent grid: as many CTAs as fit at once (two per SM when the stages are small, as for
    // absorb), so that the slowest SM's share of units stays small
    int per_sm = 1;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, head_gemm_kernel, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int slots = per_sm * sms;
    const int grid = units < slots ? units : slots;
    return launch_pdl(head_gemm_kernel, dim3(grid), dim3(kThreads), (size_t)smem, s, wmap, xmap, omap, a);
}

}  // namespace

cudaError_t launch_absorb_sm103(const uint16_t* q_nope, int64_t snt, int64_t snh, const uint16_t* q_pe,
                                int64_t spt, int64_t sph, const uint16_t* w_uk_t, uint16_t* q_out, int T, int H,
                                cudaStream_t s) {
    HeadGemmArgs a{};
    a.T = T;
    a.H = H;
    a.K = kP;
    a.M_total = kL;
    a.n_tile = pick_n_tile(T);
    a.stages = 3;  // small stages: two CTAs share an SM
    a.x_f32 = 0;
    a.out = q_out;
    a.out_f32 = 0;
    a.out_st = (int64_t)H * kD;
    a.out_sh = kD;
    a.q_pe = q_pe;
    a.pe_st = spt;
    a.pe_sh = sph;
    return launch_head_gemm(a, w_uk_t, q_nope, snt, snh, s);
}

cudaError_t launch_out_proj_sm103(const void* o_latent, int in_dtype, const uint16_t* w_uv, void* o,
                                  int out_dtype, int T, int H, cudaStream_t s) {
    HeadGemmArgs a{};
    a.T = T;
    a.H = H;
    a.K = kL;
    a.M_total = kV;
    a.n_tile = pick_n_tile(T);
    a.stages = kStages;
    a.x_f32 = in_dtype == MLA_DT_F32;
    a.out = o;
    a.out_f32 = out_dtype == MLA_DT_F32;
    a.out_st = (int64_t)H * kV;
    a.out_sh = kV;
    a.q_pe = nullptr;
    return launch_head_gemm(a, w_uv, o_latent, (int64_t)H * kL, kL, s);
}

// Up-projection of gathered latent rows: out[h, j, m] = sum_l x[j, l] * W[h] with W_UK_T[h]
// ([H][128][512], K-major) for k_nope or W_UV[h] ([H][512][128]) for v; x [rows, 512] bf16
// with row stride x_st; out [H, rows, 128] bf16 (head-major: one head's rows are contiguous).
cudaError_t launch_up_proj_sm103(const uint16_t* x, int64_t x_st, int rows, const uint16_t* w, bool w_is_uk,
                                 uint16_t* out, int H, cudaStream_t s) {
    HeadGemmArgs a{};
    a.T = rows;
    a.H = H;
    a.K = kL;
    a.M_total = 128;
    // 256 tokens per unit when there are enough rows: each unit then reads 128 KB of weights and
    // 256 KB of activations for 2 x 128 x 256 x 512 flops, a quarter less L2 traffic per flop
    // than 128-token units (the two 256-column accumulators fill TMEM: one CTA per SM)
    a.n_tile = rows >= 256 ? 256 : pick_n_tile(rows);
    a.stages = kStages;
    a.x_f32 = 0;
    a.out = out;
    a.out_f32 = 0;
    a.out_st = 128;
    a.out_sh = (int64_t)rows * 128;
    a.out_m_ext = 128;
    a.q_pe = nullptr;
    a.x_shared = 1;
    a.w_kmajor = w_is_uk ? 1 : 0;
    return launch_head_gemm(a, w, x, x_st, kL, s);
}

}  // namespace mla
