// fp8_expand.cu -- first stage of the FP8-cache decode: expand the pages a batch reads from the
// 584-byte FP8 rows into exact bf16 rows plus per-token scales.
//
// The FP8 row ([vLLM-MLA, cache shape section]; [Triton-MLA, FP8 section]) is 576 OCP E4M3
// bytes, then k_scale (fp32, byte 576) and v_scale (fp32, byte 580): K = e4m3 * k_scale over the
// 576 dims, V = e4m3 * v_scale over the first 512. A 584-byte row stride is not a multiple of 16
// bytes, so the tensor-memory-access unit cannot tile these rows, and every second row starts
// 8 bytes off a 16-byte boundary. This kernel therefore re-lays the rows out, page by page, as
// 1152-byte bf16 rows holding the e4m3 values exactly (e4m3 -> bf16 is lossless) and one
// (k_scale, v_scale) pair per token. The decode kernel then reads them with TMA like a bf16
// cache and applies the two scales in fp32 where they belong: k_scale to the token's score,
// v_scale to its softmax weight before the PV product.
//
// Layout written (dense, indexed by request, not by physical block):
//   expanded row (b * mp + pg) * 64 + r  <-  cache[block_table[b, pg], r]      [*, 576] bf16
//   scales[same index]                    =  (k_scale, v_scale)                  [*, 2]   fp32
// for every page pg < ceil(min(seq_lens[b], max_blocks * 64) / 64). A block-table entry outside
// [0, num_blocks) raises MLA_DEV_BAD_BLOCK_ID and expands to zeros.
#include <cuda_fp16.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace mla {
namespace {

constexpr int kWarps = 8;

__global__ void __launch_bounds__(kWarps * 32) fp8_expand_kernel(DecodeArgs p) {
    ptx::griddep_launch_dependents();
    ptx::griddep_wait();  // it overwrites workspace the preceding kernel may still read
    const int b = blockIdx.x, pg = blockIdx.y;
    int seq = p.seq_lens[b];
    const int cap = p.max_blocks * kPage;
    seq = seq < 0 ? 0 : (seq > cap ? cap : seq);
    if (pg * kPage >= seq) return;
    const int32_t blk = p.block_table[(size_t)b * p.max_blocks + pg];
    const bool bad = blk < 0 || (int64_t)blk >= p.num_blocks;
    if (bad && threadIdx.x == 0 && p.dev_status) atomicOr(p.dev_status, MLA_DEV_BAD_BLOCK_ID);
    const size_t out_row0 = ((size_t)b * p.fp8_mp + pg) * kPage;
    const uint8_t* src_page = p.cache + (bad ? 0 : (size_t)blk * kPage * kFp8RowBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int r = warp; r < kPage; r += kWarps) {
        const uint8_t* src = src_page + (size_t)r * kFp8RowBytes;
        uint4* dst = reinterpret_cast<uint4*>(p.fp8_rows + (out_row0 + r) * kD);
        // 72 eight-byte chunks of e4m3 (rows are 8-byte aligned: 584 = 73 * 8), then the scales
        for (int k = lane; k < 72; k += 32) {
            uint2 v = bad ? make_uint2(0, 0) : *reinterpret_cast<const uint2*>(src + 8 * k);
            dst[k] = make_uint4(ptx::e4m3x2_to_bf16x2(v.x & 0xffffu), ptx::e4m3x2_to_bf16x2(v.x >> 16),
                                ptx::e4m3x2_to_bf16x2(v.y & 0xffffu), ptx::e4m3x2_to_bf16x2(v.y >> 16));
        }
        if (lane == 0) {
            float2 sc = make_float2(0.f, 0.f);
            if (!bad) sc = *reinterpret_cast<const float2*>(src + kD);
            reinterpret_cast<float2*>(p.fp8_scales)[out_row0 + r] = sc;
        }
    }
}

}  // namespace

cudaError_t launch_fp8_expand(const DecodeArgs& a, cudaStream_t s) {
    if (a.B == 0 || a.fp8_mp == 0) return cudaSuccess;
    dim3 grid(a.B, a.fp8_mp);
    return launch_pdl(fp8_expand_kernel, grid, dim3(kWarps * 32), 0, s, a);
}

}  // namespace mla
