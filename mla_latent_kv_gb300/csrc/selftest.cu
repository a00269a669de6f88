// selftest.cu -- mla_selftest_wait_timeout: the bounded-wait path, exercised on purpose.
//
// Every pipeline wait in this library's kernels goes through ptx::wait_bar(), which gives up after
// a fixed time, raises MLA_DEV_WAIT_TIMEOUT in the caller's status word and returns false, so that
// a kernel whose producer never delivers winds down instead of hanging the GPU. This entry point
// runs that same wait on an mbarrier that nothing ever arrives on: the wait must run out, report
// the timeout and let the kernel exit, and the context must stay usable for the next call.
// mla_selftest_e4m3_widen runs the FP8 decode kernel's e4m3 -> bf16 widening on all 256 codes.
#include <cuda_runtime.h>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace {

using namespace mla::ptx;

// One thread waits for phase 0 of a fresh barrier whose single expected arrival never comes.
// out[0]: milliseconds of global time the wait took; out[1]: what wait_bar returned (0 or 1).
__global__ void wait_timeout_kernel(int32_t* dev_status, int32_t* out) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        bar_init(smem_addr(&bar), 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint64_t t0 = global_timer_ns();
        const bool ok = wait_bar(smem_addr(&bar), 0, &abort_flag, dev_status);
        const uint64_t t1 = global_timer_ns();
        out[0] = (int32_t)((t1 - t0) / 1000000ull);
        out[1] = ok ? 1 : 0;
    }
}

}  // namespace

extern "C" mla_status mla_selftest_wait_timeout(int32_t* dev_status, int32_t* out, mla_stream_t stream) {
    if (dev_status == nullptr || out == nullptr)
        return mla::set_error(MLA_ERR_INVALID_ARG, "mla_selftest_wait_timeout: dev_status and out are required");
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(dev_status, out);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return mla::set_error(MLA_ERR_CUDA, "mla_selftest_wait_timeout: launch: %s", cudaGetErrorString(e));
    return MLA_OK;
}

namespace {

using namespace mla::ptx;

// Code c = 4 * threadIdx.x + k (k = 0..3) through the same widening the FP8 decode kernel uses.
__global__ void e4m3_widen_kernel(uint16_t* out) {
    const uint32_t c0 = 4u * threadIdx.x;
    const uint32_t w = c0 | (c0 + 1) << 8 | (c0 + 2) << 16 | (c0 + 3) << 24;
    uint32_t lo, hi;
    e4m3x4_to_bf16x4(w, lo, hi);
    out[c0] = (uint16_t)(lo & 0xffffu);
    out[c0 + 1] = (uint16_t)(lo >> 16);
    out[c0 + 2] = (uint16_t)(hi & 0xffffu);
    out[c0 + 3] = (uint16_t)(hi >> 16);
}

}  // namespace

extern "C" mla_status mla_selftest_e4m3_widen(uint16_t* out, mla_stream_t stream) {
    if (out == nullptr) return mla::set_error(MLA_ERR_INVALID_ARG, "mla_selftest_e4m3_widen: out is required");
    e4m3_widen_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(out);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return mla::set_error(MLA_ERR_CUDA, "mla_selftest_e4m3_widen: launch: %s", cudaGetErrorString(e));
    return MLA_OK;
}
