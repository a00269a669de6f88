// noalloc.cu -- mla_decode_noalloc: the decode entry point for callers that cannot allocate.
//
// Some callers cannot allocate device memory at the moment they decode: serving loops that run
// under a fixed device-memory budget with every buffer made at start-up, host runtimes that
// forbid device allocations after their initialisation, and call paths with no way to carry a
// workspace pointer down to the attention call. For them this entry point takes the split-KV
// scratch (the per-split partial outputs and LSEs) from one file-scope device array instead of
// a caller-provided workspace, so a decode call needs only its inputs and outputs.
//
// The array is kNoAllocScratchBytes (64 MiB) on every device that uses it and stays there until
// the process exits. All calls share it: calls whose kernels overlap on the GPU (e.g. on two
// streams) race on it and must be serialised by the caller. Its contents persist from call to
// call; nothing in it needs to start at zero, because every partial the merge reads is written
// by the same call's decode kernel first.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself. Host code must not pass &g_noalloc_scratch to a kernel: on the host this
// name is only a stand-in for the symbol; the device address comes from cudaGetSymbolAddress.
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mutex;
struct ScratchEntry {
    unsigned long long ctx_id;  // unique id of the context the address belongs to (0: unknown)
    void* addr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Unique id of the calling thread's current CUDA context, or 0 when there is none or the driver
// does not offer the query. The two driver entry points are fetched once through the runtime,
// so the library keeps no link-time dependency on libcuda.
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

unsigned long long current_context_id() {
    std::call_once(g_ctx_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
    });
    if (!g_ctx_current || !g_ctx_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the scratch array in the current device's context. The first call on a
// device does the lookup (which may load this file's device code onto that device); make that
// first call before any stream capture. Later calls reuse the address while the device's
// context stays the same; after a device reset (a new primary context, with a new copy of the
// array) the next call looks the address up again.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    const unsigned long long id = current_context_id();
    if (g_scratch[dev].addr == nullptr || id == 0 || g_scratch[dev].ctx_id != id) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch[dev].addr = p;
        g_scratch[dev].ctx_id = current_context_id();  // the lookup makes the primary context current
    }
    *out = g_scratch[dev].addr;
    return cudaSuccess;
}

}  // namespace

extern "C" size_t mla_decode_noalloc_max_workspace_bytes(void) { return kNoAllocScratchBytes; }

extern "C" mla_status mla_decode_noalloc(const void* q, const void* kv_cache, mla_kv_dtype kv_dtype,
                                         int64_t num_blocks, const int32_t* block_table, int max_blocks,
                                         const int32_t* seq_lens, int max_seq_len, int B, int Sq, int H,
                                         float scale, int num_splits, void* o_latent, mla_dtype o_dtype,
                                         float* lse, int32_t* dev_status, mla_stream_t stream) {
    // Refuse a split plan whose partials do not fit, before anything touches a device (argument
    // errors of other kinds are reported by mla_decode below).
    if (B > 0 && Sq > 0 && H >= 1 && H <= MLA_MAX_HEADS && num_splits >= -1 && max_seq_len >= 0) {
        const int S = mla_resolve_num_splits(num_splits, B, Sq, H, max_seq_len);
        if (S >= 1) {
            const size_t need = mla_decode_workspace_bytes_kv(kv_dtype, B, Sq, H, S, max_seq_len);
            if (need > kNoAllocScratchBytes)
                return mla::set_error(MLA_ERR_WORKSPACE_TOO_SMALL,
                                      "mla_decode_noalloc: %d splits x B*Sq=%lld x H=%d need %zu bytes of "
                                      "scratch, more than its fixed %zu bytes; use fewer splits or mla_decode",
                                      S, (long long)B * Sq, H, need, kNoAllocScratchBytes);
        }
    }
    void* ws = nullptr;
    const cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess)
        return mla::set_error(MLA_ERR_CUDA, "mla_decode_noalloc: address of the scratch array: %s (%s)",
                              cudaGetErrorName(e), cudaGetErrorString(e));
    return mla_decode(q, kv_cache, kv_dtype, num_blocks, block_table, max_blocks, seq_lens, max_seq_len, B, Sq, H,
                      scale, num_splits, ws, kNoAllocScratchBytes, o_latent, o_dtype, lse, dev_status, stream);
}
