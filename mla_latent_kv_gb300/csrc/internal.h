// internal.h -- shared declarations of the CUDA library (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_latent_kv.h"

namespace mla {

constexpr int kL = MLA_KV_LORA_RANK;  // 512 latent dims (also the V width)
constexpr int kR = MLA_ROPE_DIM;      // 64 rope dims
constexpr int kD = MLA_HEAD_DIM;      // 576 = one cached row / one absorbed query
constexpr int kP = MLA_NOPE_DIM;      // 128
constexpr int kV = MLA_V_DIM;         // 128
constexpr int kPage = MLA_PAGE_SIZE;  // 64 tokens per page
constexpr int kBf16RowBytes = 2 * kD; // 1152
constexpr int kFp8RowBytes = kD + 8;  // 584

// Everything a decode launch needs, resolved and validated on the host.
struct DecodeArgs {
    const uint16_t* q;          // bf16 [B, Sq, H, 576]
    const uint8_t* cache;       // [num_blocks, 64, row_bytes]
    int kv_dtype;
    int64_t num_blocks;
    const int32_t* block_table; // [B, max_blocks]
    int max_blocks;
    const int32_t* seq_lens;    // [B]
    int max_seq_len;
    int B, Sq, H;               // requests, uniform query rows per request (1 for packed rows), heads
    int rows;                   // query rows: B * Sq, or the packed total
    const int32_t* qsl;         // packed rows: request b owns rows [qsl[b], qsl[b + 1]); else null
    float scale;
    int num_splits;             // resolved, >= 1
    float* part_o;              // [B*Sq, S, H, 512] fp32 (num_splits > 1)
    float* part_lse;            // [B*Sq, S, H]     fp32 (num_splits > 1)
    void* o_latent;             // [B, Sq, H, 512]
    int o_dtype;                // mla_dtype
    float* lse;                 // [B, Sq, H] or null
    int32_t* dev_status;        // or null
    // Device-built schedule (num_splits == -2): unit u covers tokens [y, z) of query row x and
    // writes partial slot w (-1: the row's final output); row r's partials are slots
    // [rows[r].x, rows[r].x + rows[r].y) when rows[r].y > 1. Null in the uniform-split modes.
    const int4* plan_units;
    const int2* plan_rows;
    const int* plan_count;      // [0] units actually planned, [1] split rows (rows with partials)
    const int* plan_split_rows; // the split rows' indices, plan_count[1] of them
    int plan_max_units;         // the grid is sized for this many units
};

// Request b, position t and query length of query row r: uniform rows are r = b * Sq + t;
// packed rows belong to the last request whose first row is <= r (binary search of qsl).
__device__ __forceinline__ void row_request(const DecodeArgs& p, int r, int* b, int* t, int* q_len) {
    if (p.qsl == nullptr) {
        *b = r / p.Sq;
        *t = r % p.Sq;
        *q_len = p.Sq;
        return;
    }
    int lo = 0, hi = p.B - 1;  // invariant: qsl[lo] <= r
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.qsl[mid] <= r)
            lo = mid;
        else
            hi = mid - 1;
    }
    *b = lo;
    *t = r - p.qsl[lo];
    *q_len = p.qsl[lo + 1] - p.qsl[lo];
}

// Visible tokens of query row r: seq_len - (q_len - 1 - t), clamped at 0, with seq_len clamped
// to what the block table can hold; an out-of-range seq_len sets
// MLA_DEV_SEQ_TOO_LONG when `report`.
__device__ __forceinline__ int visible_tokens(const DecodeArgs& p, int r, bool report) {
    int b, t, q_len;
    row_request(p, r, &b, &t, &q_len);
    int seq = p.seq_lens[b];
    const int cap = p.max_blocks * MLA_PAGE_SIZE;
    if (seq > cap || seq > p.max_seq_len || seq < 0) {
        if (report && p.dev_status) atomicOr(p.dev_status, MLA_DEV_SEQ_TOO_LONG);
        seq = seq < 0 ? 0 : (seq > cap ? cap : seq);
    }
    const int n = seq - (q_len - 1 - t);
    return n < 0 ? 0 : n;
}

// Upper bound of planned units (num_splits == -2) for B * Sq query rows on `pairs` SM pairs.
inline int64_t plan_max_units(int64_t rows, int pairs) { return rows + 2 * (int64_t)pairs; }

// Workspace carve-up of a decode call (the same for both cache formats): the device-built
// schedule, then the split-KV partials; every region starts on a 256-byte boundary.
struct WorkspaceLayout {
    size_t plan, part_o, part_lse, total;
    int64_t partial_slots;  // rows of part_o / part_lse
};
// `rows` query rows (split partials per row); B, kv_dtype and max_seq_len do not change it.
WorkspaceLayout workspace_layout(int kv_dtype, int B, int64_t rows, int H, int num_splits, int max_seq_len);

// Token range [j0, j1) of split s of a row with n visible tokens: the row is cut into
// num_splits page-aligned chunks of round_up(ceil(n / S), 64) tokens; trailing splits may be
// empty. The same rule is used by every decode kernel.
__host__ __device__ inline void split_range(int n, int S, int s, int* j0, int* j1) {
    int per = (n + S - 1) / S;
    int chunk = ((per + kPage - 1) / kPage) * kPage;
    int a = s * chunk;
    int e = a + chunk;
    *j0 = a < n ? a : n;
    *j1 = e < n ? e : n;
}

// Launch with programmatic stream serialization: the kernel may start while the preceding
// kernel of the stream finishes, once that kernel has signalled (griddepcontrol); every kernel
// of this library calls ptx::griddep_wait() before it touches data another of its kernels writes.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Record an error for mla_last_error_detail() and return `st` (printf-style message).
mla_status set_error(mla_status st, const char* fmt, ...);

cudaError_t launch_decode_sm103(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_fp8_sm103(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_plan(const DecodeArgs& a, int pairs, cudaStream_t s);
cudaError_t launch_cache_write(const uint16_t* kv_c, int64_t st_c, const uint16_t* k_pe, int64_t st_pe,
                               const int64_t* slots, int T, uint8_t* cache, int kv_dtype, int64_t num_blocks,
                               float kv_scale, int32_t* dev_status, cudaStream_t s);
cudaError_t launch_absorb_sm103(const uint16_t* q_nope, int64_t snt, int64_t snh, const uint16_t* q_pe,
                                int64_t spt, int64_t sph, const uint16_t* w_uk_t, uint16_t* q_out, int T, int H,
                                cudaStream_t s);
cudaError_t launch_out_proj_sm103(const void* o_latent, int in_dtype, const uint16_t* w_uv, void* o,
                                  int out_dtype, int T, int H, cudaStream_t s);
cudaError_t launch_up_proj_sm103(const uint16_t* x, int64_t x_st, int rows, const uint16_t* w, bool w_is_uk,
                                 uint16_t* out, int H, cudaStream_t s);

// ---- prefill, the compute-friendly route ---------------------------------------------------
// Rows of one segment gathered into a contiguous workspace: the latent part x [rows, 512] and the
// rope part kpe [rows, 64], both bf16 holding the stored values exactly (FP8 codes are not scaled
// here), plus per-row (k_scale, v_scale) for an FP8 cache (1 for rows taken from kv_c / k_pe).
// Segments: the new tokens (kPrefillNew), one context chunk (kPrefillChunk), or every request's
// context followed by its new tokens (kPrefillAll: request b's rows start at cu_ctx[b] + qsl[b]).
enum { kPrefillChunk = 0, kPrefillNew = 1, kPrefillAll = 2 };
struct PrefillGather {
    int mode;
    const int32_t* qsl;         // [B + 1] (kPrefillAll)
    const uint16_t* kv_c;       // new tokens' rows (row strides st_c, st_pe)
    int64_t st_c;
    const uint16_t* k_pe;
    int64_t st_pe;
    const uint8_t* cache;       // context chunk: packed context rows [c0, c0 + rows)
    int kv_dtype;
    int64_t num_blocks;
    const int32_t* block_table;
    int max_blocks;
    const int32_t* cu_ctx;      // [B + 1] prefix sums of the context lengths
    int B;
    int64_t c0;
    int rows;
    uint16_t* x;
    uint16_t* kpe;
    float2* scales;             // FP8 only
    int32_t* dev_status;
};

// One attention segment: every query row of the requests attends to its keys in the segment.
// kPrefillNew: the keys are the request's own new tokens (key i visible to query row t iff
// i <= t). kPrefillChunk: the request's rows of the context chunk [c0, c1), all visible.
// kPrefillAll: the request's context and then its new tokens (key p visible to query row t iff
// p <= ctx + t). The result is written (merge = 0) or merged by LSE into o / lse (merge = 1).
struct PrefillAttn {
    const uint16_t* q;          // [T, H, 192]
    const uint16_t* kn;         // [H, key_rows, 128] up-projected k_nope (head-major)
    const uint16_t* v;          // [H, key_rows, 128] up-projected v (head-major)
    const uint16_t* kpe;        // [key_rows, 64]
    const float2* scales;       // FP8 only: per key row (k_scale, v_scale)
    int key_rows;
    const int32_t* qsl;         // [B + 1]
    const int32_t* cu_ctx;      // [B + 1]
    int B, H, T, max_q_len;
    int mode;
    int64_t c0, c1;
    float scale;
    int merge;
    float* o;                   // [T, H, 128]
    float* lse;                 // [T, H]
    int32_t* dev_status;
};
cudaError_t launch_prefill_cu_ctx(const int32_t* ctx_lens, int B, int32_t* cu_ctx, int32_t* dev_status,
                                  cudaStream_t s);
cudaError_t launch_prefill_gather(const PrefillGather& g, cudaStream_t s);
cudaError_t launch_prefill_attn(const PrefillAttn& a, cudaStream_t s);

}  // namespace mla
