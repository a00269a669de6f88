// mla_api.cu -- the extern "C" boundary: host-side validation, split planning and launches.
//
// Nothing here allocates, frees or synchronises: every call validates its arguments, resolves
// the split plan from host-known quantities only (the pages' "no sync" rule for metadata,
// [vLLM-MLA, metadata section]: host upper bounds instead of device lengths) and enqueues
// kernels on the caller's stream.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "internal.h"

namespace {

thread_local char g_detail[512] = "";

mla_status fail(mla_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof g_detail, fmt, ap);
    va_end(ap);
    return st;
}

mla_status ok() {
    g_detail[0] = '\0';
    return MLA_OK;
}

mla_status cuda_fail(cudaError_t e, const char* what) {
    return fail(MLA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return sms;
}

}  // namespace

namespace mla {
WorkspaceLayout workspace_layout(int kv_dtype, int B, int64_t rows, int H, int num_splits, int max_seq_len) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    WorkspaceLayout w{};
    if (B <= 0 || rows <= 0 || H <= 0) return w;
    size_t off = 0;
    int64_t slots = num_splits > 1 ? rows * num_splits : 0;
    if (num_splits == -2) {  // device-built schedule: header, unit list, per-row slots
        const int sms = device_sm_count();
        if (sms < 1) return w;
        slots = plan_max_units(rows, sms / 2 > 0 ? sms / 2 : 1);
        w.plan = 0;
        off = up(256 + (size_t)slots * sizeof(int4)) + up((size_t)rows * sizeof(int2)) + up((size_t)rows * sizeof(int));
    }
    if (slots > 0) {
        const size_t units = (size_t)slots * H;
        w.part_o = off;
        w.part_lse = off + up(units * kL * sizeof(float));
        off = w.part_lse + up(units * sizeof(float));
        w.partial_slots = slots;
    }
    w.total = off;
    return w;
}

mla_status set_error(mla_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof g_detail, fmt, ap);
    va_end(ap);
    return st;
}
}  // namespace mla

extern "C" {

const char* mla_status_string(mla_status s) {
    switch (s) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
        case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
        case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
        case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    }
    return "MLA_ERR_UNKNOWN";
}

const char* mla_last_error_detail(void) { return g_detail; }

int64_t mla_kv_row_bytes(mla_kv_dtype kv_dtype) {
    switch (kv_dtype) {
        case MLA_KV_BF16: return mla::kBf16RowBytes;
        case MLA_KV_FP8_E4M3_SCALED: return mla::kFp8RowBytes;
    }
    return -1;
}

int mla_default_num_splits(int max_seq_len, int sm_count) {
    if (max_seq_len < 0 || sm_count < 1) return -1;
    int ideal = std::max(1, max_seq_len / 512);
    int p2 = 1;
    while (p2 < ideal) p2 *= 2;
    return std::min(p2, 2 * sm_count);
}

int mla_resolve_num_splits(int num_splits, int B, int Sq, int H, int max_seq_len) {
    if (num_splits > 0) return num_splits;
    if (num_splits < -2 || B < 0 || Sq < 1 || H < 1 || max_seq_len < 0) return -1;
    if (num_splits == -2) return device_sm_count() >= 1 ? -2 : -1;  // decided per row on the device
    int sms = device_sm_count();
    if (sms < 1) return -1;
    if (num_splits == 0) return mla_default_num_splits(max_seq_len, sms);
    // More query rows than SM pairs: the units run in several waves, and how they pack depends on
    // the rows' lengths, which only the device has. -1 then builds the schedule there (as -2).
    if ((int64_t)B * Sq > std::max(1, sms / 2)) return -2;
    // GB300 plan: each unit (one query row x one split) occupies one pair of SMs. Estimate the
    // time of S splits as  waves(S) * (pages_per_split(S) + o) * t_page  plus the partial-state
    // traffic of the split path, and take the cheapest S. o is a unit's fixed cost (pipeline
    // fill, Q load, epilogue, wave tail) in page-times. Measurements of the bf16 kernel put it
    // near 18 (one split of 64 pages: 115 us; of 228 pages: 344 us, i.e. 1.4 us per page and
    // 25 us per unit); a smaller value is used because the host sees only max_seq_len, and a
    // ragged batch's longest row is better split than the uniform model says.
    constexpr double kUnitOverheadPages = 8.0;
    const int slots = std::max(1, sms / 2);
    const int64_t rows = (int64_t)B * Sq;
    const int pages = std::max(1, (max_seq_len + mla::kPage - 1) / mla::kPage);
    if (rows == 0) return 1;
    const double page_bytes = (double)mla::kPage * mla::kBf16RowBytes;
    const double partial_bytes_per_unit = (double)H * (mla::kL + 1) * 4.0 * 2.0;  // write + read
    double best = 1e300;
    int best_s = 1;
    for (int S = 1; S <= pages; ++S) {
        int64_t units = rows * S;
        int64_t waves = (units + slots - 1) / slots;
        int per = (pages + S - 1) / S;
        double t = (double)waves * (per + kUnitOverheadPages) * page_bytes * slots;  // at the wave rate
        if (S > 1) t += (double)units * partial_bytes_per_unit;
        if (t < best * 0.999) {
            best = t;
            best_s = S;
        }
    }
    return best_s;
}

size_t mla_decode_workspace_bytes(int B, int Sq, int H, int num_splits) {
    if (Sq <= 0) return 0;
    return mla::workspace_layout(MLA_KV_BF16, B, (int64_t)B * Sq, H, num_splits, 0).total;
}

size_t mla_decode_workspace_bytes_kv(mla_kv_dtype kv_dtype, int B, int Sq, int H, int num_splits, int max_seq_len) {
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3_SCALED) return 0;
    if (Sq <= 0) return 0;
    return mla::workspace_layout(kv_dtype, B, (int64_t)B * Sq, H, num_splits, max_seq_len).total;
}

size_t mla_decode_varlen_workspace_bytes(mla_kv_dtype kv_dtype, int B, int total_q, int H, int num_splits,
                                         int max_seq_len) {
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3_SCALED) return 0;
    return mla::workspace_layout(kv_dtype, B, total_q, H, num_splits, max_seq_len).total;
}

mla_status mla_absorb_q(const void* q_nope, int64_t snt, int64_t snh, const void* q_pe, int64_t spt,
                        int64_t sph, const void* W_UK_T, void* q_out, int T, int H, mla_stream_t stream) {
    if (T < 0) return fail(MLA_ERR_INVALID_ARG, "mla_absorb_q: T=%d < 0", T);
    if (H < 1 || H > MLA_MAX_HEADS)
        return fail(MLA_ERR_UNSUPPORTED, "mla_absorb_q: H=%d outside [1, %d]", H, MLA_MAX_HEADS);
    if (T == 0) return ok();
    if (!q_nope || !W_UK_T || !q_out) return fail(MLA_ERR_INVALID_ARG, "mla_absorb_q: null pointer");
    if (!aligned16(q_nope) || !aligned16(W_UK_T) || !aligned16(q_out) || (q_pe && !aligned16(q_pe)))
        return fail(MLA_ERR_UNSUPPORTED, "mla_absorb_q: pointers must be 16-byte aligned");
    if (snt < 0 || snh < 0 || snt % 8 || snh % 8 || (q_pe && (spt < 0 || sph < 0 || spt % 8 || sph % 8)))
        return fail(MLA_ERR_UNSUPPORTED, "mla_absorb_q: strides must be non-negative multiples of 8");
    if (snh < mla::kP && H > 1)
        return fail(MLA_ERR_INVALID_ARG, "mla_absorb_q: q_nope head stride %lld < 128", (long long)snh);
    if (snt == 0 && T > 1)
        return fail(MLA_ERR_UNSUPPORTED, "mla_absorb_q: q_nope token stride 0 (broadcast) is not supported");
    cudaError_t e = mla::launch_absorb_sm103((const uint16_t*)q_nope, snt, snh, (const uint16_t*)q_pe, spt,
                                           sph, (const uint16_t*)W_UK_T, (uint16_t*)q_out, T, H,
                                           (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "mla_absorb_q launch");
    return ok();
}

}  // extern "C"

namespace {

// Shared body of mla_decode (uniform Sq rows per request, qsl == nullptr) and mla_decode_varlen
// (packed rows, qsl = query_start_loc, Sq == 1): `rows` query rows of q / o_latent / lse.
mla_status decode_impl(const void* q, const void* kv_cache, mla_kv_dtype kv_dtype, int64_t num_blocks,
                       const int32_t* block_table, int max_blocks, const int32_t* seq_lens, const int32_t* qsl,
                       int max_seq_len, int B, int Sq, int64_t rows, int H, float scale, int num_splits,
                       void* workspace, size_t workspace_bytes, void* o_latent, mla_dtype o_dtype, float* lse,
                       int32_t* dev_status, mla_stream_t stream) {
    if (H < 1 || H > MLA_MAX_HEADS)
        return fail(MLA_ERR_UNSUPPORTED, "mla_decode: H=%d outside [1, %d]", H, MLA_MAX_HEADS);
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3_SCALED)
        return fail(MLA_ERR_INVALID_ARG, "mla_decode: unknown kv_dtype %d", (int)kv_dtype);
    if (o_dtype != MLA_DT_F32 && o_dtype != MLA_DT_BF16)
        return fail(MLA_ERR_INVALID_ARG, "mla_decode: unknown o_dtype %d", (int)o_dtype);
    if (max_seq_len < 0 || max_blocks < 0 || num_blocks < 0)
        return fail(MLA_ERR_INVALID_ARG, "mla_decode: negative max_seq_len/max_blocks/num_blocks");
    if ((int64_t)max_seq_len > (int64_t)max_blocks * mla::kPage)
        return fail(MLA_ERR_INVALID_ARG, "mla_decode: max_seq_len=%d exceeds max_blocks*64=%lld", max_seq_len,
                    (long long)max_blocks * mla::kPage);
    if (!(std::isfinite(scale)) || scale <= 0.f)
        return fail(MLA_ERR_INVALID_ARG, "mla_decode: scale must be finite and > 0");
    if (num_splits < -2) return fail(MLA_ERR_INVALID_ARG, "mla_decode: num_splits=%d < -2", num_splits);
    if (B == 0 || rows == 0) return ok();
    if (!q || !o_latent || !seq_lens || (max_seq_len > 0 && (!kv_cache || !block_table)))
        return fail(MLA_ERR_INVALID_ARG, "mla_decode: null pointer");
    if (rows > INT32_MAX) return fail(MLA_ERR_UNSUPPORTED, "mla_decode: %lld query rows too many", (long long)rows);
    if (!aligned16(q) || (kv_cache && !aligned16(kv_cache)) || !aligned16(o_latent))
        return fail(MLA_ERR_UNSUPPORTED, "mla_decode: q, kv_cache and o_latent must be 16-byte aligned");
    if (num_blocks > (int64_t)(INT32_MAX / mla::kPage))
        return fail(MLA_ERR_UNSUPPORTED, "mla_decode: num_blocks=%lld too large (max %d)", (long long)num_blocks,
                    INT32_MAX / mla::kPage);
    int S = mla_resolve_num_splits(num_splits, (int)rows, 1, H, max_seq_len);
    const bool planned = S == -2;
    if (S < 1 && !planned) return fail(MLA_ERR_CUDA, "mla_decode: could not resolve num_splits (no CUDA device?)");
    if (rows * H > (int64_t)INT32_MAX)
        return fail(MLA_ERR_UNSUPPORTED, "mla_decode: rows*H=%lld too large", (long long)(rows * H));
    const int pairs = planned ? std::max(1, device_sm_count() / 2) : 1;
    const int64_t max_units = planned ? mla::plan_max_units(rows, pairs) : rows * S;
    if (max_units > (int64_t)1 << 30)
        return fail(MLA_ERR_UNSUPPORTED, "mla_decode: %lld work units too many", (long long)max_units);
    const mla::WorkspaceLayout wl = mla::workspace_layout(kv_dtype, B, rows, H, S, max_seq_len);
    const size_t need = wl.total;
    if (need > 0 && (workspace == nullptr || workspace_bytes < need))
        return fail(MLA_ERR_WORKSPACE_TOO_SMALL,
                    "mla_decode: workspace %zu bytes < %zu needed (%d splits)",
                    workspace ? workspace_bytes : (size_t)0, need, S);
    if (need > 0 && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(MLA_ERR_UNSUPPORTED, "mla_decode: workspace must be 256-byte aligned");

    mla::DecodeArgs a{};
    a.q = (const uint16_t*)q;
    a.cache = (const uint8_t*)kv_cache;
    a.kv_dtype = kv_dtype;
    a.num_blocks = num_blocks;
    a.block_table = block_table;
    a.max_blocks = max_blocks;
    a.seq_lens = seq_lens;
    a.max_seq_len = max_seq_len;
    a.B = B;
    a.Sq = Sq;
    a.rows = (int)rows;
    a.qsl = qsl;
    a.H = H;
    a.scale = scale;
    a.num_splits = planned ? 1 : S;
    if (wl.partial_slots > 0) {
        a.part_o = (float*)((char*)workspace + wl.part_o);
        a.part_lse = (float*)((char*)workspace + wl.part_lse);
    }
    if (planned) {
        char* base = (char*)workspace + wl.plan;
        a.plan_count = (const int*)base;
        a.plan_units = (const int4*)(base + 256);
        const size_t rows_off = (256 + (size_t)max_units * sizeof(int4) + 255) / 256 * 256;
        a.plan_rows = (const int2*)(base + rows_off);
        a.plan_split_rows = (const int*)(base + rows_off + ((size_t)rows * sizeof(int2) + 255) / 256 * 256);
        a.plan_max_units = (int)max_units;
    }
    const bool fp8 = kv_dtype == MLA_KV_FP8_E4M3_SCALED;
    a.o_latent = o_latent;
    a.o_dtype = o_dtype;
    a.lse = lse;
    a.dev_status = dev_status;
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e = cudaSuccess;
    if (planned) {
        e = mla::launch_plan(a, pairs, st);
        if (e != cudaSuccess) return cuda_fail(e, "mla_decode schedule launch");
    }
    e = fp8 ? mla::launch_decode_fp8_sm103(a, st) : mla::launch_decode_sm103(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "mla_decode launch");
    if (planned || S > 1) {
        e = mla::launch_merge(a, st);
        if (e != cudaSuccess) return cuda_fail(e, "mla_decode merge launch");
    }
    return ok();
}

}  // namespace

extern "C" {

mla_status mla_decode(const void* q, const void* kv_cache, mla_kv_dtype kv_dtype, int64_t num_blocks,
                      const int32_t* block_table, int max_blocks, const int32_t* seq_lens, int max_seq_len,
                      int B, int Sq, int H, float scale, int num_splits, void* workspace,
                      size_t workspace_bytes, void* o_latent, mla_dtype o_dtype, float* lse,
                      int32_t* dev_status, mla_stream_t stream) {
    if (B < 0) return fail(MLA_ERR_INVALID_ARG, "mla_decode: B=%d < 0", B);
    if (Sq < 1) return fail(MLA_ERR_INVALID_ARG, "mla_decode: Sq=%d < 1", Sq);
    return decode_impl(q, kv_cache, kv_dtype, num_blocks, block_table, max_blocks, seq_lens, nullptr, max_seq_len,
                       B, Sq, (int64_t)B * Sq, H, scale, num_splits, workspace, workspace_bytes, o_latent, o_dtype,
                       lse, dev_status, stream);
}

mla_status mla_decode_varlen(const void* q, const void* kv_cache, mla_kv_dtype kv_dtype, int64_t num_blocks,
                             const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                             const int32_t* query_start_loc, int max_seq_len, int B, int total_q, int H,
                             float scale, int num_splits, void* workspace, size_t workspace_bytes, void* o_latent,
                             mla_dtype o_dtype, float* lse, int32_t* dev_status, mla_stream_t stream) {
    if (B < 0 || total_q < 0) return fail(MLA_ERR_INVALID_ARG, "mla_decode_varlen: B=%d, total_q=%d", B, total_q);
    if (total_q > 0 && !query_start_loc) return fail(MLA_ERR_INVALID_ARG, "mla_decode_varlen: null query_start_loc");
    return decode_impl(q, kv_cache, kv_dtype, num_blocks, block_table, max_blocks, seq_lens, query_start_loc,
                       max_seq_len, B, 1, total_q, H, scale, num_splits, workspace, workspace_bytes, o_latent,
                       o_dtype, lse, dev_status, stream);
}

mla_status mla_cache_write(const void* kv_c, int64_t kv_c_stride_t, const void* k_pe, int64_t k_pe_stride_t,
                           const int64_t* slot_mapping, int T, void* kv_cache, mla_kv_dtype kv_dtype,
                           int64_t num_blocks, float kv_scale, int32_t* dev_status, mla_stream_t stream) {
    if (T < 0) return fail(MLA_ERR_INVALID_ARG, "mla_cache_write: T=%d < 0", T);
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3_SCALED)
        return fail(MLA_ERR_INVALID_ARG, "mla_cache_write: unknown kv_dtype %d", (int)kv_dtype);
    if (num_blocks < 0) return fail(MLA_ERR_INVALID_ARG, "mla_cache_write: num_blocks < 0");
    if (!(kv_scale >= 0.f) || std::isinf(kv_scale))
        return fail(MLA_ERR_INVALID_ARG, "mla_cache_write: kv_scale must be finite and >= 0 (0 = per-token)");
    if (T == 0) return ok();
    if (!kv_c || !k_pe || !slot_mapping || !kv_cache) return fail(MLA_ERR_INVALID_ARG, "mla_cache_write: null pointer");
    if (!aligned16(kv_c) || !aligned16(k_pe) || !aligned16(kv_cache))
        return fail(MLA_ERR_UNSUPPORTED, "mla_cache_write: kv_c, k_pe and kv_cache must be 16-byte aligned");
    if (kv_c_stride_t < mla::kL || k_pe_stride_t < mla::kR || kv_c_stride_t % 8 || k_pe_stride_t % 8)
        return fail(MLA_ERR_UNSUPPORTED, "mla_cache_write: row strides must be multiples of 8 covering the row");
    if (num_blocks > (int64_t)1 << 40) return fail(MLA_ERR_UNSUPPORTED, "mla_cache_write: num_blocks too large");
    cudaError_t e = mla::launch_cache_write((const uint16_t*)kv_c, kv_c_stride_t, (const uint16_t*)k_pe,
                                            k_pe_stride_t, slot_mapping, T, (uint8_t*)kv_cache, kv_dtype,
                                            num_blocks, kv_scale, dev_status, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "mla_cache_write launch");
    return ok();
}

mla_status mla_out_proj(const void* o_latent, mla_dtype in_dtype, const void* W_UV, void* o, mla_dtype out_dtype,
                        int T, int H, mla_stream_t stream) {
    if (T < 0) return fail(MLA_ERR_INVALID_ARG, "mla_out_proj: T=%d < 0", T);
    if (H < 1 || H > MLA_MAX_HEADS)
        return fail(MLA_ERR_UNSUPPORTED, "mla_out_proj: H=%d outside [1, %d]", H, MLA_MAX_HEADS);
    if ((in_dtype != MLA_DT_F32 && in_dtype != MLA_DT_BF16) || (out_dtype != MLA_DT_F32 && out_dtype != MLA_DT_BF16))
        return fail(MLA_ERR_INVALID_ARG, "mla_out_proj: unknown dtype");
    if (T == 0) return ok();
    if (!o_latent || !W_UV || !o) return fail(MLA_ERR_INVALID_ARG, "mla_out_proj: null pointer");
    if (!aligned16(o_latent) || !aligned16(W_UV) || !aligned16(o))
        return fail(MLA_ERR_UNSUPPORTED, "mla_out_proj: pointers must be 16-byte aligned");
    cudaError_t e = mla::launch_out_proj_sm103(o_latent, in_dtype, (const uint16_t*)W_UV, o, out_dtype, T, H,
                                              (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "mla_out_proj launch");
    return ok();
}

}  // extern "C"

// ---------------------------------------------------------------------------------------------
// Prefill (compute-friendly route)
// ---------------------------------------------------------------------------------------------
namespace {

struct PrefillLayout {
    size_t cu_ctx, x, kpe, scales, kn, v, lse, total;
    int64_t rows;  // rows of one segment's workspace
};

PrefillLayout prefill_layout(int B, int total_q, int H, int64_t chunk_rows) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    PrefillLayout w{};
    w.rows = chunk_rows + total_q;  // one pass over context + new rows when the context fits
    size_t off = 0;
    w.cu_ctx = off;
    off += up((size_t)(B + 1) * sizeof(int32_t));
    w.x = off;
    off += up((size_t)w.rows * mla::kL * 2);
    w.kpe = off;
    off += up((size_t)w.rows * mla::kR * 2);
    w.scales = off;
    off += up((size_t)w.rows * 2 * sizeof(float));
    w.kn = off;
    off += up((size_t)w.rows * H * 128 * 2);
    w.v = off;
    off += up((size_t)w.rows * H * 128 * 2);
    w.lse = off;
    off += up((size_t)total_q * H * sizeof(float));
    w.total = off;
    return w;
}

// The chunk rule, walked over the host copy of the context lengths; calls emit(chunk, b, pos, n).
template <class F>
void plan_chunks(const int32_t* ctx, int B, int64_t budget, F&& emit) {
    int64_t chunk = 0, used = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t len = ctx[b] > 0 ? ctx[b] : 0;
        int64_t pos = 0;
        while (pos < len) {
            int64_t n = len - pos;
            const int64_t room = budget - used;
            if (n > room) {
                n = room / mla::kPage * mla::kPage;  // whole pages only, so the next piece starts on one
                if (n == 0) {
                    ++chunk;
                    used = 0;
                    continue;
                }
            }
            emit(chunk, b, pos, n);
            used += n;
            pos += n;
        }
    }
}

}  // namespace

extern "C" {

size_t mla_prefill_workspace_bytes(int B, int total_q, int H, int64_t chunk_rows) {
    if (B < 1 || total_q < 0 || H < 1 || H > MLA_MAX_HEADS || chunk_rows < mla::kPage) return 0;
    return prefill_layout(B, total_q, H, chunk_rows).total;
}

int64_t mla_prefill_chunk_plan(const int32_t* ctx_lens_host, int B, int64_t chunk_rows, int64_t* pieces,
                               int64_t max_pieces) {
    if (chunk_rows < mla::kPage || B < 0 || (B > 0 && !ctx_lens_host)) return -1;
    int64_t n = 0;
    plan_chunks(ctx_lens_host, B, chunk_rows, [&](int64_t c, int b, int64_t pos, int64_t len) {
        if (pieces && n < max_pieces) {
            pieces[4 * n] = c;
            pieces[4 * n + 1] = b;
            pieces[4 * n + 2] = pos;
            pieces[4 * n + 3] = len;
        }
        ++n;
    });
    return n;
}

mla_status mla_prefill(const void* q, const void* kv_c, int64_t kv_c_stride_t, const void* k_pe,
                       int64_t k_pe_stride_t, const void* kv_cache, mla_kv_dtype kv_dtype, int64_t num_blocks,
                       const int32_t* block_table, int max_blocks, const int32_t* ctx_lens,
                       const int32_t* query_start_loc, const int32_t* ctx_lens_host,
                       const int32_t* query_start_loc_host, int B, int H, const void* W_UK_T, const void* W_UV,
                       float scale, int64_t chunk_rows, void* workspace, size_t workspace_bytes, float* o,
                       float* lse, int32_t* dev_status, mla_stream_t stream) {
    if (B < 1) return fail(MLA_ERR_INVALID_ARG, "mla_prefill: B=%d < 1", B);
    if (H < 1 || H > MLA_MAX_HEADS)
        return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: H=%d outside [1, %d]", H, MLA_MAX_HEADS);
    if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3_SCALED)
        return fail(MLA_ERR_INVALID_ARG, "mla_prefill: unknown kv_dtype %d", (int)kv_dtype);
    if (chunk_rows < mla::kPage)
        return fail(MLA_ERR_INVALID_ARG, "mla_prefill: chunk_rows=%lld < 64", (long long)chunk_rows);
    if (chunk_rows > ((int64_t)1 << 24))
        return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: chunk_rows=%lld above 2^24", (long long)chunk_rows);
    if (!(scale > 0.f) || std::isinf(scale))
        return fail(MLA_ERR_INVALID_ARG, "mla_prefill: scale must be finite and > 0");
    if (!ctx_lens_host || !query_start_loc_host) return fail(MLA_ERR_INVALID_ARG, "mla_prefill: null host metadata");
    if (query_start_loc_host[0] != 0) return fail(MLA_ERR_INVALID_ARG, "mla_prefill: query_start_loc[0] != 0");
    if (num_blocks < 0 || max_blocks < 0)
        return fail(MLA_ERR_INVALID_ARG, "mla_prefill: negative num_blocks/max_blocks");
    int max_q = 0;
    int64_t total_ctx = 0;
    for (int b = 0; b < B; ++b) {
        const int ql = query_start_loc_host[b + 1] - query_start_loc_host[b];
        if (ql < 0) return fail(MLA_ERR_INVALID_ARG, "mla_prefill: query_start_loc decreases at %d", b);
        max_q = std::max(max_q, ql);
        if (ctx_lens_host[b] < 0 || (int64_t)ctx_lens_host[b] > (int64_t)max_blocks * mla::kPage)
            return fail(MLA_ERR_INVALID_ARG, "mla_prefill: ctx_lens[%d]=%d outside [0, max_blocks*64]", b,
                        ctx_lens_host[b]);
        total_ctx += ctx_lens_host[b];
    }
    const int total_q = query_start_loc_host[B];
    if (total_ctx > INT32_MAX)
        return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: %lld context rows too many", (long long)total_ctx);
    if (total_q == 0) return ok();
    if (!q || !kv_c || !k_pe || !ctx_lens || !query_start_loc || !W_UK_T || !W_UV || !o || !workspace ||
        (total_ctx > 0 && (!kv_cache || !block_table)))
        return fail(MLA_ERR_INVALID_ARG, "mla_prefill: null pointer");
    if (!aligned16(q) || !aligned16(kv_c) || !aligned16(k_pe) || !aligned16(W_UK_T) || !aligned16(W_UV) ||
        !aligned16(o) || (kv_cache && !aligned16(kv_cache)))
        return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: pointers must be 16-byte aligned");
    if (kv_c_stride_t < mla::kL || k_pe_stride_t < mla::kR || kv_c_stride_t % 8 || k_pe_stride_t % 8)
        return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: row strides must be multiples of 8 covering the row");
    const PrefillLayout L = prefill_layout(B, total_q, H, chunk_rows);
    if (workspace_bytes < L.total)
        return fail(MLA_ERR_WORKSPACE_TOO_SMALL, "mla_prefill: workspace %zu < %zu bytes", workspace_bytes, L.total);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u)
        return fail(MLA_ERR_UNSUPPORTED, "mla_prefill: workspace must be 256-byte aligned");

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* cu_ctx = reinterpret_cast<int32_t*>(ws + L.cu_ctx);
    uint16_t* x = reinterpret_cast<uint16_t*>(ws + L.x);
    uint16_t* kpe = reinterpret_cast<uint16_t*>(ws + L.kpe);
    float2* scales = reinterpret_cast<float2*>(ws + L.scales);
    uint16_t* kn = reinterpret_cast<uint16_t*>(ws + L.kn);
    uint16_t* vv = reinterpret_cast<uint16_t*>(ws + L.v);
    float* lse_out = lse ? lse : reinterpret_cast<float*>(ws + L.lse);
    const cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = mla::launch_prefill_cu_ctx(ctx_lens, B, cu_ctx, dev_status, s);
    if (e != cudaSuccess) return cuda_fail(e, "mla_prefill prefix-sum launch");

    mla::PrefillAttn a{};
    a.q = static_cast<const uint16_t*>(q);
    a.kn = kn;
    a.v = vv;
    a.kpe = kpe;
    a.qsl = query_start_loc;
    a.cu_ctx = cu_ctx;
    a.B = B;
    a.H = H;
    a.T = total_q;
    a.max_q_len = max_q;
    a.scale = scale;
    a.o = o;
    a.lse = lse_out;
    a.dev_status = dev_status;
    // one segment: gather, the two up-projections, attention
    auto segment = [&](const mla::PrefillGather& g, bool fp8) -> mla_status {
        cudaError_t err = mla::launch_prefill_gather(g, s);
        if (err != cudaSuccess) return cuda_fail(err, "mla_prefill gather launch");
        err = mla::launch_up_proj_sm103(x, mla::kL, g.rows, static_cast<const uint16_t*>(W_UK_T), true, kn, H, s);
        if (err != cudaSuccess) return cuda_fail(err, "mla_prefill k up-projection launch");
        err = mla::launch_up_proj_sm103(x, mla::kL, g.rows, static_cast<const uint16_t*>(W_UV), false, vv, H, s);
        if (err != cudaSuccess) return cuda_fail(err, "mla_prefill v up-projection launch");
        a.key_rows = g.rows;
        a.scales = fp8 ? scales : nullptr;
        err = mla::launch_prefill_attn(a, s);
        if (err != cudaSuccess) return cuda_fail(err, "mla_prefill attention launch");
        return MLA_OK;
    };
    // The whole context fits the row budget: one pass over every request's context followed by
    // its new tokens, the same attention as the page's new-token segment, context chunks and
    // merge, with the merge done by the online softmax itself.
    if (total_ctx <= chunk_rows) {
        mla::PrefillGather g{};
        g.mode = mla::kPrefillAll;
        g.qsl = query_start_loc;
        g.kv_c = static_cast<const uint16_t*>(kv_c);
        g.st_c = kv_c_stride_t;
        g.k_pe = static_cast<const uint16_t*>(k_pe);
        g.st_pe = k_pe_stride_t;
        g.cache = static_cast<const uint8_t*>(kv_cache);
        g.kv_dtype = kv_dtype;
        g.num_blocks = num_blocks;
        g.block_table = block_table;
        g.max_blocks = max_blocks;
        g.cu_ctx = cu_ctx;
        g.B = B;
        g.rows = (int)(total_ctx + total_q);
        g.x = x;
        g.kpe = kpe;
        g.scales = scales;
        g.dev_status = dev_status;
        a.mode = mla::kPrefillAll;
        a.merge = 0;
        const mla_status st = segment(g, kv_dtype == MLA_KV_FP8_E4M3_SCALED);
        if (st != MLA_OK) return st;
        return ok();
    }
    // 1. the new tokens, causal among themselves
    {
        mla::PrefillGather g{};
        g.mode = mla::kPrefillNew;
        g.kv_c = static_cast<const uint16_t*>(kv_c);
        g.st_c = kv_c_stride_t;
        g.k_pe = static_cast<const uint16_t*>(k_pe);
        g.st_pe = k_pe_stride_t;
        g.rows = total_q;
        g.x = x;
        g.kpe = kpe;
        a.mode = mla::kPrefillNew;
        a.merge = 0;
        const mla_status st = segment(g, false);
        if (st != MLA_OK) return st;
    }
    // 2. the context, chunk by chunk, merged into the running result
    std::vector<int64_t> cu_host((size_t)B + 1, 0);
    for (int b = 0; b < B; ++b) cu_host[b + 1] = cu_host[b] + ctx_lens_host[b];
    int64_t cur = -1, c0 = 0, c1 = 0;
    mla_status st = MLA_OK;
    auto flush = [&]() {
        if (cur < 0 || st != MLA_OK) return;
        mla::PrefillGather g{};
        g.mode = mla::kPrefillChunk;
        g.cache = static_cast<const uint8_t*>(kv_cache);
        g.kv_dtype = kv_dtype;
        g.num_blocks = num_blocks;
        g.block_table = block_table;
        g.max_blocks = max_blocks;
        g.cu_ctx = cu_ctx;
        g.B = B;
        g.c0 = c0;
        g.rows = (int)(c1 - c0);
        g.x = x;
        g.kpe = kpe;
        g.scales = scales;
        g.dev_status = dev_status;
        a.mode = mla::kPrefillChunk;
        a.merge = 1;
        a.c0 = c0;
        a.c1 = c1;
        st = segment(g, kv_dtype == MLA_KV_FP8_E4M3_SCALED);
    };
    plan_chunks(ctx_lens_host, B, chunk_rows, [&](int64_t c, int b, int64_t pos, int64_t n) {
        if (c != cur) {
            flush();
            cur = c;
            c0 = cu_host[b] + pos;
        }
        c1 = cu_host[b] + pos + n;
    });
    flush();
    if (st != MLA_OK) return st;
    return ok();
}

}  // extern "C"
