/*
 * mla_latent_kv.h -- C ABI of the GB300 (sm_103a) MLA latent-KV decode library.
 *
 * The library runs the decode hot path of Multi-head Latent Attention after matrix absorption:
 *
 *   mla_absorb_q   q_nope [T,H,128] x W_UK_T [H,128,512] -> q [T,H,576] = [ql_nope || q_pe]
 *   mla_decode     q [B,Sq,H,576] over a paged latent cache [num_blocks,64,576]
 *                  -> o_latent [B,Sq,H,512], lse [B,Sq,H]   (MQA: all heads read one KV row)
 *   mla_out_proj   o_latent [T,H,512] x W_UV [H,512,128] -> o [T,H,128]
 *
 * Sources, cited as [page, section]:
 *   [vLLM-MLA]   "vLLM 源码完全拆解(三十七):MLA 注意力后端——矩阵吸收之后,576 维 latent KV
 *                如何被四种内核读走" (vLLM source teardown 37: the MLA attention backend)
 *   [TRT-TP]     "TensorRT-LLM 源码完全拆解(十二):注意力层的张量并行" (absorption section)
 *   [Triton-MLA] "Triton und MLA: portable Attention und Latent-Space-Attention"
 *
 * Conventions shared by every call:
 *   - All tensor arguments are DEVICE pointers owned by the caller, unless a parameter says
 *     otherwise. The library never allocates, frees or synchronises inside these calls; every
 *     launch is asynchronous on `stream` (NULL = the legacy default stream).
 *   - Arguments are validated on the host before anything is launched. On any error the call
 *     returns a non-zero mla_status, launches nothing, and mla_last_error_detail() (per host
 *     thread) describes the failure. Unsupported shapes fail loudly; there is no fallback path
 *     ([vLLM-MLA, multi-GPU section]: capability mismatches raise instead of degrading).
 *   - Faults that only the device can see (a block-table entry outside [0, num_blocks), a
 *     seq_len larger than max_blocks*64, a bounded wait that ran out) are OR-ed as MLA_DEV_*
 *     bits into the optional int32 `dev_status` in device memory; the caller reads it after
 *     synchronising. The kernels never trap.
 *   - bf16 means IEEE bfloat16 bits; all layouts are row-major, last index fastest.
 */
#ifndef MLA_LATENT_KV_H
#define MLA_LATENT_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* mla_stream_t;

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,         /* null pointer, negative size, inconsistent arguments */
    MLA_ERR_UNSUPPORTED = 2,         /* valid but outside what the kernels implement */
    MLA_ERR_WORKSPACE_TOO_SMALL = 3, /* split-KV workspace smaller than required */
    MLA_ERR_CUDA = 4                 /* a CUDA runtime call failed (see detail string) */
} mla_status;

/* Cache row formats ([vLLM-MLA, cache shape section]):
 *   MLA_KV_BF16            576 bf16 = 1152 bytes: [kv_c (512) || k_pe (64)]
 *   MLA_KV_FP8_E4M3_SCALED 576 OCP-FP8-E4M3 bytes, then k_scale (fp32, byte 576) and v_scale
 *                          (fp32, byte 580) = 584 bytes. K = e4m3 * k_scale over all 576 dims,
 *                          V = e4m3 * v_scale over the first 512 dims. */
typedef enum { MLA_KV_BF16 = 0, MLA_KV_FP8_E4M3_SCALED = 1 } mla_kv_dtype;

/* Element type of o_latent (decode output / out_proj input) and of o. */
typedef enum { MLA_DT_F32 = 0, MLA_DT_BF16 = 1 } mla_dtype;

/* DeepSeek-V3 MLA shape ([vLLM-MLA, model layer section]); the only shape implemented, as in
 * the Cutlass and FlashMLA backends ([vLLM-MLA, Cutlass MLA and FlashMLA sections]). */
#define MLA_KV_LORA_RANK 512
#define MLA_ROPE_DIM 64
#define MLA_HEAD_DIM 576 /* cached row / absorbed query width */
#define MLA_NOPE_DIM 128
#define MLA_V_DIM 128
#define MLA_PAGE_SIZE 64
#define MLA_MAX_HEADS 128

/* Device status bits (OR-ed into *dev_status). */
#define MLA_DEV_BAD_BLOCK_ID 0x1 /* a needed block_table entry was outside [0, num_blocks) */
#define MLA_DEV_SEQ_TOO_LONG 0x2 /* seq_lens[b] > max_blocks * 64 or > max_seq_len */
#define MLA_DEV_WAIT_TIMEOUT 0x4 /* a bounded pipeline wait expired; outputs are invalid */
#define MLA_DEV_BAD_SLOT 0x8     /* mla_cache_write: a slot at or beyond num_blocks * 64 (skipped) */

/* Human-readable name of a status. Never NULL. */
const char* mla_status_string(mla_status s);

/* Detail of the last failing call on this host thread ("" if none). Never NULL. */
const char* mla_last_error_detail(void);

/* Self-test of the bounded-wait path that guards every pipeline wait in the kernels: one thread
 * waits on an mbarrier that nothing arrives on. The wait gives up after the library's limit (2 s
 * of global time), ORs MLA_DEV_WAIT_TIMEOUT into *dev_status and the kernel returns.
 *   dev_status  device int32, caller-owned (zero it first)
 *   out         device int32[2], caller-owned: out[0] = milliseconds the wait took, out[1] = 1 if
 *               the wait reported success (it must not), else 0
 * Asynchronous on `stream`; read both after a synchronise. MLA_ERR_INVALID_ARG if a pointer is
 * NULL, MLA_ERR_CUDA if the launch fails. */
mla_status mla_selftest_wait_timeout(int32_t* dev_status, int32_t* out, mla_stream_t stream);

/* Self-test of the FP8 decode kernel's e4m3 -> bf16 widening ([vLLM-MLA, cache-shape section]:
 * OCP FP8 E4M3 codes; the decode widens them to bf16 before the tensor-core MMAs): writes, for
 * every code c = 0..255, the bf16 bits the kernel produces for it.
 *   out   device uint16[256], caller-owned
 * Every finite code's value is a bf16 value, and the kernel must produce it exactly (subnormal
 * codes included); the two NaN codes 0x7F and 0xFF, which mla_cache_write never stores (it
 * saturates), come out as +480 and -480. Asynchronous on `stream`. MLA_ERR_INVALID_ARG if out is
 * NULL, MLA_ERR_CUDA if the launch fails. */
mla_status mla_selftest_e4m3_widen(uint16_t* out, mla_stream_t stream);

/* Bytes of one cached token row: 1152 (bf16) or 584 (FP8), -1 for an unknown format
 * ([vLLM-MLA, cache shape section]; [vLLM-MLA, numbers section]). Host only. */
int64_t mla_kv_row_bytes(mla_kv_dtype kv_dtype);

/* The Triton backend's split count ([vLLM-MLA, Triton MLA section], _compute_num_kv_splits):
 * min(next_pow2(max(1, max_seq_len / 512)), 2 * sm_count). Host only; -1 if an argument is < 0
 * or sm_count < 1. */
int mla_default_num_splits(int max_seq_len, int sm_count);

/* Effective split count mla_decode will use for a `num_splits` request on the current CUDA
 * device:  > 0  that many splits (forced);
 *            0  mla_default_num_splits(max_seq_len, SM count of the device);
 *           -1  this library's own choice for GB300. With more query rows (B*Sq) than SM
 *               pairs the units run in several waves whose packing depends on the rows'
 *               lengths, so -1 resolves to -2 (returned as -2). Otherwise, from max_seq_len
 *               alone: each of the B*Sq*S units runs on one pair of SMs, and S minimises
 *               waves(S) * (pages per split + a fixed per-unit cost of 8 page-times) plus the
 *               partial states' traffic, for S up to the number of 64-token pages.
 *           -2  no uniform count: a schedule is built on the device from seq_lens (no host
 *               synchronisation, [vLLM-MLA, metadata section]: FlashMLA's decode metadata
 *               carries a scheduler plan). Every query row is cut into page-aligned units of
 *               about c pages, with c chosen from the total and longest row lengths by a model
 *               of how the device's 2-SM clusters run the units; a row that gets one unit writes
 *               its output directly. Returned as -2.
 * Returns -1 on invalid arguments or if the SM count cannot be queried. Host only, no sync. */
int mla_resolve_num_splits(int num_splits, int B, int Sq, int H, int max_seq_len);

/* Bytes of split-KV workspace mla_decode needs for `num_splits` resolved splits: 0 when
 * num_splits == 1, else B*Sq*num_splits*H*(512 + 1)*4 rounded up to 256 (fp32 partial outputs
 * and partial LSEs, [vLLM-MLA, Triton MLA section]: attn_logits (B, N, splits, 512 + 1), fp32
 * because the LSE precision decides the merge). num_splits == -2 (device-built schedule): the
 * schedule (256 B + 16 B per unit + 12 B per query row) and partials for B*Sq + SMs units, each
 * region 256-byte aligned. Host only. */
size_t mla_decode_workspace_bytes(int B, int Sq, int H, int num_splits);

/* Bytes of workspace mla_decode needs for a cache of format kv_dtype. It equals
 * mla_decode_workspace_bytes for both formats: the FP8 cache's e4m3 values are widened to bf16
 * (losslessly) in shared memory inside the attention kernel, and k_scale / v_scale are applied
 * there in fp32, so the FP8 format needs no scratch of its own; max_seq_len does not change the
 * result. 0 for an unknown kv_dtype or a non-positive shape. Host only. */
size_t mla_decode_workspace_bytes_kv(mla_kv_dtype kv_dtype, int B, int Sq, int H, int num_splits,
                                     int max_seq_len);

/*
 * Query absorption ([vLLM-MLA, two-algorithms section]: ql_nope = q_nope W_UK^T, concatenated
 * with q_pe; [TRT-TP, absorption section]: fused_q = [q_nope W_kb^T || q_pe]):
 *     q_out[t, h, l]       = sum_p q_nope[t, h, p] * W_UK_T[h, p, l]   (l < 512, fp32 accumulate,
 *                                                                        rounded once to bf16)
 *     q_out[t, h, 512 + r] = q_pe[t, h, r]                              (r < 64, copied)
 *   q_nope  bf16, element (t, h, p) at q_nope[t*q_nope_stride_t + h*q_nope_stride_h + p]
 *   q_pe    bf16, element (t, h, r) at q_pe[t*q_pe_stride_t + h*q_pe_stride_h + r]; may be NULL,
 *           in which case q_out[..., 512:576] is left untouched
 *   W_UK_T  bf16 [H, 128, 512] contiguous (vLLM's W_UK.permute(1, 2, 0))
 *   q_out   bf16 [T, H, 576] contiguous; must not overlap the inputs
 * Strides are in elements and must be multiples of 8 (16-byte rows for TMA); q_nope_stride_t
 * must be non-zero when T > 1 and q_nope_stride_h >= 128 when H > 1. All pointers 16-byte
 * aligned. 1 <= H <= 128, T >= 0 (T == 0 launches nothing).
 */
mla_status mla_absorb_q(const void* q_nope, int64_t q_nope_stride_t, int64_t q_nope_stride_h,
                        const void* q_pe, int64_t q_pe_stride_t, int64_t q_pe_stride_h,
                        const void* W_UK_T, void* q_out, int T, int H, mla_stream_t stream);

/*
 * Paged MQA decode over the latent cache ([vLLM-MLA, two-algorithms section]:
 * o = SDPA([ql_nope, q_pe], [kv_c, k_pe], kv_c); [vLLM-MLA, FlashMLA section]: the cache is
 * read as a single KV head; [Triton-MLA, Datenfluss]). For every request b, query row t < Sq and
 * head h, with n = max(0, seq_lens[b] - (Sq - 1 - t)) visible tokens ([vLLM-MLA, Triton MLA
 * section]: causal multi-token rows via per-row seq_len):
 *     s_j          = scale * < q[b,t,h,0:576], K_j >                   j < n
 *     lse[b,t,h]   = ln sum_j exp(s_j)                                 (natural log, scale inside)
 *     o_latent[b,t,h,:] = sum_j exp(s_j - lse) * V_j                   (512 values)
 * where row j of request b is cache[block_table[b, j / 64], j % 64, :], K_j is its 576 values
 * and V_j its first 512 values (dequantised per row for the FP8 format). A row with n == 0
 * gets o_latent = 0 and lse = -inf. `scale` is the caller's softmax scale; for DeepSeek-V3 it
 * is 1/sqrt(192), not 1/sqrt(576) ([vLLM-MLA, two-algorithms section]).
 *
 *   q           bf16 [B, Sq, H, 576] contiguous (16-byte aligned)
 *   kv_cache    [num_blocks, 64, row] bytes, row = mla_kv_row_bytes(kv_dtype) (16-byte aligned)
 *   block_table int32 [B, max_blocks] contiguous; only entries j/64 for j < seq_lens[b] are read
 *   seq_lens    int32 [B]: KV tokens of request b INCLUDING its Sq new ones (already written)
 *   max_seq_len host upper bound of seq_lens (used for planning; exceeding it sets
 *               MLA_DEV_SEQ_TOO_LONG and the row's output is undefined)
 *   num_splits  split-KV request, see mla_resolve_num_splits (1 = no split, deterministic
 *               per-row reduction order independent of the batch, [vLLM-MLA, FlashMLA section])
 *   workspace   device scratch of >= mla_decode_workspace_bytes_kv(kv_dtype, B, Sq, H,
 *               resolved splits, max_seq_len) bytes, 256-byte aligned (may be NULL when that is
 *               0); contents on entry are ignored
 *   o_latent    [B, Sq, H, 512] of o_dtype (fp32 recommended; bf16 rounds the result once)
 *   lse         fp32 [B, Sq, H], may be NULL
 *   dev_status  int32 device word or NULL; MLA_DEV_* bits are OR-ed into it, never cleared
 * Limits: 1 <= H <= 128, Sq >= 1, B >= 0 (B == 0 launches nothing), page size 64. FP8
 * precision: k_scale multiplies the fp32 score and v_scale the fp32 softmax weight before its
 * one rounding to bf16 for the PV product.
 */
mla_status mla_decode(const void* q, const void* kv_cache, mla_kv_dtype kv_dtype, int64_t num_blocks,
                      const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                      int max_seq_len, int B, int Sq, int H, float scale, int num_splits,
                      void* workspace, size_t workspace_bytes, void* o_latent, mla_dtype o_dtype,
                      float* lse, int32_t* dev_status, mla_stream_t stream);

/*
 * mla_decode over packed query rows of varying length per request ([vLLM-MLA, metadata section]:
 * VARLEN query-length support, a speculative-decoding verification batch mixing requests with
 * 1, 2, 3 ... query tokens). Request b owns query rows [query_start_loc[b], query_start_loc[b+1])
 * (int32 [B + 1] in device memory, non-decreasing, query_start_loc[0] == 0,
 * query_start_loc[B] == total_q); its row t sees n = max(0, seq_lens[b] - (q_len_b - 1 - t))
 * tokens. q is bf16 [total_q, H, 576], o_latent [total_q, H, 512], lse fp32 [total_q, H]; all
 * other arguments and results as mla_decode, with the workspace from
 * mla_decode_varlen_workspace_bytes. A request may have no query rows.
 */
size_t mla_decode_varlen_workspace_bytes(mla_kv_dtype kv_dtype, int B, int total_q, int H, int num_splits,
                                         int max_seq_len);
mla_status mla_decode_varlen(const void* q, const void* kv_cache, mla_kv_dtype kv_dtype, int64_t num_blocks,
                             const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                             const int32_t* query_start_loc, int max_seq_len, int B, int total_q, int H,
                             float scale, int num_splits, void* workspace, size_t workspace_bytes, void* o_latent,
                             mla_dtype o_dtype, float* lse, int32_t* dev_status, mla_stream_t stream);

/*
 * Output up-projection ([vLLM-MLA, two-algorithms section], _v_up_proj: per-head batched GEMM,
 * written token-major):
 *     o[t, h, v] = sum_l o_latent[t, h, l] * W_UV[h, l, v]      (512 -> 128, fp32 accumulate)
 *   o_latent  [T, H, 512] contiguous, fp32 or bf16 (in_dtype)
 *   W_UV      bf16 [H, 512, 128] contiguous (vLLM's W_UV.transpose(0, 1))
 *   o         [T, H, 128] contiguous, fp32 or bf16 (out_dtype); must not overlap the inputs
 * 1 <= H <= 128, T >= 0. Pointers 16-byte aligned.
 */
mla_status mla_out_proj(const void* o_latent, mla_dtype in_dtype, const void* W_UV, void* o,
                        mla_dtype out_dtype, int T, int H, mla_stream_t stream);

/*
 * KV cache write, the step before decode ([vLLM-MLA, cache write section]: the latent and k_pe
 * land in the cache in one kernel, at the slot the block manager assigned each token). Token t's
 * row [kv_c[t, 0:512] || k_pe[t, 0:64]] goes to slot s = slot_mapping[t] = block * 64 + in-page
 * offset of kv_cache; s < 0 marks a padding token and is skipped.
 *   MLA_KV_BF16             the 576 bf16 values are copied (1152-byte row).
 *   MLA_KV_FP8_E4M3_SCALED  every value is stored as e4m3(x * (1 / scale)), rounded to nearest
 *                           even and saturated at +-448, with scale = kv_scale when kv_scale > 0
 *                           (one static scale, as vLLM's per-layer scale), else amax(|row|) / 448
 *                           over the row's 576 values (1 for an all-zero row); amax / 448, the
 *                           reciprocal and the product are binary32, each correctly rounded. k_scale (byte 576) and v_scale (byte 580) both
 *                           receive the scale ([vLLM-MLA, cache shape and numbers sections]).
 *   kv_c          bf16, element (t, d) at kv_c[t * kv_c_stride_t + d]   (stride % 8 == 0)
 *   k_pe          bf16, element (t, r) at k_pe[t * k_pe_stride_t + r]   (stride % 8 == 0)
 *   slot_mapping  int64 [T] in device memory
 *   kv_cache      [num_blocks, 64, mla_kv_row_bytes(kv_dtype)] bytes, 16-byte aligned
 * A slot at or beyond num_blocks * 64 sets MLA_DEV_BAD_SLOT in *dev_status (if given) and the
 * token is skipped. T >= 0 (T == 0 launches nothing). Pointers 16-byte aligned.
 */
mla_status mla_cache_write(const void* kv_c, int64_t kv_c_stride_t, const void* k_pe, int64_t k_pe_stride_t,
                           const int64_t* slot_mapping, int T, void* kv_cache, mla_kv_dtype kv_dtype,
                           int64_t num_blocks, float kv_scale, int32_t* dev_status, mla_stream_t stream);

/*
 * Prefill, the compute-friendly route ([vLLM-MLA, Prefill section]; [vLLM-MLA, two-algorithms
 * section]). A prefill request b has ctx_b tokens already in the paged cache (positions
 * 0 .. ctx_b - 1) and q_b new tokens (positions ctx_b .. ctx_b + q_b - 1), packed request after
 * request: request b owns rows [query_start_loc[b], query_start_loc[b + 1]) of q, kv_c and k_pe.
 * Keys and values are up-projected per head, not absorbed:
 *     k_j = [ c_j . W_UK_T[h]^T (128) || k_pe_j (64) ],   v_j = c_j . W_UV[h]  (128)
 *     o[t, h, :] = sum_j softmax_j(scale * <q[t, h, :], k_j>) v_j,   lse[t, h] = ln sum_j exp(...)
 * over the request's context and its new tokens 0 .. t (causal); the new tokens' rows come from
 * kv_c / k_pe, not from the cache. When the whole context fits in chunk_rows rows, one pass covers
 * every request's context followed by its new tokens (the online softmax merges them). Otherwise
 * the page's order runs: the new tokens first, then the context in chunks of at most chunk_rows
 * gathered rows (each request's context cut at page boundaries; the plan of
 * mla_prefill_chunk_plan), every chunk's partial result merged into the running one by LSE
 * (merge_attn_states). Both give the same attention. FP8 rows are dequantised with k_scale on the
 * key side (k_nope and k_pe) and v_scale on the value side.
 *   q             bf16 [total_q, H, 192] contiguous: q_nope (128) || q_pe (64), RoPE applied
 *   kv_c, k_pe    bf16 new-token rows, element (t, d) at kv_c[t * kv_c_stride_t + d] (d < 512),
 *                 k_pe[t * k_pe_stride_t + r] (r < 64); strides multiples of 8
 *   kv_cache      [num_blocks, 64, row] (bf16 or FP8 rows); only context rows are read
 *   block_table   int32 [B, max_blocks], device; ctx_lens int32 [B] and query_start_loc int32
 *                 [B + 1], device; ctx_lens_host / query_start_loc_host: the same values in host
 *                 memory (they size the launches and the chunk plan; no device read-back)
 *   W_UK_T        bf16 [H, 128, 512], W_UV bf16 [H, 512, 128] (the layouts of mla_absorb_q and
 *                 mla_out_proj)
 *   chunk_rows    context rows gathered and up-projected at a time, >= 64 (the page's budget is
 *                 min(max(8 * max_len, 4 * max_seqs * 64), 65536) rows)
 *   workspace     >= mla_prefill_workspace_bytes(B, total_q, H, chunk_rows) bytes (up-projected
 *                 K / V for chunk_rows + total_q rows), 256-byte aligned, owned by the caller,
 *                 contents undefined after the call
 *   o             fp32 [total_q, H, 128]; lse fp32 [total_q, H] or NULL
 * 1 <= H <= 128; 0 <= ctx_lens[b] <= max_blocks * 64. Bad block ids set MLA_DEV_BAD_BLOCK_ID,
 * a device ctx_lens value outside that range MLA_DEV_SEQ_TOO_LONG. Pointers 16-byte aligned.
 * Everything is enqueued on `stream`; nothing is allocated or synchronised.
 */
size_t mla_prefill_workspace_bytes(int B, int total_q, int H, int64_t chunk_rows);
/* The context chunk plan: up to max_pieces rows of 4 int64 (chunk, request, first position,
 * tokens), in order; returns the number of pieces (pieces may be NULL to count), or -1 for
 * chunk_rows < 64. A request whose remaining context fits the open chunk goes in whole; else as
 * many whole pages as fit; a chunk with no room for a page is closed. */
int64_t mla_prefill_chunk_plan(const int32_t* ctx_lens_host, int B, int64_t chunk_rows, int64_t* pieces,
                               int64_t max_pieces);
mla_status mla_prefill(const void* q, const void* kv_c, int64_t kv_c_stride_t, const void* k_pe,
                       int64_t k_pe_stride_t, const void* kv_cache, mla_kv_dtype kv_dtype, int64_t num_blocks,
                       const int32_t* block_table, int max_blocks, const int32_t* ctx_lens,
                       const int32_t* query_start_loc, const int32_t* ctx_lens_host,
                       const int32_t* query_start_loc_host, int B, int H, const void* W_UK_T, const void* W_UV,
                       float scale, int64_t chunk_rows, void* workspace, size_t workspace_bytes, float* o,
                       float* lse, int32_t* dev_status, mla_stream_t stream);

/*
 * mla_decode without a workspace argument, for callers that cannot allocate device memory when
 * they decode: serving loops that run under a fixed device-memory budget with every buffer made
 * at start-up, host runtimes that forbid device allocations after initialisation, and call paths
 * that cannot carry a workspace pointer down to the attention call. (The pages have no
 * counterpart of this call; it only changes where the decode scratch lives.)
 *
 * Same arguments, meaning and results as mla_decode, minus workspace / workspace_bytes. The
 * split-KV partials live in one file-scope device array of mla_decode_noalloc_max_workspace_bytes()
 * bytes (64 MiB), held on every device that uses it until the process exits; a call whose
 * mla_decode_workspace_bytes_kv exceeds that (only split-KV partials count, for both cache
 * formats) is refused with MLA_ERR_WORKSPACE_TOO_SMALL. The first call on a
 * device looks up the array's device address (once per device, with that device current); make
 * that first call before any stream capture. The address is reused while the device's context
 * stays the same; after a device reset the next call looks it up again (and is then again a
 * first call). The size check comes before any launch. Nothing
 * here calls cudaMalloc,
 * cudaFree or any allocating library routine. All calls share the array: calls whose kernels
 * overlap on the GPU (e.g. issued on different streams) race on it and must be serialised by
 * the caller. The array keeps the last call's contents; no result depends on them.
 */
size_t mla_decode_noalloc_max_workspace_bytes(void);
mla_status mla_decode_noalloc(const void* q, const void* kv_cache, mla_kv_dtype kv_dtype, int64_t num_blocks,
                              const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                              int max_seq_len, int B, int Sq, int H, float scale, int num_splits,
                              void* o_latent, mla_dtype o_dtype, float* lse, int32_t* dev_status,
                              mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_LATENT_KV_H */
