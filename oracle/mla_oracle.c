/*
 * mla_oracle.c -- plain, slow, fp64 CPU oracle for MLA decode over a paged latent KV cache.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU-baseline /
 * reference leg load this file. It shares no code, header, table or constant with the CUDA
 * library; the two meet only in the seeded input arrays that both are handed.
 *
 * Every function below widens the stored bf16 / e4m3 bytes exactly to double and then follows
 * the pages' definitions step by step, with no blocking, fusion or reordering beyond what the
 * definition itself states. Sources, cited as  [page, section]:
 *
 *   [vLLM-MLA]  "vLLM 源码完全拆解(三十七):MLA 注意力后端——矩阵吸收之后,576 维 latent KV
 *               如何被四种内核读走" (vLLM source teardown 37: the MLA attention backend)
 *   [TRT-TP]    "TensorRT-LLM 源码完全拆解(十二):注意力层的张量并行——head 怎么切、MLA 为什么
 *               不能照切" (TensorRT-LLM teardown 12: attention tensor parallelism)
 *   [Triton-MLA] "Triton und MLA: portable Attention und Latent-Space-Attention"
 *
 * Readings the pages leave open (each also listed in the design notes):
 *   - lse is the natural log of sum_j exp(scale * q.k_j), i.e. the scale is inside
 *     ([Triton-MLA, Entwurfsmotivation]: "lse_base_on_e" true).
 *   - a row with no visible tokens has o = 0 and lse = -inf ([vLLM-MLA, Prefill section]:
 *     empty partials are written as output 0, lse -inf).
 *   - seq_lens counts the KV tokens of a request including its Sq new ones; query row t of
 *     Sq sees seq_len - (Sq-1-t) tokens, clamped at 0 ([vLLM-MLA, Triton MLA section]).
 *   - An FP8 row holds 576 e4m3 bytes, then k_scale (fp32) at byte 576 and v_scale (fp32)
 *     at byte 580; K dims are dequantised with k_scale and V dims with v_scale
 *     ([vLLM-MLA, cache shape section]: two fp32 scales, one for K and one for V).
 *
 * Build: gcc -O2 -fopenmp -shared -fPIC (OpenMP only splits independent (row, head) items
 * across cores; each item is computed by the same sequential loops).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Dimensions fixed by the DeepSeek-V3 shape quoted in [vLLM-MLA, model layer section]:
 * kv_lora_rank 512, qk_rope_head_dim 64, qk_nope_head_dim 128, v_head_dim 128. */
#define ORC_L 512
#define ORC_R 64
#define ORC_D (ORC_L + ORC_R) /* 576: one cached row = [kv_c (512) || k_pe (64)] */
#define ORC_P 128
#define ORC_V 128
#define ORC_PAGE 64 /* FlashMLA's only page size, [vLLM-MLA, cache shape section] */

enum { ORC_KV_BF16 = 0, ORC_KV_FP8 = 1 };

/* ------------------------------------------------------------------------------------------
 * Element formats, decoded from their definitions.
 * ---------------------------------------------------------------------------------------- */

/* bfloat16 is the upper half of an IEEE-754 binary32 word. */
double oracle_bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 is NaN; exponent field 0 encodes subnormals m/8 * 2^-6. */
double oracle_e4m3_value(uint8_t b)
{
    int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(8.0 + (double)m, e - 10); /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

void oracle_widen_bf16(const uint16_t* src, int64_t n, double* dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_bf16_value(src[i]);
}

void oracle_widen_e4m3(const uint8_t* src, int64_t n, double* dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = oracle_e4m3_value(src[i]);
}

/* Bytes per cached token per layer: 576 x 2 for bf16, 576 + 2 x 4 for FP8
 * ([vLLM-MLA, cache shape section]; [vLLM-MLA, numbers section]). */
int64_t oracle_row_bytes(int kv_dtype)
{
    return kv_dtype == ORC_KV_BF16 ? (int64_t)ORC_D * 2 : (int64_t)ORC_D + 2 * 4;
}

/* ------------------------------------------------------------------------------------------
 * Paged cache access: token j of a request lives in physical block block_table[j / 64],
 * row j % 64 ([vLLM-MLA, FlashMLA section]: cache [num_pages, page_size, 576] + block table).
 * Writes the K view (576 values) and the V view (first 512 values of the same row).
 * Returns -1 if the block id is outside [0, num_blocks).
 * ---------------------------------------------------------------------------------------- */
typedef struct {
    const uint8_t* base;
    int kv_dtype;
    int64_t num_blocks;
} orc_cache;

static int orc_fetch(const orc_cache* c, const int32_t* bt_row, int64_t j, double* k, double* v)
{
    int64_t blk = bt_row[j / ORC_PAGE];
    int64_t off = j % ORC_PAGE;
    if (blk < 0 || blk >= c->num_blocks)
        return -1;
    int64_t rb = oracle_row_bytes(c->kv_dtype);
    const uint8_t* row = c->base + (blk * ORC_PAGE + off) * rb;
    if (c->kv_dtype == ORC_KV_BF16) {
        for (int d = 0; d < ORC_D; ++d) {
            uint16_t h;
            memcpy(&h, row + 2 * d, 2);
            k[d] = oracle_bf16_value(h);
        }
        for (int d = 0; d < ORC_L; ++d)
            v[d] = k[d]; /* V is the latent part of the same row ([vLLM-MLA, cache shape]) */
    } else {
        float ks, vs;
        memcpy(&ks, row + ORC_D, 4);
        memcpy(&vs, row + ORC_D + 4, 4);
        for (int d = 0; d < ORC_D; ++d)
            k[d] = oracle_e4m3_value(row[d]) * (double)ks;
        for (int d = 0; d < ORC_L; ++d)
            v[d] = oracle_e4m3_value(row[d]) * (double)vs;
    }
    return 0;
}

/* Number of KV tokens visible to query row t of a request with Sq query rows
 * ([vLLM-MLA, Triton MLA section]: seq_lens + arange(1 - q, 1), clamped at 0). */
int64_t oracle_row_len(int32_t seq_len, int Sq, int t)
{
    int64_t n = (int64_t)seq_len - (int64_t)(Sq - 1 - t);
    return n < 0 ? 0 : n;
}

/* ------------------------------------------------------------------------------------------
 * Absorbed attention of ONE query row and ONE head over tokens [j0, j1) of its request
 * ([vLLM-MLA, two-algorithms section], data-movement-friendly form):
 *     s_j  = scale * < q(576), [kv_c_j || k_pe_j] >
 *     lse  = ln sum_j exp(s_j)
 *     o    = sum_j exp(s_j - lse) * kv_c_j            (512-dim latent output)
 * Two plain passes: all logits and their max, then the weights and the weighted sum.
 * An empty range gives o = 0, lse = -inf. Returns -1 on a bad block id.
 * ---------------------------------------------------------------------------------------- */
int oracle_attend_range(const double* q, const orc_cache* c, const int32_t* bt_row,
                        int64_t j0, int64_t j1, double scale, double* o, double* lse)
{
    for (int d = 0; d < ORC_L; ++d)
        o[d] = 0.0;
    if (j1 <= j0) {
        *lse = -INFINITY;
        return 0;
    }
    int64_t n = j1 - j0;
    double* s = (double*)malloc((size_t)n * sizeof(double));
    double k[ORC_D], v[ORC_L];
    double m = -INFINITY;
    int rc = 0;
    for (int64_t j = j0; j < j1 && rc == 0; ++j) {
        if (orc_fetch(c, bt_row, j, k, v) != 0) {
            rc = -1;
            break;
        }
        double dot = 0.0;
        for (int d = 0; d < ORC_D; ++d)
            dot += q[d] * k[d];
        s[j - j0] = scale * dot;
        if (s[j - j0] > m)
            m = s[j - j0];
    }
    if (rc == 0) {
        double sum = 0.0;
        for (int64_t j = j0; j < j1; ++j) {
            orc_fetch(c, bt_row, j, k, v);
            double w = exp(s[j - j0] - m);
            sum += w;
            for (int d = 0; d < ORC_L; ++d)
                o[d] += w * v[d];
        }
        for (int d = 0; d < ORC_L; ++d)
            o[d] /= sum;
        *lse = m + log(sum);
    }
    free(s);
    return rc;
}

/* ------------------------------------------------------------------------------------------
 * Merge of S partial states of one (row, head) ([vLLM-MLA, Prefill section], merge_attn_states;
 * [vLLM-MLA, Triton MLA section], stage 2 of split-KV):
 *     M = max_s lse_s,  w_s = exp(lse_s - M),  lse = M + ln sum_s w_s,  o = sum_s w_s o_s / sum_s w_s
 * Partials with lse = -inf carry zero weight; if all are empty, o = 0 and lse = -inf.
 * ---------------------------------------------------------------------------------------- */
void oracle_merge(const double* o_parts, const double* lse_parts, int S, double* o, double* lse)
{
    double M = -INFINITY;
    for (int s = 0; s < S; ++s)
        if (lse_parts[s] > M)
            M = lse_parts[s];
    for (int d = 0; d < ORC_L; ++d)
        o[d] = 0.0;
    if (M == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double wsum = 0.0;
    for (int s = 0; s < S; ++s) {
        if (lse_parts[s] == -INFINITY)
            continue;
        double w = exp(lse_parts[s] - M);
        wsum += w;
        for (int d = 0; d < ORC_L; ++d)
            o[d] += w * o_parts[(int64_t)s * ORC_L + d];
    }
    for (int d = 0; d < ORC_L; ++d)
        o[d] /= wsum;
    *lse = M + log(wsum);
}

/* ------------------------------------------------------------------------------------------
 * Batched absorbed decode (route A) over a selection of (b, t, h) items.
 *   q          [B, Sq, H, 576] fp64 (already absorbed and concatenated)
 *   cache      raw bytes, [num_blocks, 64, row_bytes]
 *   block_table[B, max_blocks] int32, seq_lens [B] int32
 *   sel        n_sel triples (b, t, h); NULL means every item in (b, t, h) order
 *   chunk      0: attend over the whole row at once. > 0: split the row's tokens into ranges of
 *              `chunk` tokens, attend each range separately and combine them with oracle_merge
 *              (the split-KV path, [vLLM-MLA, Triton MLA section]).
 *   o_latent   [n_items, 512], lse [n_items]
 * Returns 0, or -1 if any visited block id was out of range.
 * ---------------------------------------------------------------------------------------- */
int oracle_decode_absorbed(const double* q, const uint8_t* cache, int kv_dtype, int64_t num_blocks,
                           const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                           int B, int Sq, int H, double scale, int64_t chunk,
                           const int32_t* sel, int64_t n_sel, double* o_latent, double* lse)
{
    orc_cache c = {cache, kv_dtype, num_blocks};
    int64_t n_items = sel ? n_sel : (int64_t)B * Sq * H;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t i = 0; i < n_items; ++i) {
        int64_t b, t, h;
        if (sel) {
            b = sel[3 * i];
            t = sel[3 * i + 1];
            h = sel[3 * i + 2];
        } else {
            b = i / ((int64_t)Sq * H);
            t = (i / H) % Sq;
            h = i % H;
        }
        const double* qr = q + ((b * Sq + t) * H + h) * ORC_D;
        const int32_t* bt = block_table + b * (int64_t)max_blocks;
        int64_t n = oracle_row_len(seq_lens[b], Sq, (int)t);
        double* o = o_latent + i * ORC_L;
        if (chunk <= 0) {
            bad |= oracle_attend_range(qr, &c, bt, 0, n, scale, o, &lse[i]) != 0;
        } else {
            int64_t S = n == 0 ? 1 : (n + chunk - 1) / chunk;
            double* op = (double*)malloc((size_t)S * ORC_L * sizeof(double));
            double* lp = (double*)malloc((size_t)S * sizeof(double));
            for (int64_t s = 0; s < S; ++s) {
                int64_t j0 = s * chunk, j1 = j0 + chunk < n ? j0 + chunk : n;
                bad |= oracle_attend_range(qr, &c, bt, j0, j1, scale, op + s * ORC_L, &lp[s]) != 0;
            }
            oracle_merge(op, lp, (int)S, o, &lse[i]);
            free(op);
            free(lp);
        }
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------------------
 * Query absorption ([vLLM-MLA, weight-preparation and two-algorithms sections];
 * [TRT-TP, absorption section]):
 *     ql_nope[t, h, l] = sum_p q_nope[t, h, p] * W_UK_T[h, p, l]     (128 -> 512)
 *     q[t, h, :] = [ ql_nope[t, h, :] || q_pe[t, h, :] ]              (576)
 * q_nope element (t, h, p) is at t*sn_t + h*sn_h + p; q_pe (t, h, r) at t*sp_t + h*sp_h + r.
 * W_UK_T is [H, 128, 512] (vLLM layout W_UK.permute(1, 2, 0)). Output q_out [T, H, 576] fp64.
 * ---------------------------------------------------------------------------------------- */
void oracle_absorb_q(const uint16_t* q_nope, int64_t sn_t, int64_t sn_h, const uint16_t* q_pe,
                     int64_t sp_t, int64_t sp_h, const uint16_t* w_uk_t, int T, int H, double* q_out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t th = 0; th < (int64_t)T * H; ++th) {
        int64_t t = th / H, h = th % H;
        double qn[ORC_P];
        for (int p = 0; p < ORC_P; ++p)
            qn[p] = oracle_bf16_value(q_nope[t * sn_t + h * sn_h + p]);
        double* out = q_out + th * ORC_D;
        for (int l = 0; l < ORC_L; ++l) {
            double acc = 0.0;
            for (int p = 0; p < ORC_P; ++p)
                acc += qn[p] * oracle_bf16_value(w_uk_t[(h * ORC_P + p) * ORC_L + l]);
            out[l] = acc;
        }
        for (int r = 0; r < ORC_R; ++r)
            out[ORC_L + r] = oracle_bf16_value(q_pe[t * sp_t + h * sp_h + r]);
    }
}

/* ------------------------------------------------------------------------------------------
 * Output up-projection ([vLLM-MLA, two-algorithms section], _v_up_proj):
 *     o[t, h, v] = sum_l o_latent[t, h, l] * W_UV[h, l, v]          (512 -> 128)
 * o_latent [T, H, 512] fp64, W_UV [H, 512, 128] bf16, o [T, H, 128] fp64.
 * ---------------------------------------------------------------------------------------- */
void oracle_out_proj(const double* o_latent, const uint16_t* w_uv, int T, int H, double* o)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t th = 0; th < (int64_t)T * H; ++th) {
        int64_t h = th % H;
        const double* x = o_latent + th * ORC_L;
        for (int vv = 0; vv < ORC_V; ++vv) {
            double acc = 0.0;
            for (int l = 0; l < ORC_L; ++l)
                acc += x[l] * oracle_bf16_value(w_uv[(h * ORC_L + l) * ORC_V + vv]);
            o[th * ORC_V + vv] = acc;
        }
    }
}

/* ------------------------------------------------------------------------------------------
 * Non-absorbed decode (route N, the "compute-friendly" form of [vLLM-MLA, two-algorithms
 * section]): every visible cached latent is up-projected per head into full K and V,
 *     k_nope_j[p] = sum_l kv_c_j[l] * W_UK[l, h, p]   (W_UK[l, h, p] = W_UK_T[h, p, l])
 *     v_j[v]      = sum_l kv_c_j[l] * W_UV[h, l, v]
 *     s_j = scale * ( <q_nope, k_nope_j> + <q_pe, k_pe_j> )            (192-dim dot product)
 * followed by standard softmax attention:  o = sum_j p_j v_j  (128), lse = ln sum_j exp(s_j).
 * It also returns o_latent = sum_j p_j kv_c_j (512) so that decode can be checked on its own.
 * For an FP8 cache the K-side latent uses k_scale and the V-side latent v_scale.
 *   q_nope [B, Sq, H, 128] bf16, q_pe [B, Sq, H, 64] bf16 (contiguous)
 * Outputs per selected item: o [., 128], o_latent [., 512], lse [.].
 * ---------------------------------------------------------------------------------------- */
int oracle_decode_nonabsorbed(const uint16_t* q_nope, const uint16_t* q_pe, const uint8_t* cache,
                              int kv_dtype, int64_t num_blocks, const int32_t* block_table,
                              int max_blocks, const int32_t* seq_lens, const uint16_t* w_uk_t,
                              const uint16_t* w_uv, int B, int Sq, int H, double scale,
                              const int32_t* sel, int64_t n_sel, double* o, double* o_latent,
                              double* lse)
{
    orc_cache c = {cache, kv_dtype, num_blocks};
    int64_t n_items = sel ? n_sel : (int64_t)B * Sq * H;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t i = 0; i < n_items; ++i) {
        int64_t b, t, h;
        if (sel) {
            b = sel[3 * i];
            t = sel[3 * i + 1];
            h = sel[3 * i + 2];
        } else {
            b = i / ((int64_t)Sq * H);
            t = (i / H) % Sq;
            h = i % H;
        }
        int64_t qi = (b * Sq + t) * H + h;
        double qn[ORC_P], qp[ORC_R];
        for (int p = 0; p < ORC_P; ++p)
            qn[p] = oracle_bf16_value(q_nope[qi * ORC_P + p]);
        for (int r = 0; r < ORC_R; ++r)
            qp[r] = oracle_bf16_value(q_pe[qi * ORC_R + r]);
        const int32_t* bt = block_table + b * (int64_t)max_blocks;
        int64_t n = oracle_row_len(seq_lens[b], Sq, (int)t);
        double* oo = o + i * ORC_V;
        double* ol = o_latent + i * ORC_L;
        for (int d = 0; d < ORC_V; ++d)
            oo[d] = 0.0;
        for (int d = 0; d < ORC_L; ++d)
            ol[d] = 0.0;
        if (n == 0) {
            lse[i] = -INFINITY;
            continue;
        }
        double* s = (double*)malloc((size_t)n * sizeof(double));
        double k[ORC_D], cv[ORC_L];
        double m = -INFINITY;
        int rc = 0;
        /* pass 1: logits through the up-projected key */
        for (int64_t j = 0; j < n; ++j) {
            if (orc_fetch(&c, bt, j, k, cv) != 0) {
                rc = -1;
                break;
            }
            double dot = 0.0;
            for (int p = 0; p < ORC_P; ++p) {
                double kn = 0.0;
                for (int l = 0; l < ORC_L; ++l)
                    kn += k[l] * oracle_bf16_value(w_uk_t[(h * ORC_P + p) * ORC_L + l]);
                dot += qn[p] * kn;
            }
            for (int r = 0; r < ORC_R; ++r)
                dot += qp[r] * k[ORC_L + r];
            s[j] = scale * dot;
            if (s[j] > m)
                m = s[j];
        }
        if (rc != 0) {
            bad = 1;
            free(s);
            continue;
        }
        /* pass 2: softmax weights, up-projected values */
        double sum = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            orc_fetch(&c, bt, j, k, cv);
            double w = exp(s[j] - m);
            sum += w;
            for (int vv = 0; vv < ORC_V; ++vv) {
                double val = 0.0;
                for (int l = 0; l < ORC_L; ++l)
                    val += cv[l] * oracle_bf16_value(w_uv[(h * ORC_L + l) * ORC_V + vv]);
                oo[vv] += w * val;
            }
            for (int l = 0; l < ORC_L; ++l)
                ol[l] += w * cv[l];
        }
        for (int d = 0; d < ORC_V; ++d)
            oo[d] /= sum;
        for (int d = 0; d < ORC_L; ++d)
            ol[d] /= sum;
        lse[i] = m + log(sum);
        free(s);
    }
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------------------------------
 * Split count used by the Triton backend ([vLLM-MLA, Triton MLA section], _compute_num_kv_splits;
 * [Triton-MLA, Schlüsseldateien]):  min(next_pow2(max(1, max_seq_len // 512)), 2 * sm_count).
 * ---------------------------------------------------------------------------------------- */
int oracle_default_num_splits(int max_seq_len, int sm_count)
{
    int ideal = max_seq_len / 512;
    if (ideal < 1)
        ideal = 1;
    int p2 = 1;
    while (p2 < ideal)
        p2 *= 2;
    int cap = 2 * sm_count;
    return p2 < cap ? p2 : cap;
}

/* ------------------------------------------------------------------------------------------
 * E4M3 encoding, from the format's definition: the finite value nearest to x, ties to the code
 * with an even mantissa (round to nearest even), magnitudes beyond the largest finite value
 * (448) saturate to it, NaN stays NaN. Found by plain search over the 127 non-negative finite
 * codes, so that nothing but the decoder above is assumed.
 * ---------------------------------------------------------------------------------------- */
uint8_t oracle_e4m3_encode(float x)
{
    if (isnan(x))
        return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double a = fabs((double)x);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double err = fabs(oracle_e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

/* ------------------------------------------------------------------------------------------
 * KV cache write ([vLLM-MLA, cache write section]): token t's row [kv_c[t] (512) || k_pe[t]
 * (64)] is stored at slot s = slot_mapping[t] = block * 64 + offset (the block manager's
 * physical block and in-page offset); s < 0 marks a padding token and is skipped.
 *   bf16 cache: the 576 bf16 values are copied.
 *   FP8 cache (584-byte rows, [vLLM-MLA, cache shape and numbers sections]): the row's scale is
 *   kv_scale when kv_scale > 0 (one static scale, as the page's scale parameter), otherwise
 *   amax(|x|) / 448 over the row's 576 values (1 when amax is 0). The write multiplies each
 *   value by the scale's reciprocal ([vLLM-MLA, cache write section]: with a scale of exactly 1
 *   the multiplication is the step that can be skipped) and stores e4m3(x * (1 / scale));
 *   k_scale (byte 576) and v_scale (byte 580) both hold the scale. amax / 448, 1 / scale, the
 *   product and the rounding decision are all taken in binary32, the precision the device uses.
 * Returns the number of tokens whose slot lies beyond the cache (those rows are skipped).
 * ---------------------------------------------------------------------------------------- */
int64_t oracle_cache_write(const uint16_t* kv_c, int64_t st_c, const uint16_t* k_pe, int64_t st_pe,
                           const int64_t* slot_mapping, int64_t T, int kv_dtype, float kv_scale,
                           uint8_t* cache, int64_t num_blocks)
{
    const int64_t rb = oracle_row_bytes(kv_dtype);
    int64_t bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        const int64_t s = slot_mapping[t];
        if (s < 0)
            continue;
        if (s >= num_blocks * ORC_PAGE) {
            ++bad;
            continue;
        }
        uint16_t row[ORC_D];
        for (int d = 0; d < ORC_L; ++d)
            row[d] = kv_c[t * st_c + d];
        for (int r = 0; r < ORC_R; ++r)
            row[ORC_L + r] = k_pe[t * st_pe + r];
        uint8_t* dst = cache + s * rb;
        if (kv_dtype == ORC_KV_BF16) {
            memcpy(dst, row, sizeof row);
            continue;
        }
        float scale = kv_scale;
        if (!(scale > 0.0f)) {
            float amax = 0.0f;
            for (int d = 0; d < ORC_D; ++d) {
                const float a = fabsf((float)oracle_bf16_value(row[d]));
                if (a > amax)
                    amax = a;
            }
            scale = amax > 0.0f ? amax / 448.0f : 1.0f;
        }
        const float inv = 1.0f / scale;
        for (int d = 0; d < ORC_D; ++d)
            dst[d] = oracle_e4m3_encode((float)oracle_bf16_value(row[d]) * inv);
        memcpy(dst + ORC_D, &scale, 4);
        memcpy(dst + ORC_D + 4, &scale, 4);
    }
    return bad;
}

/* ------------------------------------------------------------------------------------------
 * Variable-length query rows ([vLLM-MLA, metadata section]: the VARLEN query-length support
 * lets a speculative-decoding verification batch mix requests with 1, 2, 3 ... query tokens).
 * Query rows are packed request after request: request b owns rows
 * [query_start_loc[b], query_start_loc[b + 1]), and its row t sees
 * seq_lens[b] - (q_len_b - 1 - t) tokens (clamped at 0), as a uniform batch with Sq = q_len_b.
 * q is [total_q, H, 576]; o_latent [total_q, H, 512]; lse [total_q, H].
 * ---------------------------------------------------------------------------------------- */
int oracle_decode_varlen(const double* q, const uint8_t* cache, int kv_dtype, int64_t num_blocks,
                         const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                         const int32_t* query_start_loc, int B, int H, double scale,
                         double* o_latent, double* lse)
{
    orc_cache c = {cache, kv_dtype, num_blocks};
    const int64_t total_q = query_start_loc[B];
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t i = 0; i < total_q * H; ++i) {
        const int64_t r = i / H, h = i % H;
        int b = 0;
        while (b < B && query_start_loc[b + 1] <= r)
            ++b;
        const int q_len = query_start_loc[b + 1] - query_start_loc[b];
        const int t = (int)(r - query_start_loc[b]);
        const int32_t* bt = block_table + (int64_t)b * max_blocks;
        const int64_t n = oracle_row_len(seq_lens[b], q_len, t);
        bad |= oracle_attend_range(q + (r * H + h) * ORC_D, &c, bt, 0, n, scale, o_latent + i * ORC_L, &lse[i]) != 0;
    }
    return bad ? -1 : 0;
}

/* ==========================================================================================
 * Prefill, the compute-friendly route ([vLLM-MLA, Prefill section]). A prefill request b has
 * ctx_lens[b] tokens already in the paged cache (its context, positions 0 .. ctx-1) and q_len_b
 * new tokens (positions ctx .. ctx + q_len - 1), packed request after request by
 * query_start_loc. Keys and values are up-projected per head (no absorption):
 *     k_nope_j[p] = sum_l c_j[l] W_UK_T[h, p, l],   k_j = [k_nope_j (128) || k_pe_j (64)]
 *     v_j[v]      = sum_l c_j[l] W_UV[h, l, v]
 * and attention is standard MHA with a 192-dim q.k and a 128-dim output. The page's order:
 *   1. the new tokens attend causally among themselves (new token i is visible to query t of
 *      the same request iff i <= t); their k/v come from the step's own kv_c / k_pe;
 *   2. the context is processed in chunks of at most chunk_rows gathered rows: each chunk is
 *      gathered from the paged cache (FP8 rows dequantised: the K side with k_scale, the V side
 *      with v_scale), up-projected, and attended by every query of the requests it holds (all
 *      context tokens precede the new ones, so no mask); the chunk results are accumulated;
 *   3. the context result (prefix) and the new-token result (suffix) are merged by their lse
 *      (merge_attn_states); a request without context has an empty prefix (o = 0, lse = -inf).
 * ======================================================================================== */

/* Merge of two partial states of one (row, head) with n output dims -- the same formula as
 * oracle_merge, for the prefix / suffix pair:  M = max(lse_a, lse_b), w = exp(lse - M). */
static void orc_merge_pair(double* o_acc, double* lse_acc, const double* o_new, double lse_new, int n)
{
    const double la = *lse_acc;
    const double M = la > lse_new ? la : lse_new;
    if (M == -INFINITY)
        return; /* both empty: o stays 0, lse -inf */
    const double wa = la == -INFINITY ? 0.0 : exp(la - M);
    const double wb = lse_new == -INFINITY ? 0.0 : exp(lse_new - M);
    for (int d = 0; d < n; ++d)
        o_acc[d] = (wa * o_acc[d] + wb * o_new[d]) / (wa + wb);
    *lse_acc = M + log(wa + wb);
}

/* ------------------------------------------------------------------------------------------
 * Context chunk plan ([vLLM-MLA, Prefill section]: the contexts are packed into chunks of at
 * most row_budget rows; a request that does not fit is cut, and every chunk starts on a page
 * boundary of its request). Requests are taken in order; a request's remaining context goes
 * into the open chunk whole if it fits, otherwise as many whole pages as still fit, and a chunk
 * with no room for a page is closed. Each emitted piece is (chunk, request, first position,
 * token count); pieces of one chunk are consecutive. chunk_rows < 64 is rejected (-1), as no
 * page would fit. Returns the number of pieces (pieces may be NULL to count them).
 * ---------------------------------------------------------------------------------------- */
int64_t oracle_prefill_chunks(const int32_t* ctx_lens, int B, int64_t chunk_rows, int64_t* pieces)
{
    if (chunk_rows < ORC_PAGE)
        return -1;
    int64_t n = 0, chunk = 0, used = 0;
    for (int b = 0; b < B; ++b) {
        int64_t pos = 0;
        const int64_t len = ctx_lens[b] > 0 ? ctx_lens[b] : 0;
        while (pos < len) {
            int64_t take = len - pos;
            if (take > chunk_rows - used) {
                take = (chunk_rows - used) / ORC_PAGE * ORC_PAGE;
                if (take == 0) { /* no whole page fits: close the chunk */
                    ++chunk;
                    used = 0;
                    continue;
                }
            }
            if (pieces) {
                pieces[4 * n + 0] = chunk;
                pieces[4 * n + 1] = b;
                pieces[4 * n + 2] = pos;
                pieces[4 * n + 3] = take;
            }
            ++n;
            used += take;
            pos += take;
        }
    }
    return n;
}

/* Up-projection of one latent row for head h: k_nope (128) from the K-side latent ck, v (128)
 * from the V-side latent cv (the same values for a bf16 cache). */
static void orc_up_project(const double* ck, const double* cv, const uint16_t* w_uk_t,
                           const uint16_t* w_uv, int64_t h, double* k_nope, double* v)
{
    for (int p = 0; p < ORC_P; ++p) {
        double acc = 0.0;
        for (int l = 0; l < ORC_L; ++l)
            acc += ck[l] * oracle_bf16_value(w_uk_t[(h * ORC_P + p) * ORC_L + l]);
        k_nope[p] = acc;
    }
    for (int vv = 0; vv < ORC_V; ++vv) {
        double acc = 0.0;
        for (int l = 0; l < ORC_L; ++l)
            acc += cv[l] * oracle_bf16_value(w_uv[(h * ORC_L + l) * ORC_V + vv]);
        v[vv] = acc;
    }
}

/* Standard attention of one query (192 dims: q_nope 128 || q_pe 64) over n keys, each 192 dims
 * (k_nope || k_pe) with a 128-dim value: two plain passes (logits and their max, then weights
 * and the weighted sum). n = 0 gives o = 0, lse = -inf. */
static void orc_mha_row(const double* q, const double* k, const double* v, int64_t n, double scale,
                        double* o, double* lse)
{
    for (int d = 0; d < ORC_V; ++d)
        o[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return;
    }
    double* s = (double*)malloc((size_t)n * sizeof(double));
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < ORC_P + ORC_R; ++d)
            dot += q[d] * k[j * (ORC_P + ORC_R) + d];
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double w = exp(s[j] - m);
        sum += w;
        for (int d = 0; d < ORC_V; ++d)
            o[d] += w * v[j * ORC_V + d];
    }
    for (int d = 0; d < ORC_V; ++d)
        o[d] /= sum;
    *lse = m + log(sum);
    free(s);
}

/* ------------------------------------------------------------------------------------------
 *   q          [total_q, H, 192] bf16 (q_nope || q_pe per head, RoPE already applied)
 *   kv_c_new   [total_q, 512] bf16, k_pe_new [total_q, 64] bf16: the new tokens' latent rows
 *   cache      raw bytes [num_blocks, 64, row_bytes] holding each request's context
 *   ctx_lens   [B], query_start_loc [B + 1] (total_q = query_start_loc[B])
 *   chunk_rows the context row budget per chunk (>= 64)
 *   o          [total_q, H, 128], lse [total_q, H]
 * Returns 0, -1 on a bad block id, -2 on chunk_rows < 64.
 * ---------------------------------------------------------------------------------------- */
int oracle_prefill(const uint16_t* q, const uint16_t* kv_c_new, const uint16_t* k_pe_new,
                   const uint8_t* cache, int kv_dtype, int64_t num_blocks, const int32_t* block_table,
                   int max_blocks, const int32_t* ctx_lens, const int32_t* query_start_loc, int B, int H,
                   const uint16_t* w_uk_t, const uint16_t* w_uv, double scale, int64_t chunk_rows,
                   double* o, double* lse)
{
    const int KD = ORC_P + ORC_R; /* 192 */
    const int64_t total_q = query_start_loc[B];
    const int64_t n_pieces = oracle_prefill_chunks(ctx_lens, B, chunk_rows, NULL);
    if (n_pieces < 0)
        return -2;
    int64_t* pieces = (int64_t*)malloc((size_t)(n_pieces > 0 ? n_pieces : 1) * 4 * sizeof(int64_t));
    oracle_prefill_chunks(ctx_lens, B, chunk_rows, pieces);
    orc_cache c = {cache, kv_dtype, num_blocks};

    /* row r of the packed queries belongs to request req[r] */
    int* req = (int*)malloc((size_t)(total_q > 0 ? total_q : 1) * sizeof(int));
    for (int b = 0; b < B; ++b)
        for (int64_t r = query_start_loc[b]; r < query_start_loc[b + 1]; ++r)
            req[r] = b;

    /* ---- step 1: the new tokens (suffix) ---- */
    double* kn = (double*)malloc((size_t)(total_q > 0 ? total_q : 1) * H * KD * sizeof(double));
    double* vn = (double*)malloc((size_t)(total_q > 0 ? total_q : 1) * H * ORC_V * sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < total_q * H; ++i) {
        const int64_t r = i / H, h = i % H;
        double cl[ORC_L];
        for (int l = 0; l < ORC_L; ++l)
            cl[l] = oracle_bf16_value(kv_c_new[r * ORC_L + l]);
        /* key / value rows stored head-major so that one head's keys are contiguous */
        double* kk = kn + (h * total_q + r) * KD;
        orc_up_project(cl, cl, w_uk_t, w_uv, h, kk, vn + (h * total_q + r) * ORC_V);
        for (int e = 0; e < ORC_R; ++e)
            kk[ORC_P + e] = oracle_bf16_value(k_pe_new[r * ORC_R + e]);
    }
    double* o_suf = (double*)malloc((size_t)(total_q > 0 ? total_q : 1) * H * ORC_V * sizeof(double));
    double* l_suf = (double*)malloc((size_t)(total_q > 0 ? total_q : 1) * H * sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < total_q * H; ++i) {
        const int64_t r = i / H, h = i % H;
        const int b = req[r];
        const int64_t first = query_start_loc[b];
        double qq[ORC_P + ORC_R];
        for (int d = 0; d < KD; ++d)
            qq[d] = oracle_bf16_value(q[(r * H + h) * KD + d]);
        /* causal: new tokens first .. r of the request */
        orc_mha_row(qq, kn + (h * total_q + first) * KD, vn + (h * total_q + first) * ORC_V,
                    r - first + 1, scale, o_suf + i * ORC_V, &l_suf[i]);
    }
    free(kn);
    free(vn);

    /* ---- step 2: the context, chunk by chunk (prefix) ---- */
    for (int64_t i = 0; i < total_q * H; ++i) {
        for (int d = 0; d < ORC_V; ++d)
            o[i * ORC_V + d] = 0.0;
        lse[i] = -INFINITY;
    }
    int bad = 0;
    int64_t p0 = 0;
    while (p0 < n_pieces) {
        int64_t p1 = p0;
        int64_t rows = 0;
        while (p1 < n_pieces && pieces[4 * p1] == pieces[4 * p0])
            rows += pieces[4 * p1++ + 3];
        /* gather the chunk's rows (K-side and V-side latent + rope) */
        double* gk = (double*)malloc((size_t)rows * ORC_D * sizeof(double));
        double* gv = (double*)malloc((size_t)rows * ORC_L * sizeof(double));
        int64_t at = 0;
        for (int64_t p = p0; p < p1; ++p) {
            const int b = (int)pieces[4 * p + 1];
            const int32_t* bt = block_table + (int64_t)b * max_blocks;
            for (int64_t j = 0; j < pieces[4 * p + 3]; ++j, ++at)
                if (orc_fetch(&c, bt, pieces[4 * p + 2] + j, gk + at * ORC_D, gv + at * ORC_L) != 0) {
                    bad = 1;
                    for (int d = 0; d < ORC_D; ++d)
                        gk[at * ORC_D + d] = 0.0;
                    for (int d = 0; d < ORC_L; ++d)
                        gv[at * ORC_L + d] = 0.0;
                }
        }
        /* up-project every gathered row for every head */
        double* kc = (double*)malloc((size_t)rows * H * KD * sizeof(double));
        double* vc = (double*)malloc((size_t)rows * H * ORC_V * sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t i = 0; i < rows * H; ++i) {
            const int64_t j = i / H, h = i % H;
            double* kk = kc + (h * rows + j) * KD;
            orc_up_project(gk + j * ORC_D, gv + j * ORC_L, w_uk_t, w_uv, h, kk, vc + (h * rows + j) * ORC_V);
            for (int e = 0; e < ORC_R; ++e)
                kk[ORC_P + e] = gk[j * ORC_D + ORC_L + e];
        }
        /* every query of a request in this chunk attends to all of that request's rows here */
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t i = 0; i < total_q * H; ++i) {
            const int64_t r = i / H, h = i % H;
            const int b = req[r];
            int64_t off = 0, n = 0;
            for (int64_t p = p0; p < p1; ++p) {
                if (pieces[4 * p + 1] == b) {
                    n = pieces[4 * p + 3];
                    break;
                }
                off += pieces[4 * p + 3];
            }
            if (n == 0)
                continue; /* an empty partial carries no weight */
            double qq[ORC_P + ORC_R], oc[ORC_V], lc;
            for (int d = 0; d < KD; ++d)
                qq[d] = oracle_bf16_value(q[(r * H + h) * KD + d]);
            orc_mha_row(qq, kc + (h * rows + off) * KD, vc + (h * rows + off) * ORC_V, n, scale, oc, &lc);
            orc_merge_pair(o + i * ORC_V, &lse[i], oc, lc, ORC_V);
        }
        free(gk);
        free(gv);
        free(kc);
        free(vc);
        p0 = p1;
    }

    /* ---- step 3: merge prefix and suffix ---- */
    for (int64_t i = 0; i < total_q * H; ++i)
        orc_merge_pair(o + i * ORC_V, &lse[i], o_suf + i * ORC_V, l_suf[i], ORC_V);
    free(o_suf);
    free(l_suf);
    free(req);
    free(pieces);
    return bad ? -1 : 0;
}
