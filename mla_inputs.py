"""Seeded synthetic inputs for MLA latent-KV decode.

This module is shared by the CUDA path's tests/benchmark and by the CPU oracle's callers. It
holds no attention arithmetic: it only draws seeded random numbers, rounds them to the storage
formats (bf16, OCP FP8 E4M3) and lays them out as a paged cache with a block table, following
the shapes of the workloads below. Poisoned bytes (NaN) fill every cache row that no request
may read, so an over-read shows up as NaN in the outputs.

Workloads (DeepSeek-V3 MLA shape: kv_lora_rank 512, rope 64, qk_nope 128, v 128, page 64):
  tiny     B=2,   Sq=1, H=16,  ctx {128, 300},               bf16 cache, seed 0
  dsv3     B=64,  Sq=1, H=128, ctx 4096,                     bf16 cache, seed 1
  ragged   B=128, Sq=1, H=128, ctx log-uniform in [1, 32768] bf16 cache, seed 2
  fp8      B=128, Sq=1, H=128, ctx 8192,                     FP8 cache (584-byte rows), seed 3
  long_mtp B=4,   Sq=2, H=128, ctx 131072 (causal rows),     bf16 cache, seed 4
q and cache values are N(0,1); W_UK_T / W_UV are N(0, 1/512); scale = 1/sqrt(192).
"""
from __future__ import annotations

import math

import numpy as np

L, R, D, P, V, PAGE = 512, 64, 576, 128, 128, 64
KV_BF16, KV_FP8 = 0, 1
ROW_BYTES = {KV_BF16: 2 * D, KV_FP8: D + 8}
BF16_NAN = 0x7FC0
E4M3_NAN = 0x7F
# softmax scale of the 192-dim (128 nope + 64 rope) query-key product, rounded once to fp32
SCALE = float(np.float32(1.0 / math.sqrt(P + R)))

WORKLOADS = {
    "tiny": dict(B=2, Sq=1, H=16, lens=[128, 300], kv=KV_BF16, seed=0),
    "dsv3": dict(B=64, Sq=1, H=128, lens=[4096] * 64, kv=KV_BF16, seed=1),
    "ragged": dict(B=128, Sq=1, H=128, lens="loguniform", kv=KV_BF16, seed=2),
    "fp8": dict(B=128, Sq=1, H=128, lens=[8192] * 128, kv=KV_FP8, seed=3),
    "long_mtp": dict(B=4, Sq=2, H=128, lens=[131072] * 4, kv=KV_BF16, seed=4),
}


# ------------------------------------------------------------------ storage formats
def to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); returns uint16 bits."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def to_e4m3_bits(y) -> np.ndarray:
    """Encode float64 values as OCP FP8 E4M3 codes: round to nearest, ties to even, saturating
    at +-448 (the largest finite value)."""
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), 448.0)
    code = np.zeros(a.shape, np.int64)
    sub = a < 2.0 ** -6
    # subnormals and zero: steps of 2^-9; a result of 8 steps is the smallest normal (code 8)
    code[sub] = np.rint(a[sub] * 2.0 ** 9).astype(np.int64)
    nrm = ~sub
    if nrm.any():
        _, ex = np.frexp(a[nrm])          # a = f * 2^ex, f in [0.5, 1)
        e = ex - 1                        # floor(log2 a), in [-6, 8]
        q = np.rint(a[nrm] / np.ldexp(1.0, e - 3)).astype(np.int64)  # in [8, 16]
        carry = q == 16
        e = np.where(carry, e + 1, e)
        q = np.where(carry, 8, q)
        c = ((e + 7) << 3) | (q - 8)
        code[nrm] = np.minimum(c, 0x7E)   # rounding up past 448 saturates
    sign = np.signbit(y).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


# ------------------------------------------------------------------ lengths and paging
def draw_lengths(spec, B, rng) -> np.ndarray:
    if isinstance(spec, str) and spec == "loguniform":
        u = rng.uniform(0.0, math.log(32768.0), size=B)
        lens = np.clip(np.floor(np.exp(u)), 1, 32768).astype(np.int64)
        forced = [1, 63, 64, 65, 128, 32768]
        lens[: min(B, len(forced))] = forced[: min(B, len(forced))]
        return lens.astype(np.int32)
    return np.asarray(spec, dtype=np.int32)


def make_block_table(lens, rng, spare_blocks=16, extra_cols=0):
    """Random physical placement: num_blocks = sum(ceil(len/64)) + spare, shuffled ids; table
    entries past a request's last page are -1 (never to be read)."""
    pages = (np.asarray(lens, np.int64) + PAGE - 1) // PAGE
    max_blocks = int(max(1, pages.max() if len(pages) else 1)) + extra_cols
    num_blocks = int(pages.sum()) + spare_blocks
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((len(pages), max_blocks), -1, np.int32)
    k = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[k:k + n]
        k += n
    return bt, num_blocks


def valid_row_mask(lens, block_table, num_blocks) -> np.ndarray:
    """[num_blocks, 64] bool: rows that hold a token some request may read."""
    mask = np.zeros((num_blocks, PAGE), bool)
    for b, n in enumerate(np.asarray(lens, np.int64)):
        for p in range((n + PAGE - 1) // PAGE):
            mask[block_table[b, p], : min(PAGE, n - p * PAGE)] = True
    return mask


def make_cache(num_blocks, kv, rng, valid=None, poison=True, chunk_blocks=512):
    """Cache bytes [num_blocks, 64 * row_bytes] (uint8). bf16: N(0,1) values. FP8: N(0,1) values
    quantised per token row with s = amax(|x|)/448 (s = 1 if the row is all zero), the 576 codes
    followed by k_scale = v_scale = s as two little-endian fp32."""
    rb = ROW_BYTES[kv]
    cache = np.empty((num_blocks, PAGE, rb), np.uint8)
    for b0 in range(0, num_blocks, chunk_blocks):
        b1 = min(num_blocks, b0 + chunk_blocks)
        x = rng.standard_normal((b1 - b0, PAGE, D), dtype=np.float32)
        if kv == KV_BF16:
            cache[b0:b1] = to_bf16_bits(x).view(np.uint8).reshape(b1 - b0, PAGE, rb)
        else:
            amax = np.abs(x).max(axis=-1)
            s = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
            codes = to_e4m3_bits(x.astype(np.float64) / s[..., None].astype(np.float64))
            cache[b0:b1, :, :D] = codes
            sc = np.stack([s, s], axis=-1).astype("<f4")
            cache[b0:b1, :, D:] = sc.view(np.uint8).reshape(b1 - b0, PAGE, 8)
    if poison and valid is not None:
        bad = ~valid
        if kv == KV_BF16:
            cache.view(np.uint16)[bad] = BF16_NAN
        else:
            cache[bad, :D] = E4M3_NAN
            nan4 = np.array([np.nan], "<f4").view(np.uint8)
            cache[bad, D:D + 4] = nan4
            cache[bad, D + 4:D + 8] = nan4
    return cache.reshape(num_blocks, PAGE * rb)


def normal_bf16(rng, shape, std=1.0) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x = x * np.float32(std)
    return to_bf16_bits(x)


# ------------------------------------------------------------------ cases
def decode_case(B, Sq, H, lens, kv=KV_BF16, seed=0, spare_blocks=16, poison=True, extra_cols=0):
    """Inputs of mla_decode. Returns a dict of numpy arrays (bf16 as uint16 bits)."""
    rng = np.random.default_rng(seed)
    lens = draw_lengths(lens, B, rng)
    bt, num_blocks = make_block_table(lens, rng, spare_blocks, extra_cols)
    valid = valid_row_mask(lens, bt, num_blocks) if poison else None
    cache = make_cache(num_blocks, kv, rng, valid, poison)
    q = normal_bf16(rng, (B, Sq, H, D))
    return dict(B=B, Sq=Sq, H=H, kv=kv, seq_lens=lens, block_table=bt, num_blocks=num_blocks,
                cache=cache, q=q, scale=SCALE)


def workload_case(name, **over):
    w = dict(WORKLOADS[name])
    w.update(over)
    return decode_case(w["B"], w["Sq"], w["H"], w["lens"], kv=w["kv"], seed=w["seed"])


def e2e_case(B, Sq, H, lens, kv=KV_BF16, seed=0):
    """Inputs of the three calls chained: q_nope/q_pe [B,Sq,H,128/64], W_UK_T [H,128,512],
    W_UV [H,512,128], plus the paged cache of decode_case."""
    c = decode_case(B, Sq, H, lens, kv=kv, seed=seed)
    rng = np.random.default_rng(seed + 1000)
    c["q_nope"] = normal_bf16(rng, (B, Sq, H, P))
    c["q_pe"] = normal_bf16(rng, (B, Sq, H, R))
    c["w_uk_t"] = normal_bf16(rng, (H, P, L), std=1.0 / math.sqrt(512.0))
    c["w_uv"] = normal_bf16(rng, (H, L, V), std=1.0 / math.sqrt(512.0))
    return c


def absorb_case(T, H, seed=0):
    rng = np.random.default_rng(seed)
    return dict(T=T, H=H, q_nope=normal_bf16(rng, (T, H, P)), q_pe=normal_bf16(rng, (T, H, R)),
                w_uk_t=normal_bf16(rng, (H, P, L), std=1.0 / math.sqrt(512.0)))


def out_proj_case(T, H, seed=0):
    rng = np.random.default_rng(seed)
    return dict(T=T, H=H, o_latent=rng.standard_normal((T, H, L), dtype=np.float32),
                w_uv=normal_bf16(rng, (H, L, V), std=1.0 / math.sqrt(512.0)))


def prefill_case(ctx_lens, q_lens, H, kv=KV_BF16, seed=0, spare_blocks=4, poison=True):
    """Inputs of the prefill route: request b has ctx_lens[b] tokens in the paged cache and q_lens[b]
    new tokens, packed by query_start_loc. The block table already covers the new tokens'
    positions (their cache rows are poisoned here; a test that needs them writes them). Returns a
    dict: q [T, H, 192] (q_nope || q_pe), kv_c_new [T, 512], k_pe_new [T, 64] (bf16 bits),
    W_UK_T [H, 128, 512], W_UV [H, 512, 128] (N(0, 1/512)), new_slots [T] int64 (cache slot of
    each new token), plus the cache and its metadata."""
    rng = np.random.default_rng(seed)
    ctx = np.asarray(ctx_lens, np.int32)
    ql = np.asarray(q_lens, np.int32)
    qsl = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    bt, num_blocks = make_block_table(ctx.astype(np.int64) + ql, rng, spare_blocks)
    valid = valid_row_mask(ctx, bt, num_blocks) if poison else None
    cache = make_cache(num_blocks, kv, rng, valid, poison)
    T = int(qsl[-1])
    slots = np.zeros(T, np.int64)
    for b in range(len(ctx)):
        for i in range(int(ql[b])):
            pos = int(ctx[b]) + i
            slots[qsl[b] + i] = int(bt[b, pos // PAGE]) * PAGE + pos % PAGE
    return dict(H=H, kv=kv, ctx_lens=ctx, query_start_loc=qsl, block_table=bt, num_blocks=num_blocks,
                cache=cache, q=normal_bf16(rng, (T, H, P + R)), kv_c_new=normal_bf16(rng, (T, L)),
                k_pe_new=normal_bf16(rng, (T, R)), new_slots=slots,
                w_uk_t=normal_bf16(rng, (H, P, L), std=1.0 / math.sqrt(512.0)),
                w_uv=normal_bf16(rng, (H, L, V), std=1.0 / math.sqrt(512.0)), scale=SCALE)
