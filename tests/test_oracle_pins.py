"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics (no GPU).

Each test checks the oracle against something other than itself: byte counts the pages print,
hand-worked closed forms, library routines (torch SDPA / logsumexp / float8 and bfloat16
conversions, numpy matmul), the absorption identity, and invariants of softmax and of the
split-KV merge.
"""
import math
import os

import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows[parts[0]] = parts[1:]
    return rows


# ----------------------------------------------------------------------------- layouts
def test_row_and_page_bytes_match_pages():
    g = {k: int(v[0]) for k, v in _read_table("layout_bytes.txt").items()}
    assert oracle.row_bytes(oracle.KV_BF16) == g["bf16_row_bytes"]
    assert oracle.row_bytes(oracle.KV_FP8) == g["fp8_row_bytes"]
    assert oracle.PAGE * oracle.row_bytes(oracle.KV_BF16) == g["bf16_page_bytes"]
    assert 61 * oracle.row_bytes(oracle.KV_BF16) == g["bf16_bytes_per_token_61L"]
    assert 61 * oracle.row_bytes(oracle.KV_FP8) == g["fp8_bytes_per_token_61L"]
    assert 131072 // oracle.PAGE == g["pages_for_128k"]
    # the equivalent MHA row: 128 heads x (192 QK + 128 V) x 2 bytes, about 71x the MLA row
    assert 128 * (192 + 128) * 2 == g["mha_equiv_bytes_per_token"]
    assert round(g["mha_equiv_bytes_per_token"] / g["bf16_row_bytes"]) == 71
    assert mi.ROW_BYTES[mi.KV_BF16] == g["bf16_row_bytes"]
    assert mi.ROW_BYTES[mi.KV_FP8] == g["fp8_row_bytes"]


# ----------------------------------------------------------------------------- formats
def test_e4m3_decode_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.widen_e4m3(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def test_bf16_decode_matches_torch():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 1 << 16, size=20000, dtype=np.uint16)
    ours = oracle.widen_bf16(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(ours[fin], ref[fin])


def test_input_encoders_match_library_rounding():
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(50000) * rng.choice([1e-3, 1, 50], 50000)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mi.to_bf16_bits(x), ref)
    # e4m3: compare with brute-force nearest (ties to even code) over the decoded code table
    codes = np.arange(0x7F, dtype=np.uint8)
    table = oracle.widen_e4m3(codes)
    y = np.concatenate([rng.uniform(-460, 460, 20000), rng.uniform(-0.02, 0.02, 20000),
                        (table[:-1] + table[1:]) / 2])  # exact ties
    enc = mi.to_e4m3_bits(y)
    a = np.minimum(np.abs(y), 448.0)
    dist = np.abs(a[:, None] - table[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    even = cand & (codes[None, :] % 2 == 0)
    pick = np.where(cand.sum(1) > 1, even.argmax(1), cand.argmax(1))
    assert np.array_equal(enc & 0x7F, pick.astype(np.uint8))


# ----------------------------------------------------------------------------- helpers
def _tiny_cache(rows_576, kv=oracle.KV_BF16):
    """Contiguous pages holding the given rows (float64 [n, 576], exact in bf16)."""
    n = rows_576.shape[0]
    pages = max(1, (n + 63) // 64)
    buf = np.zeros((pages * 64, 576), np.float32)
    buf[:n] = rows_576
    cache = mi.to_bf16_bits(buf).reshape(pages, 64 * 576)
    bt = np.arange(pages, dtype=np.int32)[None, :]
    return cache.view(np.uint8), bt, pages


def _q_bf16(vec576):
    return mi.to_bf16_bits(np.asarray(vec576, np.float32)).reshape(1, 1, 1, 576)


# ----------------------------------------------------------------------------- hand cases
@pytest.mark.parametrize("case", ["one_token", "two_equal", "gap_100", "three_0_1_2"])
def test_hand_cases(case):
    g = _read_table("hand_cases.txt")[case]
    exp_lse, exp_o1 = float(g[1]), float(g[3])
    dim0 = {"one_token": [3], "two_equal": [2, 2], "gap_100": [100, 0],
            "three_0_1_2": [0, 1, 2]}[case]
    o1_vals = [5, 7, 11]
    rows = np.zeros((len(dim0), 576))
    for j, v in enumerate(dim0):
        rows[j, 0] = v
        rows[j, 1] = o1_vals[j]
    cache, bt, nb = _tiny_cache(rows)
    q = np.zeros(576)
    q[0] = 1.0
    o, lse = oracle.decode_absorbed(_q_bf16(q), cache, oracle.KV_BF16, nb, bt,
                                    np.array([len(dim0)], np.int32), 1, 1, 1, 1.0)
    assert lse[0, 0, 0] == pytest.approx(exp_lse, abs=1e-13, rel=1e-14)
    assert o[0, 0, 0, 1] == pytest.approx(exp_o1, abs=1e-12)
    if case == "one_token":  # o_latent is exactly the cached latent
        assert np.array_equal(o[0, 0, 0], rows[0, :512])


def test_scale_is_a_caller_argument_and_192_not_576():
    """The softmax scale stays 1/sqrt(192) after absorption (vLLM MLA backend article, section
    on the two algorithms). A wrong 1/sqrt(576) flattens logits by sqrt(3) and must move the
    result far outside the parity tolerance."""
    assert mi.SCALE == pytest.approx(1 / math.sqrt(192), rel=1e-7)
    c = mi.decode_case(1, 1, 4, [200], seed=3)
    args = (c["q"], c["cache"], c["kv"], c["num_blocks"], c["block_table"], c["seq_lens"], 1, 1, 4)
    o_ok, lse_ok = oracle.decode_absorbed(*args, mi.SCALE)
    o_bad, lse_bad = oracle.decode_absorbed(*args, 1 / math.sqrt(576))
    assert np.abs(o_ok - o_bad).max() > 0.05
    assert np.abs(lse_ok - lse_bad).max() > 0.1
    # one token: lse is the scaled logit itself
    c1 = mi.decode_case(1, 1, 2, [1], seed=4)
    o1, l1 = oracle.decode_absorbed(c1["q"], c1["cache"], c1["kv"], c1["num_blocks"],
                                    c1["block_table"], c1["seq_lens"], 1, 1, 2, mi.SCALE)
    row = oracle.widen_bf16(c1["cache"].view(np.uint16).reshape(-1, 64, 576)[c1["block_table"][0, 0], 0])
    qd = oracle.widen_bf16(c1["q"]).reshape(2, 576)
    np.testing.assert_allclose(l1.reshape(2), mi.SCALE * (qd @ row), rtol=1e-13)
    np.testing.assert_array_equal(o1.reshape(2, 512), np.stack([row[:512]] * 2))


# ----------------------------------------------------------------------------- library pins
def _gather_rows(c, b):
    """Rows of request b in token order, gathered with numpy from the block table."""
    rb = mi.ROW_BYTES[c["kv"]]
    cache = c["cache"].reshape(c["num_blocks"], 64, rb)
    n = int(c["seq_lens"][b])
    pages = c["block_table"][b, : (n + 63) // 64]
    raw = cache[pages].reshape(-1, rb)[:n]
    if c["kv"] == mi.KV_BF16:
        k = oracle.widen_bf16(raw.view(np.uint16).reshape(n, 576))
        return k, k[:, :512]
    vals = oracle.widen_e4m3(raw[:, :576])
    ks = raw[:, 576:580].copy().view("<f4").astype(np.float64)
    vs = raw[:, 580:584].copy().view("<f4").astype(np.float64)
    return vals * ks, vals[:, :512] * vs


def _sdpa(q, k, v, scale):
    qt, kt, vt = (torch.from_numpy(np.ascontiguousarray(a))[None] for a in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0].numpy()
    lse = torch.logsumexp(scale * (qt @ kt.transpose(-1, -2)), dim=-1)[0].numpy()
    return o, lse


@pytest.mark.parametrize("kv", [mi.KV_BF16, mi.KV_FP8])
def test_nonabsorbed_matches_torch_sdpa(kv):
    """Route N against library attention on K / V built with numpy matmuls from the gathered
    rows (W_UK_T[h] is [128, 512], W_UV[h] is [512, 128])."""
    H, lens = 3, [70, 129]
    c = mi.e2e_case(2, 1, H, lens, kv=kv, seed=11)
    if kv == mi.KV_FP8:  # make v_scale differ from k_scale so a swap cannot pass
        cache = c["cache"].reshape(c["num_blocks"], 64, 584)
        vs = cache[:, :, 580:584].copy().view("<f4") * np.float32(2.0)
        cache[:, :, 580:584] = vs.view(np.uint8).reshape(cache.shape[0], 64, 4)
        c["cache"] = cache.reshape(c["num_blocks"], -1)
    o, ol, lse = oracle.decode_nonabsorbed(c["q_nope"], c["q_pe"], c["cache"], kv, c["num_blocks"],
                                           c["block_table"], c["seq_lens"], c["w_uk_t"], c["w_uv"],
                                           2, 1, H, mi.SCALE)
    wk = oracle.widen_bf16(c["w_uk_t"])
    wv = oracle.widen_bf16(c["w_uv"])
    qn = oracle.widen_bf16(c["q_nope"])
    qp = oracle.widen_bf16(c["q_pe"])
    for b in range(2):
        kfull, vlat = _gather_rows(c, b)
        for h in range(H):
            k = np.concatenate([kfull[:, :512] @ wk[h].T, kfull[:, 512:]], axis=1)  # [n, 192]
            v = vlat @ wv[h]                                                       # [n, 128]
            qv = np.concatenate([qn[b, 0, h], qp[b, 0, h]])[None]
            o_ref, lse_ref = _sdpa(qv, k, v, mi.SCALE)
            ol_ref, _ = _sdpa(qv, k, vlat, mi.SCALE)
            np.testing.assert_allclose(o[b, 0, h], o_ref[0], rtol=1e-10, atol=1e-12)
            np.testing.assert_allclose(ol[b, 0, h], ol_ref[0], rtol=1e-10, atol=1e-12)
            assert lse[b, 0, h] == pytest.approx(float(lse_ref[0]), abs=1e-11)


def test_absorb_and_out_proj_match_numpy():
    a = mi.absorb_case(5, 3, seed=12)
    q = oracle.absorb_q(a["q_nope"], a["q_pe"], a["w_uk_t"], 5, 3)
    qn = oracle.widen_bf16(a["q_nope"])
    wk = oracle.widen_bf16(a["w_uk_t"])
    ref = np.einsum("thp,hpl->thl", qn, wk)
    np.testing.assert_allclose(q[..., :512], ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_array_equal(q[..., 512:], oracle.widen_bf16(a["q_pe"]))
    b = mi.out_proj_case(4, 3, seed=13)
    o = oracle.out_proj(b["o_latent"], b["w_uv"], 4, 3)
    ref = np.einsum("thl,hlv->thv", b["o_latent"].astype(np.float64), oracle.widen_bf16(b["w_uv"]))
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------- identities
@pytest.mark.parametrize("kv", [mi.KV_BF16, mi.KV_FP8])
def test_absorption_identity(kv):
    """Absorbed (route A, fp64 unrounded ql) and non-absorbed (route N) agree to 1e-10:
    q_nope . (c W_UK) = (q_nope W_UK^T) . c, and o = (sum p c) W_UV."""
    B, Sq, H = 2, 2, 4
    c = mi.e2e_case(B, Sq, H, [1, 150], kv=kv, seed=21)
    o, ol, lse = oracle.decode_nonabsorbed(c["q_nope"], c["q_pe"], c["cache"], kv, c["num_blocks"],
                                           c["block_table"], c["seq_lens"], c["w_uk_t"], c["w_uv"],
                                           B, Sq, H, mi.SCALE)
    qa = oracle.absorb_q(c["q_nope"].reshape(B * Sq, H, 128), c["q_pe"].reshape(B * Sq, H, 64),
                         c["w_uk_t"], B * Sq, H)
    ol_a, lse_a = oracle.decode_absorbed(qa.reshape(B, Sq, H, 576), c["cache"], kv, c["num_blocks"],
                                         c["block_table"], c["seq_lens"], B, Sq, H, mi.SCALE)
    o_a = oracle.out_proj(ol_a.reshape(B * Sq, H, 512), c["w_uv"], B * Sq, H).reshape(o.shape)
    fin = np.isfinite(lse)
    assert np.array_equal(fin, np.isfinite(lse_a))
    assert not fin[0, 0].any()  # request 0 has 1 token: row t=0 sees 0 tokens
    assert np.abs(lse[fin] - lse_a[fin]).max() <= 1e-10
    assert np.abs(ol - ol_a).max() <= 1e-10
    assert np.abs(o - o_a).max() <= 1e-10


def test_softmax_weights_sum_to_one():
    """With every visible latent equal to ones, o_latent = sum_j p_j = 1."""
    c = mi.decode_case(3, 1, 8, [1, 64, 333], seed=5)
    cache = c["cache"].view(np.uint16).reshape(c["num_blocks"], 64, 576)
    valid = mi.valid_row_mask(c["seq_lens"], c["block_table"], c["num_blocks"])
    lat = cache[..., :512]
    lat[valid] = 0x3F80  # bf16 1.0
    o, lse = oracle.decode_absorbed(c["q"], c["cache"], c["kv"], c["num_blocks"], c["block_table"],
                                    c["seq_lens"], 3, 1, 8, mi.SCALE)
    assert np.abs(o - 1.0).max() <= 1e-14
    assert np.isfinite(lse).all()


@pytest.mark.parametrize("chunk", [1, 7, 64, 100, 128, 4096])
def test_split_merge_equals_unsplit(chunk):
    c = mi.decode_case(3, 2, 4, [1, 130, 700], seed=6)
    args = (c["q"], c["cache"], c["kv"], c["num_blocks"], c["block_table"], c["seq_lens"], 3, 2, 4,
            mi.SCALE)
    o0, l0 = oracle.decode_absorbed(*args)
    o1, l1 = oracle.decode_absorbed(*args, chunk=chunk)
    assert np.array_equal(np.isfinite(l0), np.isfinite(l1))
    fin = np.isfinite(l0)
    assert np.abs(l0[fin] - l1[fin]).max() <= 1e-12
    assert np.abs(o0 - o1).max() <= 1e-12


def test_merge_special_cases():
    rng = np.random.default_rng(9)
    o = rng.standard_normal((3, 512))
    lse = np.array([0.5, -np.inf, 2.0])
    m, ml = oracle.merge(o, lse)
    m2, ml2 = oracle.merge(o[[0, 2]], lse[[0, 2]])
    np.testing.assert_allclose(m, m2, rtol=0, atol=1e-15)  # an empty partial has no weight
    assert ml == pytest.approx(ml2, abs=1e-15)
    assert ml == pytest.approx(math.log(math.exp(0.5) + math.exp(2.0)), abs=1e-14)
    w = np.exp([0.5, 2.0]) / (math.exp(0.5) + math.exp(2.0))
    np.testing.assert_allclose(m, w[0] * o[0] + w[1] * o[2], atol=1e-14)
    z, zl = oracle.merge(o, np.full(3, -np.inf))
    assert zl == -math.inf and np.all(z == 0)


def test_causal_rows_match_shorter_single_row():
    """Sq=2: row t=0 sees seq_len-1 tokens, i.e. equals an Sq=1 decode with seq_len-1."""
    c = mi.decode_case(2, 2, 4, [65, 300], seed=10)
    o2, l2 = oracle.decode_absorbed(c["q"], c["cache"], c["kv"], c["num_blocks"], c["block_table"],
                                    c["seq_lens"], 2, 2, 4, mi.SCALE)
    q0 = np.ascontiguousarray(c["q"][:, :1])
    o1, l1 = oracle.decode_absorbed(q0, c["cache"], c["kv"], c["num_blocks"], c["block_table"],
                                    c["seq_lens"] - 1, 2, 1, 4, mi.SCALE)
    np.testing.assert_array_equal(o2[:, 0], o1[:, 0])
    np.testing.assert_array_equal(l2[:, 0], l1[:, 0])
    assert oracle.row_len(10, 2, 0) == 9 and oracle.row_len(10, 2, 1) == 10
    assert oracle.row_len(0, 2, 0) == 0 and oracle.row_len(1, 3, 0) == 0


def test_zero_length_rows_and_bad_block_ids():
    c = mi.decode_case(2, 1, 2, [0, 5], seed=14)
    o, lse = oracle.decode_absorbed(c["q"], c["cache"], c["kv"], c["num_blocks"], c["block_table"],
                                    c["seq_lens"], 2, 1, 2, mi.SCALE)
    assert np.all(lse[0] == -np.inf) and np.all(o[0] == 0)
    bt = c["block_table"].copy()
    bt[1, 0] = c["num_blocks"]  # out of range
    with pytest.raises(ValueError):
        oracle.decode_absorbed(c["q"], c["cache"], c["kv"], c["num_blocks"], bt, c["seq_lens"], 2, 1,
                               2, mi.SCALE)


def test_default_num_splits_rule():
    """min(next_pow2(max(1, max_seq_len // 512)), 2 * sm_count), from the Triton MLA section."""
    cases = {(131072, 152): 256, (4096, 152): 8, (8192, 152): 16, (32768, 152): 64,
             (100, 152): 1, (1536, 152): 4, (10 ** 6, 152): 304, (131072, 100): 200}
    for (n, sms), s in cases.items():
        assert oracle.default_num_splits(n, sms) == s


def test_poisoned_rows_are_never_read():
    """The seeded cache poisons every unreadable row with NaN; the oracle must stay finite."""
    c = mi.decode_case(4, 2, 4, [1, 63, 64, 65], seed=15)
    o, lse = oracle.decode_absorbed(c["q"], c["cache"], c["kv"], c["num_blocks"], c["block_table"],
                                    c["seq_lens"], 4, 2, 4, mi.SCALE)
    assert np.isfinite(o).all()
    assert np.isfinite(lse[np.array([oracle.row_len(n, 2, t) > 0 for n in c["seq_lens"]
                                     for t in range(2)]).reshape(4, 2)]).all()


# ----------------------------------------------------------------------------- cache write (FP8 quantise)
def test_e4m3_decoder_known_codes():
    """OCP E4M3 values fixed by the format: bias 7, 3 mantissa bits, S.1111.111 = NaN."""
    assert oracle.widen_e4m3([0x38])[0] == 1.0
    assert oracle.widen_e4m3([0x7E])[0] == 448.0 and oracle.widen_e4m3([0xFE])[0] == -448.0
    assert oracle.widen_e4m3([0x08])[0] == 2.0 ** -6      # smallest normal
    assert oracle.widen_e4m3([0x01])[0] == 2.0 ** -9      # smallest subnormal
    assert oracle.widen_e4m3([0x07])[0] == 7 * 2.0 ** -9  # largest subnormal
    assert oracle.widen_e4m3([0x39])[0] == 1.125
    assert np.isnan(oracle.widen_e4m3([0x7F])[0]) and np.isnan(oracle.widen_e4m3([0xFF])[0])


def test_e4m3_encoder_round_trip_ties_and_saturation():
    vals = oracle.widen_e4m3(np.arange(256, dtype=np.uint8))
    for c in list(range(0, 0x7F)) + list(range(0x80, 0xFF)):   # every finite code, both signs
        assert oracle.e4m3_encode(np.float32(vals[c])) == c, hex(c)
    for c in range(0, 0x7E):  # midpoints between neighbours round to the even code
        lo, hi = vals[c], vals[c + 1]
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2                      # exact in binary32
        assert oracle.e4m3_encode(mid) == (c if c % 2 == 0 else c + 1), hex(c)
        assert oracle.e4m3_encode(np.nextafter(mid, np.float32(0))) == c
        assert oracle.e4m3_encode(np.nextafter(mid, np.float32(1e9))) == c + 1
        assert oracle.e4m3_encode(-mid) == 0x80 | (c if c % 2 == 0 else c + 1)
    for big in (449.0, 464.0, 1000.0, 3e38):
        assert oracle.e4m3_encode(big) == 0x7E and oracle.e4m3_encode(-big) == 0xFE
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00     # tie between 0 and the smallest subnormal
    assert oracle.e4m3_encode(0.75 * 2.0 ** -9) == 0x01


def _cache_write_case(T, seed, spare=3):
    rng = np.random.default_rng(seed)
    kv_c = mi.to_bf16_bits(rng.standard_normal((T, 512)).astype(np.float32) * 2.0)
    k_pe = mi.to_bf16_bits(rng.standard_normal((T, 64)).astype(np.float32))
    nb = (T + 63) // 64 + spare
    slots = rng.permutation(nb * 64)[:T].astype(np.int64)
    return kv_c, k_pe, slots, nb


def test_cache_write_bf16_rows_land_at_their_slots():
    T = 70
    kv_c, k_pe, slots, nb = _cache_write_case(T, 70)
    slots[5] = -1                       # padding token
    slots[9] = nb * 64 + 3              # beyond the cache: counted, skipped
    cache = np.full((nb, 64 * 1152), 0xAB, np.uint8)
    assert oracle.cache_write(kv_c, k_pe, slots, oracle.KV_BF16, cache, nb) == 1
    rows = cache.reshape(nb * 64, 1152)
    for t in range(T):
        if t in (5, 9):
            continue
        expect = np.concatenate([kv_c[t], k_pe[t]]).view(np.uint8)
        np.testing.assert_array_equal(rows[slots[t]], expect)
    written = set(int(s) for i, s in enumerate(slots) if i not in (5, 9))
    untouched = [r for r in range(nb * 64) if r not in written]
    assert np.all(rows[untouched] == 0xAB)


@pytest.mark.parametrize("kv_scale", [0.0, 0.05, 1.0])
def test_cache_write_fp8_quantises_per_definition(kv_scale):
    T = 40
    kv_c, k_pe, slots, nb = _cache_write_case(T, 71)
    kv_c[3] = 0                                   # an all-zero latent ...
    k_pe[3] = 0                                   # ... and rope: amax 0 -> scale 1
    cache = np.zeros((nb, 64 * 584), np.uint8)
    assert oracle.cache_write(kv_c, k_pe, slots, oracle.KV_FP8, cache, nb, kv_scale=kv_scale) == 0
    rows = cache.reshape(nb * 64, 584)
    for t in range(T):
        r = rows[slots[t]]
        x = oracle.widen_bf16(np.concatenate([kv_c[t], k_pe[t]]))
        ks = r[576:580].copy().view(np.float32)[0]
        vs = r[580:584].copy().view(np.float32)[0]
        assert ks == vs
        if kv_scale > 0:
            assert ks == np.float32(kv_scale)
        elif t == 3:
            assert ks == 1.0 and np.all(r[:576] == 0)
            continue
        else:
            amax = np.float32(np.max(np.abs(x)))
            assert ks == np.float32(amax / np.float32(448.0))
            assert np.any((r[:576] & 0x7F) == 0x7E)          # the largest element maps to +-448
        deq = oracle.widen_e4m3(r[:576]) * float(ks)
        q = (x.astype(np.float32) * (np.float32(1.0) / ks)).astype(np.float64)  # x * (1 / scale), binary32
        inside = np.abs(q) <= 448
        # within half an e4m3 step of the exact quotient: 2^-4 relative for normals, 2^-10
        # absolute in the subnormal range; saturated values sit at +-448
        err = np.abs(deq[inside] / float(ks) - q[inside])
        assert np.all(err <= np.maximum(np.abs(q[inside]) * 2.0 ** -4, 2.0 ** -10) + 1e-12)
        assert np.all(np.abs(deq[~inside] / float(ks)) == 448.0)


def _torch_e4m3(v):
    """float8_e4m3fn codes of binary32 values, saturated to +-448 first (torch maps overflow to NaN)."""
    v = np.clip(np.asarray(v, np.float32), np.float32(-448.0), np.float32(448.0))
    return torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _reciprocal_vs_quotient_values(s):
    """Every positive finite bf16 value x whose e4m3 code differs between the binary32 product
    x * (1 / s) and the binary32 quotient x / s (both within +-448)."""
    x = (np.arange(1, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    with np.errstate(over="ignore"):
        mul = x * (np.float32(1.0) / s)
        div = x / s
    keep = (np.abs(mul) <= 448) & (np.abs(div) <= 448)
    x, mul, div = x[keep], mul[keep], div[keep]
    return x[_torch_e4m3(mul) != _torch_e4m3(div)]


@pytest.mark.parametrize("per_token", [False, True])
def test_cache_write_fp8_multiplies_by_the_reciprocal_scale(per_token):
    """The quantising write stores e4m3(x * (1 / s)), both steps rounded in binary32: the page's
    cache-write section describes the FP8 write as a multiplication by the scale factor (skipped
    when the scale is exactly 1), and with the stored scale s defined by dequant = code * s that
    factor is 1 / s. The expected bytes come from torch's float8_e4m3fn conversion of a numpy
    binary32 product, and the inputs are values for which dividing by s instead gives another
    code, so a writer that divides fails here."""
    s = np.float32(7.0)  # 1/7 is inexact in binary32
    vals = _reciprocal_vs_quotient_values(s)
    assert len(vals) >= 16
    row = np.zeros(576, np.float32)
    row[: len(vals)] = vals[:575]
    row[288: 288 + len(vals)] = -vals[:288]         # the negative side too
    kv_scale = 0.0
    if per_token:
        row[575] = 3136.0                           # amax: 3136 / 448 = 7 exactly
        assert np.float32(np.float32(3136.0) / np.float32(448.0)) == s
    else:
        kv_scale = float(s)
    bits = mi.to_bf16_bits(row)
    assert np.array_equal(oracle.widen_bf16(bits), row.astype(np.float64))  # the values are bf16
    cache = np.zeros((1, 64 * 584), np.uint8)
    slots = np.array([5], np.int64)
    assert oracle.cache_write(bits[None, :512], bits[None, 512:], slots, oracle.KV_FP8, cache, 1,
                              kv_scale=kv_scale) == 0
    r = cache.reshape(64, 584)[5]
    assert r[576:580].copy().view(np.float32)[0] == s and r[580:584].copy().view(np.float32)[0] == s
    expect = _torch_e4m3(row * (np.float32(1.0) / s))
    np.testing.assert_array_equal(r[:576], expect)
    # the same inputs divided by s give other codes: the pin tells the two readings apart
    assert np.count_nonzero(_torch_e4m3(row / s) != expect) >= 16


# ----------------------------------------------------------------------------- variable-length query rows
def test_varlen_equals_uniform_and_per_request_runs():
    """Packed rows with equal query lengths are the uniform batch; a request's rows in a mixed
    batch are that request decoded alone with Sq = its query length."""
    H = 4
    c = mi.decode_case(3, 2, H, [5, 130, 70], seed=90)
    qsl = np.array([0, 2, 4, 6], np.int32)
    o_u, lse_u = oracle.decode_absorbed(c["q"], c["cache"], c["kv"], c["num_blocks"], c["block_table"],
                                        c["seq_lens"], 3, 2, H, c["scale"])
    o_v, lse_v = oracle.decode_varlen(c["q"].reshape(6, H, 576), c["cache"], c["kv"], c["num_blocks"],
                                      c["block_table"], c["seq_lens"], qsl, H, c["scale"])
    np.testing.assert_array_equal(o_v, o_u.reshape(6, H, 512))
    np.testing.assert_array_equal(lse_v, lse_u.reshape(6, H))
    # mixed query lengths 1, 3, 0, 2 (a request may have no query rows)
    lens = [40, 200, 9, 64]
    qlens = [1, 3, 0, 2]
    d = mi.decode_case(4, 1, H, lens, seed=91)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    rng = np.random.default_rng(92)
    q = mi.to_bf16_bits(rng.standard_normal((int(qsl[-1]), H, 576)).astype(np.float32))
    o_v, lse_v = oracle.decode_varlen(q, d["cache"], d["kv"], d["num_blocks"], d["block_table"], lens, qsl, H,
                                      d["scale"])
    for b in range(4):
        if qlens[b] == 0:
            continue
        qb = q[qsl[b]:qsl[b + 1]].reshape(1, qlens[b], H, 576)
        o_b, lse_b = oracle.decode_absorbed(qb, d["cache"], d["kv"], d["num_blocks"], d["block_table"][b:b + 1],
                                            [lens[b]], 1, qlens[b], H, d["scale"])
        np.testing.assert_array_equal(o_v[qsl[b]:qsl[b + 1]], o_b[0])
        np.testing.assert_array_equal(lse_v[qsl[b]:qsl[b + 1]], lse_b[0])
    # causal: the last row of request 1 sees all 200 tokens, its first row 198
    assert np.isfinite(lse_v).all()
