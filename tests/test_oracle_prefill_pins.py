"""Pins of the oracle's prefill route (compute-friendly form: up-project, MHA, chunked context,
LSE merge) against facts that do not come from the route itself: the absorption identity (the
absorbed decode route over the same tokens gives the same attention), torch SDPA on keys and
values built with numpy matmuls, a hand-worked chunk plan, closed forms of a one-token request,
and invariance under the context chunk size. No GPU."""
import numpy as np
import pytest
import torch

import mla_inputs as mi
import oracle


def _decode_route(c, kv_write_scale=0.0):
    """The same attention through the absorbed route: write the new tokens into the cache, absorb
    q_nope through W_UK_T, run decode over ctx + q_len tokens with causal rows, up-project."""
    H = c["H"]
    T = int(c["query_start_loc"][-1])
    cache = c["cache"].copy()
    assert oracle.cache_write(c["kv_c_new"], c["k_pe_new"], c["new_slots"], c["kv"], cache, c["num_blocks"],
                              kv_scale=kv_write_scale) == 0
    q = c["q"].reshape(T, H, 192)
    qa = oracle.absorb_q(np.ascontiguousarray(q[..., :128]), np.ascontiguousarray(q[..., 128:]), c["w_uk_t"], T, H)
    seq = (c["ctx_lens"].astype(np.int64) + np.diff(c["query_start_loc"])).astype(np.int32)
    ol, lse = oracle.decode_varlen(qa, cache, c["kv"], c["num_blocks"], c["block_table"], seq,
                                   c["query_start_loc"], H, c["scale"])
    return oracle.out_proj(ol, c["w_uv"], T, H), lse


def _prefill(c, chunk_rows):
    return oracle.prefill(c["q"], c["kv_c_new"], c["k_pe_new"], c["cache"], c["kv"], c["num_blocks"],
                          c["block_table"], c["ctx_lens"], c["query_start_loc"], c["H"], c["w_uk_t"], c["w_uv"],
                          c["scale"], chunk_rows)


def test_chunk_plan_hand_example():
    # budget 128 rows; contexts 100, 0, 300, 64 (worked by hand from the rule: a request goes in
    # whole if it fits, else whole pages that fit, else the chunk is closed)
    got = oracle.prefill_chunks([100, 0, 300, 64], 128)
    want = [(0, 0, 0, 100), (1, 2, 0, 128), (2, 2, 128, 128), (3, 2, 256, 44), (3, 3, 0, 64)]
    assert [tuple(int(v) for v in r) for r in got] == want
    with pytest.raises(ValueError):
        oracle.prefill_chunks([10], 63)


@pytest.mark.parametrize("budget", [64, 100, 192, 4096])
def test_chunk_plan_invariants(budget):
    rng = np.random.default_rng(budget)
    ctx = rng.integers(0, 700, size=23).astype(np.int32)
    ctx[3] = 0
    ctx[5] = 64
    plan = oracle.prefill_chunks(ctx, budget)
    rows = {}
    for ch, b, pos, n in plan:
        assert n > 0 and pos % 64 == 0
        rows[ch] = rows.get(ch, 0) + n
        assert rows[ch] <= budget
    assert list(plan[:, 0]) == sorted(plan[:, 0])         # chunks in order
    for b in range(len(ctx)):
        mine = plan[plan[:, 1] == b]
        assert int(mine[:, 3].sum()) == int(ctx[b])       # every context row exactly once
        assert list(mine[:, 2]) == list(np.cumsum(np.concatenate([[0], mine[:-1, 3]])))[:len(mine)]


def test_prefill_equals_absorbed_decode_route():
    """Absorption identity: attention over up-projected K/V equals the absorbed MQA over the
    latent rows followed by the V up-projection, token for token (fp64, 1e-10)."""
    c = mi.prefill_case([0, 70, 130, 64], [5, 1, 67, 3], H=4, seed=11)
    o, lse = _prefill(c, 64)
    o_ref, lse_ref = _decode_route(c)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-10)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-10)


def test_prefill_fp8_context_equals_absorbed_decode_route():
    """FP8 context: the K side dequantised with k_scale and the V side with v_scale (set apart here
    so a swap shows). The new tokens are written with a power-of-two static scale, so that their
    cached FP8 rows hold exactly the bf16 values the prefill route reads from its own inputs."""
    c = mi.prefill_case([90, 0, 200], [4, 6, 2], H=3, kv=mi.KV_FP8, seed=12)
    rows = c["cache"].reshape(c["num_blocks"], 64, 584)
    vs = rows[:, :, 580:584].copy().view("<f4") * np.float32(2.0)
    rows[:, :, 580:584] = vs.view(np.uint8)
    # new tokens: e4m3 codes times 2^-6, exact in bf16
    T = int(c["query_start_loc"][-1])
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 0x7F, size=(T, 576)).astype(np.uint8) | (rng.integers(0, 2, size=(T, 576)) << 7).astype(np.uint8)
    codes[codes & 0x7F == 0x7F] = 0
    vals = oracle.widen_e4m3(codes) * 2.0 ** -6
    bits = mi.to_bf16_bits(vals.astype(np.float32))
    assert np.array_equal(oracle.widen_bf16(bits), vals)
    c["kv_c_new"], c["k_pe_new"] = np.ascontiguousarray(bits[:, :512]), np.ascontiguousarray(bits[:, 512:])
    o, lse = _prefill(c, 128)
    o_ref, lse_ref = _decode_route(c, kv_write_scale=2.0 ** -6)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-10)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-10)


@pytest.mark.parametrize("kv", [mi.KV_BF16, mi.KV_FP8])
def test_prefill_chunk_size_invariance(kv):
    c = mi.prefill_case([260, 5, 129], [3, 7, 2], H=2, kv=kv, seed=13)
    o0, l0 = _prefill(c, 10 ** 6)
    for budget in (64, 128, 200, 320):
        o, lse = _prefill(c, budget)
        np.testing.assert_allclose(o, o0, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, l0, rtol=0, atol=1e-12)


def test_prefill_without_context_matches_torch_sdpa():
    """No context: causal MHA among the new tokens. K and V are built here with numpy matmuls
    and the attention is torch's SDPA in fp64 (an independent library routine)."""
    c = mi.prefill_case([0, 0], [9, 4], H=3, seed=14)
    o, lse = _prefill(c, 64)
    H = 3
    q = oracle.widen_bf16(c["q"]).reshape(-1, H, 192)
    kvc = oracle.widen_bf16(c["kv_c_new"]).reshape(-1, 512)
    kpe = oracle.widen_bf16(c["k_pe_new"]).reshape(-1, 64)
    wk = oracle.widen_bf16(c["w_uk_t"]).reshape(H, 128, 512)
    wv = oracle.widen_bf16(c["w_uv"]).reshape(H, 512, 128)
    qsl = c["query_start_loc"]
    for b in range(2):
        s0, s1 = int(qsl[b]), int(qsl[b + 1])
        for h in range(H):
            k = np.concatenate([kvc[s0:s1] @ wk[h].T, kpe[s0:s1]], axis=1)
            v = kvc[s0:s1] @ wv[h]
            qt = torch.from_numpy(q[s0:s1, h])[None, None]
            ref = torch.nn.functional.scaled_dot_product_attention(
                qt, torch.from_numpy(k)[None, None], torch.from_numpy(v)[None, None], is_causal=True,
                scale=c["scale"])[0, 0].numpy()
            np.testing.assert_allclose(o[s0:s1, h], ref, rtol=0, atol=1e-12)
            logits = c["scale"] * (q[s0:s1, h] @ k.T)
            logits[np.triu_indices(s1 - s0, 1)] = -np.inf
            lref = torch.logsumexp(torch.from_numpy(logits), dim=1).numpy()
            np.testing.assert_allclose(lse[s0:s1, h], lref, rtol=0, atol=1e-12)


def test_prefill_one_new_token_no_context_closed_form():
    """One new token, no context: the only visible key is itself, so o = kv_c . W_UV[h] and
    lse = scale * <q, [kv_c . W_UK_T[h]^T || k_pe]>."""
    c = mi.prefill_case([0], [1], H=2, seed=15)
    o, lse = _prefill(c, 64)
    kvc = oracle.widen_bf16(c["kv_c_new"])[0]
    kpe = oracle.widen_bf16(c["k_pe_new"])[0]
    q = oracle.widen_bf16(c["q"]).reshape(1, 2, 192)[0]
    wk = oracle.widen_bf16(c["w_uk_t"]).reshape(2, 128, 512)
    wv = oracle.widen_bf16(c["w_uv"]).reshape(2, 512, 128)
    for h in range(2):
        np.testing.assert_allclose(o[0, h], kvc @ wv[h], rtol=0, atol=1e-13)
        k = np.concatenate([wk[h] @ kvc, kpe])
        assert abs(lse[0, h] - c["scale"] * float(q[h] @ k)) < 1e-13


def test_prefill_poisoned_rows_are_never_read():
    # prefill_case poisons every row but the contexts (including the new tokens' own cache rows)
    c = mi.prefill_case([64, 1, 65], [2, 3, 1], H=2, seed=16)
    o, lse = _prefill(c, 64)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
