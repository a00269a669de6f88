"""GPU parity of mla_prefill (compute-friendly route: gather, up-projection GEMMs, tcgen05
attention with the LSE merge of context chunks) against the fp64 oracle on the same seeded inputs.

Tolerances. The kernels store the up-projected k_nope and v as bf16 (the model dtype of the
projection in the pages' prefill) and round P to bf16 for the PV product. One bf16 rounding of v
moves an output by at most 2^-8 of its size, so o is held to |o - o_ref| <= 1e-2 + 2^-8 |o_ref|
elementwise plus rel L2 <= 5e-3. The rounding of k_nope moves one logit by about
scale * sqrt(128) * 2^-8 / sqrt(3) = 1.9e-3 (one standard deviation, q and k of unit size); a row
that sees a single key carries that error into its lse whole, so lse is held to 1e-2 (five
standard deviations)."""
import numpy as np
import pytest

import mla_inputs as mi
import oracle

pytestmark = pytest.mark.gpu


def _dev(c):
    import torch
    d16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)  # noqa
    return dict(
        q=d16(c["q"]), kv_c=d16(c["kv_c_new"]), k_pe=d16(c["k_pe_new"]),
        cache=torch.from_numpy(np.ascontiguousarray(c["cache"])).cuda(),
        bt=torch.from_numpy(c["block_table"]).cuda(),
        ctx=torch.from_numpy(c["ctx_lens"]).cuda(), qsl=torch.from_numpy(c["query_start_loc"]).cuda(),
        wk=d16(c["w_uk_t"]), wv=d16(c["w_uv"]))


def run_prefill(c, chunk_rows, **kw):
    import torch
    import mla_latent_kv_gb300 as mla
    d = _dev(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = mla.prefill(d["q"], d["kv_c"], d["k_pe"], d["cache"], d["bt"], d["ctx"], d["qsl"], d["wk"], d["wv"],
                         c["scale"], kv_dtype=c["kv"], chunk_rows=chunk_rows, dev_status=status,
                         num_blocks=c["num_blocks"], **kw)
    torch.cuda.synchronize()
    return o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), int(status.item())


def ref_prefill(c, chunk_rows):
    return oracle.prefill(c["q"], c["kv_c_new"], c["k_pe_new"], c["cache"], c["kv"], c["num_blocks"],
                          c["block_table"], c["ctx_lens"], c["query_start_loc"], c["H"], c["w_uk_t"], c["w_uv"],
                          c["scale"], chunk_rows)


def compare(o, lse, o_ref, lse_ref, fp8=False):
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    err = np.abs(o - o_ref)
    bound = 1e-2 + 2.0 ** -8 * np.abs(o_ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), f"max excess at {worst}: got {o[worst]}, want {o_ref[worst]}"
    rel = np.linalg.norm(o - o_ref) / max(np.linalg.norm(o_ref), 1e-30)
    assert rel <= (2e-2 if fp8 else 5e-3), rel
    assert np.abs(lse - lse_ref).max() <= 1e-2, np.abs(lse - lse_ref).max()


@pytest.mark.parametrize("chunk_rows", [64, 192, 1 << 20])
def test_prefill_small_ragged(chunk_rows):
    # contexts of 0, 70, 130 and 64 tokens (partial pages), 5 / 1 / 67 / 3 new tokens
    c = mi.prefill_case([0, 70, 130, 64], [5, 1, 67, 3], H=4, seed=21)
    o, lse, st = run_prefill(c, chunk_rows)
    assert st == 0
    compare(o, lse, *ref_prefill(c, chunk_rows))


def test_prefill_fp8_context_distinct_scales():
    c = mi.prefill_case([90, 0, 200, 333], [4, 6, 2, 9], H=3, kv=mi.KV_FP8, seed=22)
    rows = c["cache"].reshape(c["num_blocks"], 64, 584)
    vs = rows[:, :, 580:584].copy().view("<f4") * np.float32(2.0)  # v_scale = 2 k_scale
    rows[:, :, 580:584] = vs.view(np.uint8)
    o, lse, st = run_prefill(c, 128)
    assert st == 0
    compare(o, lse, *ref_prefill(c, 128), fp8=True)


def test_prefill_multiple_query_tiles_and_chunks():
    # new tokens spanning two and three 128-row query tiles (causal across tiles), contexts
    # cut into several chunks, one request without context
    c = mi.prefill_case([300, 0, 1000], [200, 130, 257], H=8, seed=23)
    o, lse, st = run_prefill(c, 256)
    assert st == 0
    compare(o, lse, *ref_prefill(c, 256))


def test_prefill_dsv3_heads():
    # H = 128 (every head's K/V slice in the up-projected workspace), one long context chunked
    c = mi.prefill_case([640, 64], [160, 40], H=128, seed=24)
    o, lse, st = run_prefill(c, 512)
    assert st == 0
    compare(o, lse, *ref_prefill(c, 512))


def test_prefill_request_without_new_tokens_and_lse_optional():
    import torch
    import mla_latent_kv_gb300 as mla
    c = mi.prefill_case([100, 64, 5], [3, 0, 2], H=2, seed=25)
    o_ref, lse_ref = ref_prefill(c, 64)
    d = _dev(c)
    o = mla.prefill(d["q"], d["kv_c"], d["k_pe"], d["cache"], d["bt"], d["ctx"], d["qsl"], d["wk"], d["wv"],
                    c["scale"], chunk_rows=64, num_blocks=c["num_blocks"])[0]
    # a call with lse=None still merges through the workspace's own lse buffer
    o2 = torch.empty_like(o)
    ws = torch.empty(mla.prefill_workspace_bytes(3, 5, 2, 64), dtype=torch.uint8, device="cuda")
    import ctypes
    ctx_h = torch.tensor(c["ctx_lens"], dtype=torch.int32)
    qsl_h = torch.tensor(c["query_start_loc"], dtype=torch.int32)
    mla._check(mla.lib().mla_prefill(
        mla._p(d["q"]), mla._p(d["kv_c"]), 512, mla._p(d["k_pe"]), 64, mla._p(d["cache"]), 0, c["num_blocks"],
        mla._p(d["bt"]), c["block_table"].shape[1], mla._p(d["ctx"]), mla._p(d["qsl"]),
        ctypes.c_void_p(ctx_h.data_ptr()), ctypes.c_void_p(qsl_h.data_ptr()), 3, 2, mla._p(d["wk"]), mla._p(d["wv"]),
        c["scale"], 64, mla._p(ws), ws.numel(), mla._p(o2), None, None, mla._stream(None)))
    torch.cuda.synchronize()
    compare(o.cpu().numpy().astype(np.float64), lse_ref, o_ref, lse_ref)
    np.testing.assert_array_equal(o.cpu().numpy(), o2.cpu().numpy())


def test_prefill_bad_block_id_is_reported():
    c = mi.prefill_case([130, 10], [2, 2], H=2, seed=26)
    c["block_table"][0, 1] = c["num_blocks"] + 7
    o, lse, st = run_prefill(c, 64)
    assert st & 0x1


def test_prefill_single_head():
    c = mi.prefill_case([200, 3], [70, 2], H=1, seed=27)
    o, lse, st = run_prefill(c, 128)
    assert st == 0
    compare(o, lse, *ref_prefill(c, 128))


def test_prefill_fp8_many_chunks_and_query_tiles():
    c = mi.prefill_case([700, 130, 0], [150, 5, 129], H=4, kv=mi.KV_FP8, seed=28)
    rows = c["cache"].reshape(c["num_blocks"], 64, 584)
    vs = rows[:, :, 580:584].copy().view("<f4") * np.float32(0.5)  # v_scale = k_scale / 2
    rows[:, :, 580:584] = vs.view(np.uint8)
    o, lse, st = run_prefill(c, 192)
    assert st == 0
    compare(o, lse, *ref_prefill(c, 192), fp8=True)


def test_prefill_causal_only_three_query_tiles():
    c = mi.prefill_case([0], [300], H=2, seed=29)
    o, lse, st = run_prefill(c, 64)
    assert st == 0
    compare(o, lse, *ref_prefill(c, 64))


def test_prefill_many_requests_packed_chunks():
    rng = np.random.default_rng(30)
    ctx = rng.integers(0, 400, size=20)
    ctx[[2, 7]] = 0
    ql = rng.integers(0, 40, size=20)
    ql[[0, 5]] = [1, 130]
    c = mi.prefill_case(list(ctx), list(ql), H=3, seed=30)
    o, lse, st = run_prefill(c, 200)  # chunks hold several requests' rows
    assert st == 0
    compare(o, lse, *ref_prefill(c, 200))


@pytest.mark.parametrize("chunk_rows", [64, 4096])
def test_prefill_chunk_sizes_meet_the_same_bound(chunk_rows):
    # a different chunking moves keys between tiles (other rounding of P); both meet the bound
    c = mi.prefill_case([900, 450], [40, 100], H=2, seed=31)
    o, lse, st = run_prefill(c, chunk_rows)
    assert st == 0
    compare(o, lse, *ref_prefill(c, chunk_rows))


def test_prefill_fp8_one_pass():
    # the whole context fits the row budget: context rows (e4m3 widened, per-row scales) and the
    # new tokens' rows (scale 1) share one workspace and one attention pass
    c = mi.prefill_case([90, 0, 200, 333], [4, 6, 150, 9], H=3, kv=mi.KV_FP8, seed=32)
    rows = c["cache"].reshape(c["num_blocks"], 64, 584)
    vs = rows[:, :, 580:584].copy().view("<f4") * np.float32(2.0)  # v_scale = 2 k_scale
    rows[:, :, 580:584] = vs.view(np.uint8)
    o, lse, st = run_prefill(c, 4096)
    assert st == 0
    compare(o, lse, *ref_prefill(c, 4096), fp8=True)
