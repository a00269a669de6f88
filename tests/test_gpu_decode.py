"""GPU parity of mla_decode (and its split-KV merge) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from parity_util import TOL_MAX_ABS, TOL_REL_L2, compare_decode, rel_l2, run_decode, torch_dev

pytestmark = pytest.mark.gpu


def _oracle(c, sel=None):
    return oracle.decode_absorbed(c["q"], c["cache"], c["kv"], c["num_blocks"], c["block_table"],
                                  c["seq_lens"], c["B"], c["Sq"], c["H"], c["scale"], sel=sel)


@pytest.mark.parametrize("num_splits", [1, 2, 3, 0, -1, -2])
def test_tiny_workload(num_splits):
    c = mi.workload_case("tiny")
    o, lse, st = run_decode(c, num_splits)
    o_ref, lse_ref = _oracle(c)
    assert st == 0
    compare_decode(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("num_splits", [1, 4, 7, 0, -2])
def test_ragged_multi_page(num_splits):
    """Several pages, ragged tails (1, 63, 64, 65 tokens...), poisoned unused rows."""
    c = mi.decode_case(6, 1, 128, [1, 63, 64, 65, 700, 1000], seed=20)
    o, lse, st = run_decode(c, num_splits)
    o_ref, lse_ref = _oracle(c)
    assert st == 0
    compare_decode(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("H", [1, 20, 100])
def test_head_counts(H):
    c = mi.decode_case(2, 1, H, [130, 7], seed=21)
    o, lse, st = run_decode(c, 2)
    o_ref, lse_ref = _oracle(c)
    assert st == 0
    compare_decode(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("num_splits", [1, 3, -2])
def test_causal_two_row_queries_and_empty_rows(num_splits):
    """Sq = 2: row t sees seq_len - (1 - t) tokens; seq_len 0 and 1 give empty rows."""
    c = mi.decode_case(4, 2, 32, [0, 1, 2, 200], seed=22)
    o, lse, st = run_decode(c, num_splits)
    o_ref, lse_ref = _oracle(c)
    assert st == 0
    assert np.all(lse_ref[0] == -np.inf) and lse_ref[1, 0, 0] == -np.inf
    compare_decode(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("num_splits", [1, 2])  # 1: every row writes bf16 directly from the epilogue
def test_bf16_output(num_splits):
    c = mi.decode_case(3, 1, 64, [5, 64, 300], seed=23)
    o, lse, st = run_decode(c, num_splits, o_dtype=1)
    o_ref, lse_ref = _oracle(c)
    # one bf16 rounding of the output adds up to half an ulp of |o|
    compare_decode(o, lse, o_ref, lse_ref, extra_abs=float(np.abs(o_ref).max()) * 2.0 ** -9)


def test_bad_block_id_sets_device_status():
    c = mi.decode_case(2, 1, 16, [100, 100], seed=24)
    bt = c["block_table"].copy()
    bt[1, 1] = c["num_blocks"] + 5  # needed entry out of range
    c2 = dict(c, block_table=bt)
    _, _, st = run_decode(c2, 1)
    assert st & 0x1
    _, _, st_ok = run_decode(c, 1)
    assert st_ok == 0


def test_batch_zero_and_workspace_checks():
    import torch
    import mla_latent_kv_gb300 as mla
    c = mi.decode_case(2, 1, 16, [100, 300], seed=25)
    d = torch_dev(c)
    q0 = d["q"][:0]
    o, lse = mla.decode(q0, d["cache"], d["block_table"][:0], d["seq_lens"][:0], 0, c["scale"], num_splits=1)
    assert o.shape[0] == 0
    with pytest.raises(mla.MlaError) as e:
        mla.decode(d["q"], d["cache"], d["block_table"], d["seq_lens"], 300, c["scale"], num_splits=4,
                   workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))
    assert e.value.status == mla.ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("kv", [mi.KV_BF16, mi.KV_FP8])
@pytest.mark.parametrize("num_splits", [-2, 3, 8])
def test_many_short_units_stay_finite(kv, num_splits):
    """Stress of the P hand-off between the two CTAs: 130 rows of 1..130 tokens (many units of
    one or two pages, and empty splits), five calls in a row on one device buffer set. Every
    call must match the oracle, with finite outputs everywhere and a clean device status."""
    import torch
    c = mi.decode_case(130, 1, 32, list(range(1, 131)), kv=kv, seed=70 + num_splits)
    d = torch_dev(c)
    o_ref, lse_ref = _oracle(c)
    for _ in range(5):
        o, lse, st = run_decode(c, num_splits, dev=d)
        assert st == 0
        assert np.isfinite(o).all() and np.isfinite(lse).all()
        compare_decode(o, lse, o_ref, lse_ref, fp8=kv == mi.KV_FP8)
    torch.cuda.synchronize()


# ----------------------------------------------------------------------------- FP8 cache
def _fp8_case(B, Sq, H, lens, seed, vscale=2.0):
    """FP8 cache with v_scale = vscale * k_scale, so that swapping the two scales cannot pass."""
    c = mi.decode_case(B, Sq, H, lens, kv=mi.KV_FP8, seed=seed)
    cache = c["cache"].reshape(c["num_blocks"], 64, 584)
    ks = cache[:, :, 576:580].copy().view("<f4")
    vs = (ks * np.float32(vscale)).astype("<f4")
    with np.errstate(invalid="ignore"):
        cache[:, :, 580:584] = vs.view(np.uint8).reshape(cache.shape[0], 64, 4)
    return dict(c, cache=cache.reshape(c["num_blocks"], -1))


@pytest.mark.parametrize("num_splits", [1, 3, -1, -2])
def test_fp8_ragged_multi_page(num_splits):
    c = _fp8_case(5, 1, 128, [1, 63, 65, 700, 1000], seed=26)
    o, lse, st = run_decode(c, num_splits)
    o_ref, lse_ref = _oracle(c)
    assert st == 0
    err = compare_decode(o, lse, o_ref, lse_ref, fp8=True)
    print("fp8 errors", err)
    # the only rounding beyond fp32 is P * v_scale -> bf16: far inside the FP8 bound
    assert err["rel_l2"] <= 5e-3 and err["lse_max"] <= 1e-3, err


@pytest.mark.parametrize("num_splits", [1, -2])  # bf16 o_latent from the FP8 kernel's epilogue / merge
def test_fp8_bf16_output(num_splits):
    c = _fp8_case(3, 1, 64, [5, 64, 300], seed=29)
    o, lse, st = run_decode(c, num_splits, o_dtype=1)
    o_ref, lse_ref = _oracle(c)
    assert st == 0
    compare_decode(o, lse, o_ref, lse_ref, fp8=True, extra_abs=float(np.abs(o_ref).max()) * 2.0 ** -9)


def test_fp8_causal_two_rows_and_heads():
    c = _fp8_case(3, 2, 20, [0, 2, 333], seed=27, vscale=0.5)
    o, lse, st = run_decode(c, 2)
    o_ref, lse_ref = _oracle(c)
    assert st == 0
    compare_decode(o, lse, o_ref, lse_ref, fp8=True)


def test_fp8_widening_is_exact_for_every_code():
    """The FP8 decode kernel widens e4m3 codes with integer and bf16 arithmetic (no conversion
    instructions). Every finite code, subnormals included, must come out as its exact value (the
    oracle's e4m3 decode); the two NaN codes, which the cache writer never stores, read +-480."""
    import torch
    import mla_latent_kv_gb300 as mla
    out = torch.zeros(256, dtype=torch.int16, device="cuda")
    mla.selftest_e4m3_widen(out)
    torch.cuda.synchronize()
    got = oracle.widen_bf16(out.cpu().numpy().view(np.uint16))
    for code in range(256):
        want = {0x7F: 480.0, 0xFF: -480.0}.get(code, None)
        if want is None:
            want = oracle.e4m3_value(code)
        assert got[code] == want, (code, got[code], want)
    # the sign of zero survives too
    assert np.signbit(got[0x80]) and not np.signbit(got[0x00])


def test_fp8_bad_block_id_sets_device_status():
    c = _fp8_case(2, 1, 16, [100, 100], seed=28)
    bt = c["block_table"].copy()
    bt[0, 1] = -3
    _, _, st = run_decode(dict(c, block_table=bt), 1)
    assert st & 0x1


# ----------------------------------------------------------------------------- full workloads
def _sampled(c, heads=(0, 37, 127)):
    sel = [(b, t, h) for b in range(c["B"]) for t in range(c["Sq"]) for h in heads if h < c["H"]]
    return np.array(sel, np.int32)


@pytest.mark.slow
@pytest.mark.parametrize("name,num_splits", [("dsv3", -1), ("dsv3", 0), ("dsv3", -2), ("ragged", -1),
                                             ("ragged", -2), ("long_mtp", 0), ("long_mtp", -1), ("long_mtp", -2),
                                             ("fp8", -1), ("fp8", 0), ("fp8", -2)])
def test_full_workload_sampled(name, num_splits):
    c = mi.workload_case(name)
    o, lse, st = run_decode(c, num_splits)
    assert st == 0
    sel = _sampled(c)
    o_ref, lse_ref = _oracle(c, sel)
    idx = (sel[:, 0] * c["Sq"] + sel[:, 1]) * c["H"] + sel[:, 2]
    compare_decode(o.reshape(-1, 512)[idx], lse.reshape(-1)[idx], o_ref, lse_ref, fp8=c["kv"] == mi.KV_FP8)
    # every row of the full output: finite, lse finite exactly where the row has tokens
    n = np.array([[oracle.row_len(int(s), c["Sq"], t) for t in range(c["Sq"])] for s in c["seq_lens"]])
    assert np.isfinite(o).all()
    assert np.array_equal(np.isfinite(lse), np.broadcast_to((n > 0)[..., None], lse.shape))


def test_batch_invariance_without_splits():
    """num_splits = 1: a request's output bits do not depend on the batch it is decoded in (its
    position, its neighbours, the batch size)."""
    c = mi.decode_case(5, 1, 128, [1000, 37, 4096, 64, 900], seed=29)
    o_all, lse_all, st = run_decode(c, 1)
    assert st == 0
    for b in (0, 2):
        sub = dict(c, B=1, q=c["q"][b:b + 1], block_table=c["block_table"][b:b + 1], seq_lens=[c["seq_lens"][b]])
        o1, lse1, st1 = run_decode(sub, 1)
        assert st1 == 0
        np.testing.assert_array_equal(o1[0], o_all[b])
        np.testing.assert_array_equal(lse1[0], lse_all[b])


def test_device_schedule_bf16_output_and_one_long_row():
    """num_splits = -2 with a batch dominated by one long row: that row is cut into several
    units (partials + merge) while the short rows write their output directly; bf16 output."""
    c = mi.decode_case(6, 1, 128, [20000, 5, 64, 65, 300, 1], seed=31)
    o, lse, st = run_decode(c, -2, o_dtype=1)
    o_ref, lse_ref = _oracle(c)
    assert st == 0
    compare_decode(o, lse, o_ref, lse_ref, extra_abs=float(np.abs(o_ref).max()) * 2.0 ** -9)


def _up256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("lens,Sq", [
    ("loguniform", 1),                      # the ragged workload's length mix
    ([4096] * 64, 1),                       # uniform: one unit per row
    ([8192] * 128, 1),                      # uniform, more rows than SM pairs
    ([131072] * 4, 2),                      # few long rows: every row split evenly
    ([20000, 5, 64, 65, 300, 1], 1),        # one long row among short ones
    ([1 + (7 * i) % 500 for i in range(1100)], 1),  # more rows than the planner's threads
    ([0, 0, 64, 0], 1),                     # empty rows
])
def test_device_schedule_is_a_partition(lens, Sq):
    """The schedule that num_splits = -2 builds on the device, read back from the workspace: every
    query row's visible tokens [0, n) are covered by its units exactly once and in order, a split
    row's partial slots are consecutive, all slots are distinct, split rows are listed exactly
    once, and the list opens with a unit of the longest length class."""
    import torch
    import mla_latent_kv_gb300 as mla
    rng = np.random.default_rng(5)
    if lens == "loguniform":
        lens = [int(x) for x in np.exp(rng.uniform(0, np.log(32768), 128))]
    B, H = len(lens), 16
    ml = max(max(lens), 1)
    mb = (ml + 63) // 64
    dev = torch.device("cuda")
    q = torch.zeros((B, Sq, H, 576), dtype=torch.bfloat16, device=dev)
    cache = torch.zeros((1, 64 * 1152), dtype=torch.uint8, device=dev)  # every page is block 0
    bt = torch.zeros((B, mb), dtype=torch.int32, device=dev)
    sl = torch.tensor(lens, dtype=torch.int32, device=dev)
    ws = torch.zeros(mla.workspace_bytes(B, Sq, H, -2, mla.KV_BF16, ml), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    mla.decode(q, cache, bt, sl, ml, 0.1, num_splits=-2, workspace=ws, dev_status=st, num_blocks=1)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    w = ws.cpu().numpy()
    rows = B * Sq
    pairs = max(1, torch.cuda.get_device_properties(0).multi_processor_count // 2)
    max_units = rows + 2 * pairs
    count, n_split = (int(x) for x in w[:8].view(np.int32))
    assert 0 < count <= max_units and 0 <= n_split <= rows
    units = w[256:256 + 16 * count].view(np.int32).reshape(count, 4)
    rows_off = _up256(256 + max_units * 16)
    row_info = w[rows_off:rows_off + 8 * rows].view(np.int32).reshape(rows, 2)
    split_off = rows_off + _up256(rows * 8)
    split_rows = w[split_off:split_off + 4 * n_split].view(np.int32)
    assert np.all((units[:, 0] >= 0) & (units[:, 0] < rows))
    slots = units[units[:, 3] >= 0, 3]
    assert len(np.unique(slots)) == len(slots) and np.all(slots < max_units)
    # longest first by length class (units of about c pages, then classes >= c/2, c/4, ...): the
    # list opens with a unit of at least half the pages of the longest
    unit_pages = (units[:, 2] - units[:, 1] + 63) // 64
    assert 2 * unit_pages[0] >= unit_pages.max()
    for r in range(rows):
        b, t = divmod(r, Sq)
        n = max(0, lens[b] - (Sq - 1 - t))
        mine = units[units[:, 0] == r]
        slot0, S = (int(x) for x in row_info[r])
        assert len(mine) == S >= 1
        mine = mine[np.argsort(mine[:, 1], kind="stable")]
        assert mine[0, 1] == 0 and mine[-1, 2] == n
        assert np.all(mine[:, 1] <= mine[:, 2])
        assert np.all(mine[1:, 1] == mine[:-1, 2])
        if S > 1:
            assert sorted(mine[:, 3].tolist()) == list(range(slot0, slot0 + S))
        else:
            assert slot0 == -1 and mine[0, 3] == -1
    split_expected = sorted(r for r in range(rows) if row_info[r, 1] > 1)
    assert sorted(split_rows.tolist()) == split_expected


def test_default_split_choice_uses_the_device_schedule_for_many_rows():
    """num_splits = -1: with more query rows than SM pairs the units run in waves whose packing
    depends on the lengths, so the library builds the schedule on the device (-2); with fewer
    rows the host's uniform split stands."""
    import torch
    import mla_latent_kv_gb300 as mla
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    assert mla.resolve_num_splits(-1, pairs + 1, 1, 128, 32768) == -2
    assert mla.resolve_num_splits(-1, (pairs + 2) // 2, 2, 128, 4096) == -2
    assert mla.resolve_num_splits(-1, 64, 1, 128, 4096) == 1
    assert mla.resolve_num_splits(-1, 4, 2, 128, 131072) > 1
    assert mla.resolve_num_splits(3, 1000, 1, 128, 4096) == 3


# ----------------------------------------------------------------------------- packed variable-length rows
def _varlen_case(lens, qlens, H, seed, kv=mi.KV_BF16):
    c = mi.decode_case(len(lens), 1, H, lens, kv=kv, seed=seed)
    qsl = np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)
    rng = np.random.default_rng(seed + 1)
    q = mi.to_bf16_bits(rng.standard_normal((int(qsl[-1]), H, 576)).astype(np.float32))
    return dict(c, q=q, qsl=qsl)


@pytest.mark.parametrize("num_splits", [1, 3, -1, -2])
@pytest.mark.parametrize("kv", [mi.KV_BF16, mi.KV_FP8])
def test_varlen_mixed_query_lengths(num_splits, kv):
    import torch
    import mla_latent_kv_gb300 as mla
    v = _varlen_case([40, 700, 9, 64, 3000, 2], [1, 3, 0, 2, 4, 2], 64, seed=33, kv=kv)
    d = torch_dev(v)
    qsl = torch.from_numpy(v["qsl"]).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = mla.decode_varlen(d["q"], d["cache"], d["block_table"], d["seq_lens"], qsl, max(v["seq_lens"]),
                               v["scale"], kv_dtype=kv, num_splits=num_splits, dev_status=st,
                               num_blocks=v["num_blocks"])
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_ref, lse_ref = oracle.decode_varlen(v["q"], v["cache"], kv, v["num_blocks"], v["block_table"], v["seq_lens"],
                                          v["qsl"], 64, v["scale"])
    from parity_util import to_f64
    compare_decode(to_f64(o), to_f64(lse), o_ref, lse_ref, fp8=kv == mi.KV_FP8)


def test_uniform_four_token_queries():
    """Sq > 2 through the uniform entry point (MTP-style rows sharing one request's cache)."""
    c = mi.decode_case(3, 4, 32, [3, 500, 129], seed=34)
    o, lse, st = run_decode(c, -1)
    o_ref, lse_ref = _oracle(c)
    assert st == 0
    compare_decode(o, lse, o_ref, lse_ref)


@pytest.mark.slow
def test_dsv3_step_with_bf16_outputs_sampled():
    """The step the benchmark times at its headline workload, on the benchmark's inputs:
    absorb -> decode (o_latent stored in bf16, the planner's split count) -> out_proj (o stored in
    bf16). Sampled rows are checked against the oracle: q absorbed in fp64, the absorbed decode
    route, then the output projection. Each bf16 store rounds once, by at most half an ulp; here
    |o_latent| and |o| stay below 0.25, where that is under 5e-4, so the stated bounds apply with
    no allowance."""
    import torch
    import mla_latent_kv_gb300 as mla
    w = mi.WORKLOADS["dsv3"]
    c = mi.e2e_case(w["B"], w["Sq"], w["H"], w["lens"], seed=w["seed"])
    B, Sq, H = c["B"], c["Sq"], c["H"]
    T = B * Sq
    dev = torch.device("cuda")
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
    q = mla.absorb_q(bf(c["q_nope"]).reshape(T, H, 128), bf(c["q_pe"]).reshape(T, H, 64), bf(c["w_uk_t"]))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ol, lse = mla.decode(q.view(B, Sq, H, 576), torch.from_numpy(c["cache"]).to(dev),
                         torch.from_numpy(c["block_table"]).to(dev),
                         torch.from_numpy(np.asarray(c["seq_lens"], np.int32)).to(dev), int(max(c["seq_lens"])),
                         c["scale"], num_splits=-1, o_dtype=mla.DT_BF16, dev_status=status,
                         num_blocks=c["num_blocks"])
    o = mla.out_proj(ol.view(T, H, 512), bf(c["w_uv"]), out_dtype=mla.DT_BF16)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert ol.dtype == torch.bfloat16 and o.dtype == torch.bfloat16

    sel = _sampled(c)
    qa = oracle.absorb_q(c["q_nope"], c["q_pe"], c["w_uk_t"], T, H)
    ol_ref, lse_ref = oracle.decode_absorbed(qa.reshape(B, Sq, H, 576), c["cache"], c["kv"], c["num_blocks"],
                                             c["block_table"], c["seq_lens"], B, Sq, H, c["scale"], sel=sel)
    rows = sel[:, 0] * Sq + sel[:, 1]
    full = np.zeros((T, H, 512))
    full[rows, sel[:, 2]] = ol_ref
    o_ref = oracle.out_proj(full, c["w_uv"], T, H)[rows, sel[:, 2]]
    assert np.abs(ol_ref).max() < 0.25 and np.abs(o_ref).max() < 0.25

    ol_gpu = ol.double().cpu().numpy().reshape(T, H, 512)[rows, sel[:, 2]]
    lse_gpu = lse.double().cpu().numpy().reshape(T, H)[rows, sel[:, 2]]
    compare_decode(ol_gpu, lse_gpu, ol_ref, lse_ref)
    o_gpu = o.double().cpu().numpy()[rows, sel[:, 2]]
    assert np.abs(o_gpu - o_ref).max() <= TOL_MAX_ABS
    assert rel_l2(o_gpu, o_ref) <= TOL_REL_L2
