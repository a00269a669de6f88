"""mla_decode_noalloc: the decode entry point for callers that cannot allocate device memory when
they decode. Its split-KV scratch is the library's own fixed device array instead of a caller
workspace. Called through the C ABI and checked against the fp64 oracle and against mla_decode
(which takes a caller workspace) under the decode tolerances, on two different calls in a row,
so that the second call runs over the scratch the first one left behind. This file is collected
last, so a run that stops at its first failure has run every other test already."""
import ctypes

import numpy as np
import pytest

import mla_inputs as mi
import oracle
from parity_util import compare_decode, run_decode, to_f64, torch_dev

pytestmark = pytest.mark.gpu

mla = pytest.importorskip("mla_latent_kv_gb300")


def _run_noalloc(c, num_splits):
    import torch
    d = torch_dev(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = mla.decode_noalloc(d["q"], d["cache"], d["block_table"], d["seq_lens"],
                                int(np.max(c["seq_lens"], initial=0)), c["scale"], kv_dtype=c["kv"],
                                num_splits=num_splits, dev_status=status, num_blocks=c["num_blocks"])
    torch.cuda.synchronize()
    return to_f64(o), to_f64(lse), int(status.item())


def _oracle(c):
    return oracle.decode_absorbed(c["q"], c["cache"], c["kv"], c["num_blocks"], c["block_table"],
                                  c["seq_lens"], c["B"], c["Sq"], c["H"], c["scale"])


def _fp8_case(B, Sq, H, lens, seed):
    """FP8 cache with v_scale = 2 * k_scale, so that a swap of the two scales cannot pass."""
    c = mi.decode_case(B, Sq, H, lens, kv=mi.KV_FP8, seed=seed)
    cache = c["cache"].reshape(c["num_blocks"], 64, 584)
    ks = cache[:, :, 576:580].copy().view("<f4")
    with np.errstate(invalid="ignore"):
        cache[:, :, 580:584] = (ks * np.float32(2.0)).astype("<f4").view(np.uint8).reshape(cache.shape[0], 64, 4)
    return dict(c, cache=cache.reshape(c["num_blocks"], -1))


@pytest.mark.parametrize("num_splits", [3, 0, -1, -2])
def test_two_calls_in_a_row_match_the_oracle_and_mla_decode(num_splits):
    cases = [mi.decode_case(6, 1, 128, [1, 63, 64, 65, 700, 1000], seed=40),
             mi.decode_case(4, 2, 64, [0, 2, 200, 517], seed=41)]
    results = [(c, _run_noalloc(c, num_splits)) for c in cases]  # back to back on the shared scratch
    for c, (o, lse, st) in results:
        assert st == 0
        o_ref, lse_ref = _oracle(c)
        compare_decode(o, lse, o_ref, lse_ref)
        o_ws, lse_ws, st_ws = run_decode(c, num_splits)
        assert st_ws == 0
        compare_decode(o, lse, o_ws, lse_ws)


def test_fp8_cache_two_calls_in_a_row():
    cases = [_fp8_case(3, 1, 32, [5, 300, 130], seed=42), _fp8_case(2, 2, 16, [70, 2], seed=43)]
    results = [(c, _run_noalloc(c, 2)) for c in cases]
    for c, (o, lse, st) in results:
        assert st == 0
        o_ref, lse_ref = _oracle(c)
        compare_decode(o, lse, o_ref, lse_ref, fp8=True)


def test_oversized_split_plan_is_refused():
    lib = mla.lib()
    cap = mla.noalloc_max_workspace_bytes()
    assert cap == 64 << 20
    B, Sq, H, S = 64, 1, 128, 8
    assert mla.workspace_bytes(B, Sq, H, S) > cap
    st = lib.mla_decode_noalloc(None, None, 0, 1, None, 1, None, 64, B, Sq, H, ctypes.c_float(0.07), S,
                                None, 0, None, None, None)
    assert st == 3  # MLA_ERR_WORKSPACE_TOO_SMALL
    assert b"mla_decode_noalloc" in lib.mla_last_error_detail()
