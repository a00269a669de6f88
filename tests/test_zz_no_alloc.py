"""mla_decode_noalloc: the decode entry point whose split-KV scratch is the library's own fixed
device array. Called through the C ABI and compared with mla_decode (which takes a caller
workspace) under the decode tolerances, on two different calls in a row, so that the second
call runs over the scratch the first one left behind."""
import ctypes

import numpy as np
import pytest

import mla_inputs as mi
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


def test_two_calls_in_a_row_match_mla_decode():
    cases = [(mi.decode_case(6, 1, 128, [1, 63, 64, 65, 700, 1000], seed=40), 3),
             (mi.decode_case(4, 2, 64, [0, 2, 200, 517], seed=41), 4)]
    results = []
    for c, S in cases:
        results.append((c, S, _run_noalloc(c, S)))
    for c, S, (o, lse, st) in results:
        assert st == 0
        o_ref, lse_ref, st_ref = run_decode(c, S)
        assert st_ref == 0
        compare_decode(o, lse, o_ref, lse_ref)


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
