"""Helpers shared by the GPU parity tests: move seeded numpy inputs to the device, run the three
library calls through the Python binding, and compare with the oracle under the stated
tolerances."""
from __future__ import annotations

import numpy as np

# Tolerances of the decode path (bf16 cache): on o and o_latent max |err| <= 1e-2 and relative
# L2 <= 5e-3; on lse |err| <= 1e-3. FP8 cache: relative L2 <= 2e-2 against an oracle fed the
# identically dequantised values.
TOL_MAX_ABS = 1e-2
TOL_REL_L2 = 5e-3
TOL_LSE = 1e-3
TOL_FP8_REL_L2 = 2e-2


def torch_dev(c):
    import torch
    dev = torch.device("cuda:0")
    out = {}
    out["q"] = torch.from_numpy(c["q"].view(np.int16)).to(dev).view(torch.bfloat16)
    out["cache"] = torch.from_numpy(c["cache"].view(np.uint8)).to(dev)
    out["block_table"] = torch.from_numpy(c["block_table"]).to(dev)
    out["seq_lens"] = torch.from_numpy(np.asarray(c["seq_lens"], np.int32)).to(dev)
    return out


def bf16_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def to_f64(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def run_decode(c, num_splits=0, o_dtype=0, dev=None, with_status=True):
    import torch
    import mla_latent_kv_gb300 as mla
    d = dev or torch_dev(c)
    status = torch.zeros(1, dtype=torch.int32, device="cuda") if with_status else None
    o, lse = mla.decode(d["q"], d["cache"], d["block_table"], d["seq_lens"], int(np.max(c["seq_lens"], initial=0)),
                        c["scale"], kv_dtype=c["kv"], num_splits=num_splits, o_dtype=o_dtype,
                        dev_status=status, num_blocks=c["num_blocks"])
    torch.cuda.synchronize()
    st = int(status.item()) if status is not None else 0
    return to_f64(o), to_f64(lse), st


def rel_l2(a, b):
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def compare_decode(o, lse, o_ref, lse_ref, fp8=False, extra_abs=0.0):
    """o / o_ref [..., 512], lse / lse_ref [...]. Rows with no visible token must be exactly
    o = 0, lse = -inf. Returns a dict of the measured errors (asserts the tolerances)."""
    o = np.asarray(o).reshape(-1, 512)
    o_ref = np.asarray(o_ref).reshape(-1, 512)
    lse = np.asarray(lse).reshape(-1)
    lse_ref = np.asarray(lse_ref).reshape(-1)
    empty = lse_ref == -np.inf
    assert np.all(lse[empty] == -np.inf), "empty rows must report lse = -inf"
    assert np.all(o[empty] == 0), "empty rows must report o = 0"
    assert np.isfinite(o).all(), "non-finite output"
    full = ~empty
    err = {"max_abs": float(np.abs(o - o_ref).max()) if o.size else 0.0,
           "rel_l2": rel_l2(o[full], o_ref[full]) if full.any() else 0.0,
           "lse_max": float(np.abs(lse[full] - lse_ref[full]).max()) if full.any() else 0.0}
    if fp8:
        assert err["rel_l2"] <= TOL_FP8_REL_L2, err
    else:
        assert err["max_abs"] <= TOL_MAX_ABS + extra_abs, err
        assert err["rel_l2"] <= TOL_REL_L2, err
        assert err["lse_max"] <= TOL_LSE, err
    return err
