"""GPU parity of mla_absorb_q and mla_out_proj, and of the three calls chained end to end, against
the fp64 oracle (the end-to-end reference is the oracle's NON-absorbed route)."""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from parity_util import TOL_MAX_ABS, TOL_REL_L2, bf16_dev, rel_l2, to_f64, torch_dev

pytestmark = pytest.mark.gpu


def _bf16_to_f64(t):
    import torch
    return t.to(torch.float64).cpu().numpy()


@pytest.mark.parametrize("T,H", [(1, 1), (2, 16), (8, 128), (64, 128), (130, 128), (300, 7)])
def test_absorb_q(T, H):
    import mla_latent_kv_gb300 as mla
    a = mi.absorb_case(T, H, seed=30 + T + H)
    qn, qp, wk = bf16_dev(a["q_nope"]), bf16_dev(a["q_pe"]), bf16_dev(a["w_uk_t"])
    q = mla.absorb_q(qn, qp, wk)
    ref = oracle.absorb_q(a["q_nope"], a["q_pe"], a["w_uk_t"], T, H)
    got = _bf16_to_f64(q)
    # one rounding of an fp32 dot product of 128 bf16 products to bf16: within one bf16 ulp
    lat = np.abs(got[..., :512] - ref[..., :512])
    assert np.all(lat <= np.abs(ref[..., :512]) * 2.0 ** -8 + 1e-5), lat.max()
    np.testing.assert_array_equal(got[..., 512:], ref[..., 512:])


def test_absorb_q_strided_views_and_no_rope():
    """q_nope / q_pe as views into one [T, H, 192] tensor; q_pe = None leaves 512: untouched."""
    import torch
    import mla_latent_kv_gb300 as mla
    T, H = 24, 32
    a = mi.absorb_case(T, H, seed=40)
    full = np.concatenate([a["q_nope"], a["q_pe"]], axis=-1)  # [T, H, 192]
    fd = bf16_dev(full)
    wk = bf16_dev(a["w_uk_t"])
    q = mla.absorb_q(fd[..., :128], fd[..., 128:], wk)
    ref = oracle.absorb_q(a["q_nope"], a["q_pe"], a["w_uk_t"], T, H)
    got = _bf16_to_f64(q)
    assert np.all(np.abs(got[..., :512] - ref[..., :512]) <= np.abs(ref[..., :512]) * 2.0 ** -8 + 1e-5)
    np.testing.assert_array_equal(got[..., 512:], ref[..., 512:])
    out = torch.full((T, H, 576), 3.0, dtype=torch.bfloat16, device="cuda")
    mla.absorb_q(fd[..., :128], None, wk, out=out)
    assert torch.all(out[..., 512:] == 3.0)


@pytest.mark.parametrize("T,H,in_bf16,out_bf16", [(1, 1, False, False), (8, 128, False, False),
                                                   (64, 128, False, False), (130, 16, True, False),
                                                   (64, 128, False, True), (300, 5, False, False)])
def test_out_proj(T, H, in_bf16, out_bf16):
    import torch
    import mla_latent_kv_gb300 as mla
    c = mi.out_proj_case(T, H, seed=50 + T + H)
    x = c["o_latent"]
    if in_bf16:
        xb = mi.to_bf16_bits(x)
        xd = bf16_dev(xb)
        ref = oracle.out_proj(xb, c["w_uv"], T, H)
    else:
        xd = torch.from_numpy(x).cuda()
        ref = oracle.out_proj(x, c["w_uv"], T, H)
    o = mla.out_proj(xd, bf16_dev(c["w_uv"]), out_dtype=mla.DT_BF16 if out_bf16 else mla.DT_F32)
    got = to_f64(o)
    extra = float(np.abs(ref).max()) * 2.0 ** -9 if out_bf16 else 0.0
    assert np.abs(got - ref).max() <= TOL_MAX_ABS + extra
    assert rel_l2(got, ref) <= TOL_REL_L2
    if not out_bf16:
        # fp32 accumulation of 512 products whose fp32 operand is carried as bf16 hi + lo: the
        # result is close to exact, far inside the decode tolerance
        assert np.abs(got - ref).max() <= 1e-4 * max(1.0, float(np.abs(ref).max()))


@pytest.mark.parametrize("B,Sq,H,lens,splits", [(2, 1, 16, [128, 300], 0), (3, 2, 128, [1, 65, 400], 3),
                                                 (4, 1, 128, [64, 1000, 2, 129], -1)])
def test_end_to_end_vs_nonabsorbed(B, Sq, H, lens, splits):
    """absorb -> decode -> out_proj on the GPU against the oracle's non-absorbed route (full K / V
    up-projection per head). o and o_latent meet the decode tolerances; lse differs from the
    non-absorbed value by the bf16 rounding of ql_nope and is reported against a 1e-2 bound."""
    import torch
    import mla_latent_kv_gb300 as mla
    c = mi.e2e_case(B, Sq, H, lens, seed=60 + B)
    d = torch_dev(c)
    qn = bf16_dev(c["q_nope"]).reshape(B * Sq, H, 128)
    qp = bf16_dev(c["q_pe"]).reshape(B * Sq, H, 64)
    q = mla.absorb_q(qn, qp, bf16_dev(c["w_uk_t"]))
    ol, lse = mla.decode(q.reshape(B, Sq, H, 576), d["cache"], d["block_table"], d["seq_lens"], max(lens),
                         c["scale"], num_splits=splits, num_blocks=c["num_blocks"])
    o = mla.out_proj(ol.reshape(B * Sq, H, 512), bf16_dev(c["w_uv"]))
    torch.cuda.synchronize()
    o_ref, ol_ref, lse_ref = oracle.decode_nonabsorbed(c["q_nope"], c["q_pe"], c["cache"], c["kv"],
                                                       c["num_blocks"], c["block_table"], c["seq_lens"],
                                                       c["w_uk_t"], c["w_uv"], B, Sq, H, c["scale"])
    ol_g, lse_g, o_g = to_f64(ol), to_f64(lse), to_f64(o).reshape(o_ref.shape)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_g), fin)
    assert np.abs(ol_g - ol_ref).max() <= TOL_MAX_ABS and rel_l2(ol_g[fin], ol_ref[fin]) <= TOL_REL_L2
    assert np.abs(o_g - o_ref).max() <= TOL_MAX_ABS and rel_l2(o_g[fin], o_ref[fin]) <= TOL_REL_L2
    lse_err = float(np.abs(lse_g[fin] - lse_ref[fin]).max())
    print(f"end-to-end lse error vs non-absorbed route: {lse_err:.2e}")
    assert lse_err <= 1e-2
