"""Host-side checks of the C ABI that need no GPU: the library loads, exports every function the
header declares, and its host-only helpers and argument validation behave as documented."""
import ctypes

import pytest

import mla_inputs as mi
import oracle

mla = pytest.importorskip("mla_latent_kv_gb300")


@pytest.fixture(scope="module")
def lib():
    from mla_latent_kv_gb300 import build
    build.build()
    return mla.lib()


def test_exports_every_declared_symbol(lib):
    names = mla.declared_functions()
    assert {"mla_absorb_q", "mla_decode", "mla_out_proj"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/mla_latent_kv.h but not exported"


def test_status_strings_and_row_bytes(lib):
    assert mla.status_string(0) == "MLA_OK"
    assert mla.status_string(3) == "MLA_ERR_WORKSPACE_TOO_SMALL"
    assert mla.status_string(99) == "MLA_ERR_UNKNOWN"
    assert mla.row_bytes(mla.KV_BF16) == 1152 == oracle.row_bytes(oracle.KV_BF16)
    assert mla.row_bytes(mla.KV_FP8) == 584 == oracle.row_bytes(oracle.KV_FP8)
    assert mla.row_bytes(7) == -1


def test_default_num_splits_agrees_with_oracle(lib):
    for n in [0, 1, 511, 512, 513, 1024, 4096, 8192, 32768, 131072, 10 ** 6]:
        for sms in [1, 76, 148, 152]:
            assert mla.default_num_splits(n, sms) == oracle.default_num_splits(n, sms), (n, sms)
    assert mla.default_num_splits(-1, 152) == -1 and mla.default_num_splits(10, 0) == -1


def test_workspace_bytes(lib):
    assert mla.workspace_bytes(64, 1, 128, 1) == 0
    ws = mla.workspace_bytes(4, 2, 128, 256)
    units = 4 * 2 * 256 * 128
    assert ws >= units * 513 * 4 and ws % 256 == 0 and ws - units * 513 * 4 < 512


def test_forced_split_count_needs_no_device(lib):
    assert lib.mla_resolve_num_splits(5, 2, 1, 16, 300) == 5
    assert lib.mla_resolve_num_splits(-2, 2, 1, 16, 300) == -1


def _decode_call(lib, **kw):
    args = dict(q=None, kv_cache=None, kv_dtype=0, num_blocks=0, block_table=None, max_blocks=0,
                seq_lens=None, max_seq_len=0, B=1, Sq=1, H=16, scale=0.07, num_splits=1, workspace=None,
                workspace_bytes=0, o_latent=None, o_dtype=0, lse=None, dev_status=None, stream=None)
    args.update(kw)
    return lib.mla_decode(*args.values())


def test_decode_validation_before_any_launch(lib):
    assert _decode_call(lib, H=0) == mla.ERR_UNSUPPORTED
    assert _decode_call(lib, H=129) == mla.ERR_UNSUPPORTED
    assert _decode_call(lib, B=-1) == mla.ERR_INVALID_ARG
    assert _decode_call(lib, Sq=0) == mla.ERR_INVALID_ARG
    assert _decode_call(lib, kv_dtype=5) == mla.ERR_INVALID_ARG
    assert _decode_call(lib, o_dtype=9) == mla.ERR_INVALID_ARG
    assert _decode_call(lib, scale=0.0) == mla.ERR_INVALID_ARG
    assert _decode_call(lib, scale=float("nan")) == mla.ERR_INVALID_ARG
    assert _decode_call(lib, max_seq_len=65, max_blocks=1) == mla.ERR_INVALID_ARG
    assert _decode_call(lib, num_splits=-3) == mla.ERR_INVALID_ARG
    assert _decode_call(lib) == mla.ERR_INVALID_ARG  # null q / o_latent
    assert b"null" in lib.mla_last_error_detail()
    assert _decode_call(lib, B=0) == mla.OK  # nothing to do, nothing launched
    bad = ctypes.c_void_p(0x1001)  # misaligned; rejected before any device access
    assert _decode_call(lib, q=bad, o_latent=bad, seq_lens=bad) == mla.ERR_UNSUPPORTED


def test_gemm_validation_before_any_launch(lib):
    f = lib.mla_absorb_q
    assert f(None, 128, 128, None, 64, 64, None, None, 4, 0, None) == mla.ERR_UNSUPPORTED
    assert f(None, 128, 128, None, 64, 64, None, None, -1, 4, None) == mla.ERR_INVALID_ARG
    assert f(None, 128, 128, None, 64, 64, None, None, 0, 4, None) == mla.OK
    assert f(None, 128, 128, None, 64, 64, None, None, 3, 4, None) == mla.ERR_INVALID_ARG
    al = ctypes.c_void_p(0x1000)
    assert f(al, 100, 128, None, 64, 64, al, al, 3, 4, None) == mla.ERR_UNSUPPORTED  # stride % 8
    g = lib.mla_out_proj
    assert g(None, 0, None, None, 0, 4, 200, None) == mla.ERR_UNSUPPORTED
    assert g(None, 7, None, None, 0, 4, 2, None) == mla.ERR_INVALID_ARG
    assert g(None, 0, None, None, 0, 0, 2, None) == mla.OK
    assert g(None, 0, None, None, 0, 4, 2, None) == mla.ERR_INVALID_ARG


def test_workload_table_matches_configs():
    w = mi.WORKLOADS
    assert (w["dsv3"]["B"], w["dsv3"]["H"], w["dsv3"]["lens"][0]) == (64, 128, 4096)
    assert (w["long_mtp"]["B"], w["long_mtp"]["Sq"], w["long_mtp"]["lens"][0]) == (4, 2, 131072)
    assert w["fp8"]["kv"] == mi.KV_FP8 and w["fp8"]["lens"][0] == 8192
    import numpy as np
    lens = mi.draw_lengths("loguniform", 128, np.random.default_rng(2))
    assert list(lens[:6]) == [1, 63, 64, 65, 128, 32768] and lens.min() >= 1 and lens.max() <= 32768


def test_workspace_bytes_by_cache_format(lib):
    up = lambda x: (x + 255) // 256 * 256
    B, Sq, H, S, L = 3, 2, 16, 4, 130
    split = up(B * Sq * S * H * 512 * 4) + up(B * Sq * S * H * 4)
    assert mla.workspace_bytes(B, Sq, H, S) == split
    assert mla.workspace_bytes(B, Sq, H, S, mla.KV_BF16, L) == split
    # the FP8 cache is widened on chip: no scratch beyond the split partials
    assert mla.workspace_bytes(B, Sq, H, S, mla.KV_FP8, L) == split
    assert mla.workspace_bytes(B, Sq, H, 1, mla.KV_FP8, L) == 0
    assert mla.workspace_bytes(B, Sq, H, 1, mla.KV_FP8, 1 << 20) == 0
    assert lib.mla_decode_workspace_bytes_kv(7, B, Sq, H, S, L) == 0


# ----------------------------------------------------------------------------- prefill host logic
@pytest.mark.parametrize("budget", [64, 100, 128, 500, 4096, 1 << 20])
def test_prefill_chunk_plan_is_bit_exact_with_oracle(lib, budget):
    import numpy as np
    rng = np.random.default_rng(budget)
    ctx = rng.integers(0, 2000, size=57).astype(np.int32)
    ctx[[0, 9, 10]] = 0
    ctx[3] = 64
    ctx[4] = 65
    got = mla.prefill_chunk_plan(ctx, budget)
    want = oracle.prefill_chunks(ctx, budget)
    assert got.dtype == want.dtype and np.array_equal(got, want)


def test_prefill_plan_and_workspace_argument_checks(lib):
    import numpy as np
    with pytest.raises(mla.MlaError):
        mla.prefill_chunk_plan([10, 20], 63)
    assert mla.prefill_workspace_bytes(4, 100, 128, 63) == 0
    assert mla.prefill_workspace_bytes(4, 100, 129, 8192) == 0
    ws = mla.prefill_workspace_bytes(4, 100, 128, 8192)
    # the per-row K / V workspace dominates: 8192 rows x 128 heads x (128 + 128) bf16
    assert ws >= 8192 * 128 * 256 * 2 and ws % 256 == 0
    assert mla.prefill_workspace_bytes(4, 10000, 16, 64) > mla.prefill_workspace_bytes(4, 100, 16, 64)
    assert int(lib.mla_prefill_chunk_plan(np.zeros(3, np.int32).ctypes.data, 3, 64, None, 0)) == 0


def test_prefill_rejects_bad_arguments_before_any_launch(lib):
    import numpy as np
    ctx = np.array([10, 0], np.int32)
    qsl = np.array([0, 3, 5], np.int32)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails first

    def call(B=2, H=4, ctx_h=ctx, qsl_h=qsl, chunk=64, scale=0.07, kv=0, ws_bytes=1 << 30, max_blocks=1):
        return int(lib.mla_prefill(fake, fake, 512, fake, 64, fake, kv, 10, fake, max_blocks, fake, fake,
                                   ctx_h.ctypes.data, qsl_h.ctypes.data, B, H, fake, fake, scale, chunk, fake,
                                   ws_bytes, fake, None, None, None))
    assert call(H=0) == mla.ERR_UNSUPPORTED
    assert call(H=129) == mla.ERR_UNSUPPORTED
    assert call(B=0) == mla.ERR_INVALID_ARG
    assert call(chunk=32) == mla.ERR_INVALID_ARG
    assert call(scale=0.0) == mla.ERR_INVALID_ARG
    assert call(kv=5) == mla.ERR_INVALID_ARG
    assert call(qsl_h=np.array([1, 3, 5], np.int32)) == mla.ERR_INVALID_ARG
    assert call(qsl_h=np.array([0, 3, 2], np.int32)) == mla.ERR_INVALID_ARG
    assert call(ctx_h=np.array([65, 0], np.int32), max_blocks=1) == mla.ERR_INVALID_ARG
    assert call(ctx_h=np.array([-1, 0], np.int32)) == mla.ERR_INVALID_ARG
    assert call(ws_bytes=100) == mla.ERR_WORKSPACE_TOO_SMALL
    # nothing to do: no query rows
    assert call(qsl_h=np.array([0, 0, 0], np.int32)) == mla.OK


def test_binding_output_buffers_match_their_dtype_code():
    # the kernels write through the output pointer with the element size of the dtype code, so
    # the binding derives the code from a given buffer and refuses one that does not fit it
    import torch
    import mla_latent_kv_gb300 as mla
    bf = torch.empty((2, 3, 512), dtype=torch.bfloat16)
    f32 = torch.empty((2, 3, 512), dtype=torch.float32)
    assert mla._dt_code(None, None) == mla.DT_F32
    assert mla._dt_code(bf, None) == mla.DT_BF16
    assert mla._dt_code(f32, None) == mla.DT_F32
    assert mla._dt_code(bf, mla.DT_F32) == mla.DT_F32  # an explicit code wins, and is then checked
    assert mla._out_buf(bf, (2, 3, 512), mla.DT_BF16, "cpu") is bf
    made = mla._out_buf(None, (4, 5), mla.DT_BF16, "cpu")
    assert made.dtype == torch.bfloat16 and tuple(made.shape) == (4, 5)
    with pytest.raises(ValueError):
        mla._out_buf(bf, (2, 3, 512), mla.DT_F32, "cpu")  # fp32 rows into a bf16 buffer
    with pytest.raises(ValueError):
        mla._out_buf(f32, (2, 4, 512), mla.DT_F32, "cpu")  # too small
    with pytest.raises(ValueError):
        mla._out_buf(f32.transpose(0, 1), (3, 2, 512), mla.DT_F32, "cpu")  # not contiguous


def test_selftest_rejects_null_pointers_before_any_launch(lib):
    import mla_latent_kv_gb300 as mla
    assert lib.mla_selftest_wait_timeout(None, None, None) == mla.ERR_INVALID_ARG
