"""GPU parity of mla_cache_write against the oracle: the written cache bytes must be identical
(bf16 copy and FP8 quantise are integer / byte results), and a decode over a cache written on
the GPU must match the oracle's decode over the cache the oracle wrote."""
import numpy as np
import pytest

import mla_inputs as mi
import oracle
from parity_util import compare_decode, run_decode

pytestmark = pytest.mark.gpu


def _case(T, seed, spare=3, scale=2.0):
    rng = np.random.default_rng(seed)
    kv_c = mi.to_bf16_bits(rng.standard_normal((T, 512)).astype(np.float32) * scale)
    k_pe = mi.to_bf16_bits(rng.standard_normal((T, 64)).astype(np.float32))
    nb = (T + 63) // 64 + spare
    slots = rng.permutation(nb * 64)[:T].astype(np.int64)
    return kv_c, k_pe, slots, nb


def _gpu_write(kv_c, k_pe, slots, kv, cache0, nb, kv_scale=0.0):
    import torch
    import mla_latent_kv_gb300 as mla
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)  # noqa
    cache = torch.from_numpy(cache0.copy()).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.cache_write(d(kv_c), d(k_pe), torch.from_numpy(slots).cuda(), cache, kv_dtype=kv, kv_scale=kv_scale,
                    dev_status=status, num_blocks=nb)
    torch.cuda.synchronize()
    return cache.cpu().numpy(), int(status.item())


@pytest.mark.parametrize("kv,kv_scale", [(mi.KV_BF16, 0.0), (mi.KV_FP8, 0.0), (mi.KV_FP8, 0.05), (mi.KV_FP8, 1.0)])
def test_cache_bytes_identical(kv, kv_scale):
    T = 300
    kv_c, k_pe, slots, nb = _case(T, 80)
    kv_c[7] = 0
    k_pe[7] = 0                        # all-zero row: scale 1
    slots[3] = -1                      # padding token
    slots[11] = nb * 64 + 5            # beyond the cache
    rb = mi.ROW_BYTES[kv]
    cache0 = np.random.default_rng(81).integers(0, 256, (nb, 64 * rb), dtype=np.uint8)  # stale contents
    ref = cache0.copy()
    assert oracle.cache_write(kv_c, k_pe, slots, kv, ref, nb, kv_scale=kv_scale) == 1
    got, st = _gpu_write(kv_c, k_pe, slots, kv, cache0, nb, kv_scale)
    assert st == 0x8
    np.testing.assert_array_equal(got, ref)


def test_strided_views_and_large_batch():
    import torch
    import mla_latent_kv_gb300 as mla
    T = 5000
    kv_c, k_pe, slots, nb = _case(T, 82, scale=30.0)
    full = np.concatenate([kv_c, k_pe, np.zeros((T, 64), np.uint16)], axis=1)  # [T, 640] rows
    ref = np.zeros((nb, 64 * 584), np.uint8)
    oracle.cache_write(full[:, :512], full[:, 512:576], slots, mi.KV_FP8, ref, nb)
    fd = torch.from_numpy(full.view(np.int16)).cuda().view(torch.bfloat16)
    cache = torch.zeros((nb, 64 * 584), dtype=torch.uint8, device="cuda")
    mla.cache_write(fd[:, :512], fd[:, 512:576], torch.from_numpy(slots).cuda(), cache, kv_dtype=mla.KV_FP8)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(cache.cpu().numpy(), ref)


def test_decode_over_gpu_written_fp8_cache():
    """Write a request's tokens with the GPU, decode them with the GPU; the oracle writes and
    decodes the same tokens on its own. Outputs meet the FP8 tolerance."""
    B, lens, H = 3, [70, 1, 200], 32
    rng = np.random.default_rng(83)
    nb = sum((n + 63) // 64 for n in lens) + 2
    perm = rng.permutation(nb)
    max_blocks = max((n + 63) // 64 for n in lens)
    bt = np.full((B, max_blocks), -1, np.int32)
    slots, k = [], 0
    for b, n in enumerate(lens):
        for pg in range((n + 63) // 64):
            bt[b, pg] = perm[k]
            k += 1
        slots += [int(bt[b, j // 64]) * 64 + j % 64 for j in range(n)]
    slots = np.array(slots, np.int64)
    T = len(slots)
    kv_c = mi.to_bf16_bits(rng.standard_normal((T, 512)).astype(np.float32))
    k_pe = mi.to_bf16_bits(rng.standard_normal((T, 64)).astype(np.float32))
    ref_cache = np.zeros((nb, 64 * 584), np.uint8)
    oracle.cache_write(kv_c, k_pe, slots, mi.KV_FP8, ref_cache, nb)
    got_cache, st = _gpu_write(kv_c, k_pe, slots, mi.KV_FP8, np.zeros_like(ref_cache), nb)
    assert st == 0
    q = mi.to_bf16_bits(rng.standard_normal((B, 1, H, 576)).astype(np.float32))
    base = dict(B=B, Sq=1, H=H, kv=mi.KV_FP8, seq_lens=lens, block_table=bt, num_blocks=nb, q=q, scale=mi.SCALE)
    o_ref, lse_ref = oracle.decode_absorbed(q, ref_cache, mi.KV_FP8, nb, bt, lens, B, 1, H, mi.SCALE)
    o, lse, st = run_decode(dict(base, cache=got_cache), 1)
    assert st == 0
    compare_decode(o, lse, o_ref, lse_ref, fp8=True)
