"""The benchmark's roofline arithmetic, pinned by hand: every reported fraction divides by these
algorithmic byte and flop counts, so they are checked here against sums written out term by term
from the problem statement (no GPU needed)."""
import importlib.util
import os

import numpy as np

import mla_inputs as mi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    m = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(m)
    return m


def _shape_only(name):
    # algorithmic() reads only the shape fields and the lengths, not the cache bytes
    w = mi.WORKLOADS[name]
    lens = np.asarray(w["lens"], np.int64)
    return dict(B=w["B"], Sq=w["Sq"], H=w["H"], kv=w["kv"], seq_lens=lens)


def test_decode_bytes_and_flops_at_the_headline_workload():
    b = _bench()
    c = _shape_only("dsv3")
    kv = 64 * 4096 * 1152         # every cached row read once: 576 bf16 = 1152 bytes
    q = 64 * 128 * 576 * 2        # absorbed q, bf16
    lse = 64 * 128 * 4            # fp32
    table = 64 * 64 * 4 + 64 * 4  # one int32 block-table entry per page, one seq_len per request
    for o_bytes in (2, 4):
        o = 64 * 128 * 512 * o_bytes
        byts, flops, kv_bytes = b.algorithmic(c, o_bytes=o_bytes)
        assert kv_bytes == kv == 301_989_888
        assert byts == kv + q + o + lse + table
    assert b.algorithmic(c, o_bytes=2)[0] == 319_865_088
    assert b.algorithmic(c, o_bytes=4)[0] == 328_253_696
    # 2 flops per multiply-add: q.k over 576 dims and p.v over 512, per (row, token, head)
    assert b.algorithmic(c)[1] == 64 * 4096 * 128 * 2 * (576 + 512) == 73_014_444_032


def test_decode_flops_follow_the_causal_row_lengths():
    # two query rows per request: row t sees seq_len - (Sq - 1 - t) tokens, the KV is read once
    b = _bench()
    c = _shape_only("long_mtp")
    byts, flops, kv_bytes = b.algorithmic(c)
    assert kv_bytes == 4 * 131072 * 1152
    assert flops == 4 * (131071 + 131072) * 128 * 2 * (576 + 512)


def test_prefill_flops():
    # 4 requests, 4096 cached + 1024 new tokens each: every row is up-projected into k_nope and v
    # (512 -> 2 x 128 per head); query t sees the 4096 cached keys and new keys 0..t
    b = _bench()
    total, up, attn = b.prefill_flops([4096] * 4, [1024] * 4, 128)
    assert up == 4 * (4096 + 1024) * 128 * 2 * 512 * 256
    assert attn == 4 * (1024 * 4096 + 1024 * 1025 // 2) * 128 * 2 * (192 + 128)
    assert total == up + attn == 2_233_550_766_080
