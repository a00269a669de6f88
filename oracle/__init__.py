"""fp64 CPU oracle for MLA latent-KV decode -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg may
import this package. It shares no code with the CUDA library (``mla_latent_kv_gb300``): the C
source ``mla_oracle.c`` is compiled on its own with gcc, and this module only marshals numpy
arrays into it. What each function computes, and which page passage it follows, is documented
in ``mla_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

KV_BF16 = 0
KV_FP8 = 1
L, R, D, P, V, PAGE = 512, 64, 576, 128, 128, 64


def build(force: bool = False) -> str:
    """Compile mla_oracle.c into _build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wno-unknown-pragmas",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.oracle_bf16_value.restype = dbl
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_value.restype = dbl
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_widen_bf16.argtypes = [vp, i64, vp]
        lib.oracle_widen_e4m3.argtypes = [vp, i64, vp]
        lib.oracle_row_bytes.restype = i64
        lib.oracle_row_bytes.argtypes = [i32]
        lib.oracle_row_len.restype = i64
        lib.oracle_row_len.argtypes = [ctypes.c_int32, i32, i32]
        lib.oracle_merge.argtypes = [vp, vp, i32, vp, vp]
        lib.oracle_decode_absorbed.restype = i32
        lib.oracle_decode_absorbed.argtypes = [vp, vp, i32, i64, vp, i32, vp, i32, i32, i32, dbl,
                                               i64, vp, i64, vp, vp]
        lib.oracle_absorb_q.argtypes = [vp, i64, i64, vp, i64, i64, vp, i32, i32, vp]
        lib.oracle_out_proj.argtypes = [vp, vp, i32, i32, vp]
        lib.oracle_decode_nonabsorbed.restype = i32
        lib.oracle_decode_nonabsorbed.argtypes = [vp, vp, vp, i32, i64, vp, i32, vp, vp, vp, i32,
                                                  i32, i32, dbl, vp, i64, vp, vp, vp]
        lib.oracle_default_num_splits.restype = i32
        lib.oracle_default_num_splits.argtypes = [i32, i32]
        lib.oracle_decode_varlen.restype = i32
        lib.oracle_decode_varlen.argtypes = [vp, vp, i32, i64, vp, i32, vp, vp, i32, i32, dbl, vp, vp]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_cache_write.restype = i64
        lib.oracle_cache_write.argtypes = [vp, i64, vp, i64, vp, i64, i32, ctypes.c_float, vp, i64]
        lib.oracle_prefill_chunks.restype = i64
        lib.oracle_prefill_chunks.argtypes = [vp, i32, i64, vp]
        lib.oracle_prefill.restype = i32
        lib.oracle_prefill.argtypes = [vp, vp, vp, vp, i32, i64, vp, i32, vp, vp, i32, i32, vp, vp, dbl, i64,
                                       vp, vp]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


# ---------------------------------------------------------------- element formats
def bf16_value(h: int) -> float:
    return _load().oracle_bf16_value(int(h))


def e4m3_value(b: int) -> float:
    return _load().oracle_e4m3_value(int(b))


def widen_bf16(a) -> np.ndarray:
    a = _u16(a)
    out = np.empty(a.shape, np.float64)
    _load().oracle_widen_bf16(_ptr(a), a.size, _ptr(out))
    return out


def widen_e4m3(a) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.uint8))
    out = np.empty(a.shape, np.float64)
    _load().oracle_widen_e4m3(_ptr(a), a.size, _ptr(out))
    return out


def row_bytes(kv_dtype: int) -> int:
    return int(_load().oracle_row_bytes(kv_dtype))


def row_len(seq_len: int, Sq: int, t: int) -> int:
    return int(_load().oracle_row_len(seq_len, Sq, t))


def default_num_splits(max_seq_len: int, sm_count: int) -> int:
    return int(_load().oracle_default_num_splits(max_seq_len, sm_count))


# ---------------------------------------------------------------- math
def merge(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge S partial (o[512], lse) states of one (row, head)."""
    o_parts = np.ascontiguousarray(o_parts, np.float64).reshape(-1, L)
    lse_parts = np.ascontiguousarray(lse_parts, np.float64).reshape(-1)
    assert o_parts.shape[0] == lse_parts.shape[0]
    o = np.empty(L, np.float64)
    lse = np.empty(1, np.float64)
    _load().oracle_merge(_ptr(o_parts), _ptr(lse_parts), lse_parts.shape[0], _ptr(o), _ptr(lse))
    return o, float(lse[0])


def _sel_array(sel):
    if sel is None:
        return None, 0
    s = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 3))
    return s, s.shape[0]


def decode_absorbed(q, cache, kv_dtype, num_blocks, block_table, seq_lens, B, Sq, H, scale,
                    chunk=0, sel=None):
    """Route A. q: fp64 [B,Sq,H,576] or bf16 bits (uint16/int16). Returns (o_latent, lse):
    shapes [B,Sq,H,512] / [B,Sq,H] when sel is None, else [n_sel,512] / [n_sel]."""
    q = np.asarray(q)
    if q.dtype != np.float64:
        q = widen_bf16(q)
    q = np.ascontiguousarray(q).reshape(B, Sq, H, D)
    cache = np.ascontiguousarray(np.asarray(cache).view(np.uint8))
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    s, n_sel = _sel_array(sel)
    n = n_sel if s is not None else B * Sq * H
    o = np.empty((n, L), np.float64)
    lse = np.empty(n, np.float64)
    rc = _load().oracle_decode_absorbed(_ptr(q), _ptr(cache), kv_dtype, int(num_blocks), _ptr(bt),
                                        bt.shape[1], _ptr(sl), B, Sq, H, float(scale), int(chunk),
                                        _ptr(s) if s is not None else None, n_sel, _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle: block id out of range")
    if s is None:
        return o.reshape(B, Sq, H, L), lse.reshape(B, Sq, H)
    return o, lse


def decode_nonabsorbed(q_nope, q_pe, cache, kv_dtype, num_blocks, block_table, seq_lens, w_uk_t,
                       w_uv, B, Sq, H, scale, sel=None):
    """Route N. Returns (o [.,128], o_latent [.,512], lse [.]) shaped like decode_absorbed."""
    qn = _u16(q_nope).reshape(B, Sq, H, P)
    qp = _u16(q_pe).reshape(B, Sq, H, R)
    cache = np.ascontiguousarray(np.asarray(cache).view(np.uint8))
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    wk = _u16(w_uk_t)
    wv = _u16(w_uv)
    s, n_sel = _sel_array(sel)
    n = n_sel if s is not None else B * Sq * H
    o = np.empty((n, V), np.float64)
    ol = np.empty((n, L), np.float64)
    lse = np.empty(n, np.float64)
    rc = _load().oracle_decode_nonabsorbed(_ptr(qn), _ptr(qp), _ptr(cache), kv_dtype, int(num_blocks),
                                           _ptr(bt), bt.shape[1], _ptr(sl), _ptr(wk), _ptr(wv), B, Sq,
                                           H, float(scale), _ptr(s) if s is not None else None, n_sel,
                                           _ptr(o), _ptr(ol), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle: block id out of range")
    if s is None:
        return o.reshape(B, Sq, H, V), ol.reshape(B, Sq, H, L), lse.reshape(B, Sq, H)
    return o, ol, lse


def absorb_q(q_nope, q_pe, w_uk_t, T, H):
    """q_nope [T,H,128] bf16, q_pe [T,H,64] bf16, W_UK_T [H,128,512] bf16 -> q [T,H,576] fp64."""
    qn = _u16(q_nope).reshape(T, H, P)
    qp = _u16(q_pe).reshape(T, H, R)
    wk = _u16(w_uk_t)
    out = np.empty((T, H, D), np.float64)
    _load().oracle_absorb_q(_ptr(qn), H * P, P, _ptr(qp), H * R, R, _ptr(wk), T, H, _ptr(out))
    return out


def out_proj(o_latent, w_uv, T, H):
    """o_latent [T,H,512] (fp64, fp32 or bf16 bits), W_UV [H,512,128] bf16 -> o [T,H,128] fp64."""
    x = np.asarray(o_latent)
    if x.dtype in (np.uint16, np.int16):
        x = widen_bf16(x)
    x = np.ascontiguousarray(x, np.float64).reshape(T, H, L)
    wv = _u16(w_uv)
    out = np.empty((T, H, V), np.float64)
    _load().oracle_out_proj(_ptr(x), _ptr(wv), T, H, _ptr(out))
    return out


def e4m3_encode(x: float) -> int:
    """Nearest OCP E4M3 code of the binary32 value x (ties to even, saturating at 448)."""
    return int(_load().oracle_e4m3_encode(float(x)))


def cache_write(kv_c, k_pe, slot_mapping, kv_dtype, cache, num_blocks, kv_scale=0.0):
    """Write T rows [kv_c || k_pe] (bf16 bit patterns, [T, 512] and [T, 64], rows may be strided
    views with unit inner stride) into `cache` (uint8, [num_blocks, 64 * row_bytes], modified in
    place) at slot_mapping (int64, < 0 = skip). Returns the number of out-of-range slots."""
    kv_c = np.asarray(kv_c)
    k_pe = np.asarray(k_pe)
    assert kv_c.dtype == np.uint16 and k_pe.dtype == np.uint16 and cache.dtype == np.uint8
    assert kv_c.strides[-1] == 2 and k_pe.strides[-1] == 2 and cache.flags.c_contiguous
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    T = slots.shape[0]
    return int(_load().oracle_cache_write(kv_c.ctypes.data, kv_c.strides[0] // 2 if T else 0, k_pe.ctypes.data,
                                         k_pe.strides[0] // 2 if T else 0, slots.ctypes.data, T, kv_dtype,
                                         float(kv_scale), cache.ctypes.data, num_blocks))


def decode_varlen(q, cache, kv_dtype, num_blocks, block_table, seq_lens, query_start_loc, H, scale):
    """Route A over packed variable-length query rows: q fp64 or bf16 bits [total_q, H, 576],
    query_start_loc [B + 1]. Returns (o_latent [total_q, H, 512], lse [total_q, H])."""
    qsl = np.ascontiguousarray(query_start_loc, np.int32)
    B = qsl.shape[0] - 1
    q = np.asarray(q)
    if q.dtype != np.float64:
        q = widen_bf16(q)
    total_q = int(qsl[-1])
    q = np.ascontiguousarray(q).reshape(total_q, H, D)
    cache = np.ascontiguousarray(np.asarray(cache).view(np.uint8))
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    o = np.empty((total_q, H, L), np.float64)
    lse = np.empty((total_q, H), np.float64)
    rc = _load().oracle_decode_varlen(_ptr(q), _ptr(cache), kv_dtype, int(num_blocks), _ptr(bt), bt.shape[1],
                                      _ptr(sl), _ptr(qsl), B, H, float(scale), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle: block id out of range")
    return o, lse


def prefill_chunks(ctx_lens, chunk_rows):
    """The context chunk plan: int64 [n, 4] rows (chunk, request, first position, tokens)."""
    cl = np.ascontiguousarray(ctx_lens, np.int32)
    lib = _load()
    n = lib.oracle_prefill_chunks(_ptr(cl), cl.shape[0], int(chunk_rows), None)
    if n < 0:
        raise ValueError("oracle: chunk_rows must hold at least one page")
    out = np.zeros((max(n, 1), 4), np.int64)
    lib.oracle_prefill_chunks(_ptr(cl), cl.shape[0], int(chunk_rows), _ptr(out))
    return out[:n]


def prefill(q, kv_c_new, k_pe_new, cache, kv_dtype, num_blocks, block_table, ctx_lens, query_start_loc, H,
            w_uk_t, w_uv, scale, chunk_rows):
    """Prefill (compute-friendly route): q bf16 bits [total_q, H, 192], the new tokens' kv_c
    [total_q, 512] and k_pe [total_q, 64] (bf16 bits), the context in the paged cache.
    Returns (o [total_q, H, 128], lse [total_q, H]) in fp64."""
    qsl = np.ascontiguousarray(query_start_loc, np.int32)
    B = qsl.shape[0] - 1
    total_q = int(qsl[-1])
    qq = _u16(q).reshape(total_q, H, P + R)
    kc = _u16(kv_c_new).reshape(total_q, L)
    kp = _u16(k_pe_new).reshape(total_q, R)
    cache = np.ascontiguousarray(np.asarray(cache).view(np.uint8))
    bt = np.ascontiguousarray(block_table, np.int32)
    cl = np.ascontiguousarray(ctx_lens, np.int32)
    wk = _u16(w_uk_t)
    wv = _u16(w_uv)
    o = np.empty((max(total_q, 1), H, V), np.float64)
    lse = np.empty((max(total_q, 1), H), np.float64)
    rc = _load().oracle_prefill(_ptr(qq), _ptr(kc), _ptr(kp), _ptr(cache), kv_dtype, int(num_blocks), _ptr(bt),
                                bt.shape[1], _ptr(cl), _ptr(qsl), B, H, _ptr(wk), _ptr(wv), float(scale),
                                int(chunk_rows), _ptr(o), _ptr(lse))
    if rc == -2:
        raise ValueError("oracle: chunk_rows must hold at least one page")
    if rc != 0:
        raise ValueError("oracle: block id out of range")
    return o[:total_q], lse[:total_q]
