"""Python binding of the GB300 MLA latent-KV decode library (libmla_latent_kv.so).

Argument marshalling only: every step of absorption, decode, split merge and output projection
runs in the library's CUDA kernels. PyTorch supplies device memory and the current stream. If the
native library has not been built, importing works but every call raises -- there is no
fallback path. Build it with ``python -m mla_latent_kv_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libmla_latent_kv.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "mla_latent_kv.h")

KV_BF16, KV_FP8 = 0, 1
DT_F32, DT_BF16 = 0, 1
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE_TOO_SMALL, ERR_CUDA = range(5)
DEV_BAD_BLOCK_ID, DEV_SEQ_TOO_LONG, DEV_WAIT_TIMEOUT = 0x1, 0x2, 0x4
L, R, D, P, V, PAGE, MAX_HEADS = 512, 64, 576, 128, 128, 64, 128

_lock = threading.Lock()
_lib = None


class MlaError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"{status_string(status)}: {detail}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load the native library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"native library missing: {LIB_PATH} "
                               "(build it with `python -m mla_latent_kv_gb300.build`)")
        l = ctypes.CDLL(LIB_PATH)
        i32, i64, vp, f32, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_size_t
        l.mla_status_string.restype = ctypes.c_char_p
        l.mla_status_string.argtypes = [i32]
        l.mla_last_error_detail.restype = ctypes.c_char_p
        l.mla_last_error_detail.argtypes = []
        l.mla_selftest_wait_timeout.restype = i32
        l.mla_selftest_wait_timeout.argtypes = [vp, vp, vp]
        l.mla_selftest_e4m3_widen.restype = i32
        l.mla_selftest_e4m3_widen.argtypes = [vp, vp]
        l.mla_kv_row_bytes.restype = i64
        l.mla_kv_row_bytes.argtypes = [i32]
        l.mla_default_num_splits.restype = i32
        l.mla_default_num_splits.argtypes = [i32, i32]
        l.mla_resolve_num_splits.restype = i32
        l.mla_resolve_num_splits.argtypes = [i32, i32, i32, i32, i32]
        l.mla_decode_workspace_bytes.restype = sz
        l.mla_decode_workspace_bytes.argtypes = [i32, i32, i32, i32]
        l.mla_decode_workspace_bytes_kv.restype = sz
        l.mla_decode_workspace_bytes_kv.argtypes = [i32, i32, i32, i32, i32, i32]
        l.mla_absorb_q.restype = i32
        l.mla_absorb_q.argtypes = [vp, i64, i64, vp, i64, i64, vp, vp, i32, i32, vp]
        l.mla_decode.restype = i32
        l.mla_decode.argtypes = [vp, vp, i32, i64, vp, i32, vp, i32, i32, i32, i32, f32, i32, vp, sz,
                                 vp, i32, vp, vp, vp]
        l.mla_decode_noalloc_max_workspace_bytes.restype = sz
        l.mla_decode_noalloc_max_workspace_bytes.argtypes = []
        l.mla_decode_noalloc.restype = i32
        l.mla_decode_noalloc.argtypes = [vp, vp, i32, i64, vp, i32, vp, i32, i32, i32, i32, f32, i32, vp, i32,
                                         vp, vp, vp]
        l.mla_decode_varlen_workspace_bytes.restype = sz
        l.mla_decode_varlen_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
        l.mla_decode_varlen.restype = i32
        l.mla_decode_varlen.argtypes = [vp, vp, i32, i64, vp, i32, vp, vp, i32, i32, i32, i32, f32, i32, vp, sz,
                                        vp, i32, vp, vp, vp]
        l.mla_cache_write.restype = i32
        l.mla_cache_write.argtypes = [vp, i64, vp, i64, vp, i32, vp, i32, i64, f32, vp, vp]
        l.mla_out_proj.restype = i32
        l.mla_out_proj.argtypes = [vp, i32, vp, vp, i32, i32, i32, vp]
        l.mla_prefill_workspace_bytes.restype = sz
        l.mla_prefill_workspace_bytes.argtypes = [i32, i32, i32, i64]
        l.mla_prefill_chunk_plan.restype = i64
        l.mla_prefill_chunk_plan.argtypes = [vp, i32, i64, vp, i64]
        l.mla_prefill.argtypes = [vp, vp, i64, vp, i64, vp, i32, i64, vp, i32, vp, vp, vp, vp, i32, i32, vp, vp,
                                  f32, i64, vp, sz, vp, vp, vp, vp]
        _lib = l
        return l


def declared_functions() -> list[str]:
    """Names of the functions include/mla_latent_kv.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\*]+\s*\*?\s*(mla_\w+)\s*\(", text, re.M)))


def status_string(status: int) -> str:
    return lib().mla_status_string(int(status)).decode()


def _check(status: int):
    if status != OK:
        raise MlaError(status, lib().mla_last_error_detail().decode())


def row_bytes(kv_dtype: int) -> int:
    return int(lib().mla_kv_row_bytes(kv_dtype))


def default_num_splits(max_seq_len: int, sm_count: int) -> int:
    return int(lib().mla_default_num_splits(max_seq_len, sm_count))


def resolve_num_splits(num_splits: int, B: int, Sq: int, H: int, max_seq_len: int) -> int:
    s = int(lib().mla_resolve_num_splits(num_splits, B, Sq, H, max_seq_len))
    if s < 1 and s != -2:  # -2: per-row schedule built on the device
        raise MlaError(ERR_INVALID_ARG, "could not resolve num_splits")
    return s


def workspace_bytes(B: int, Sq: int, H: int, num_splits: int, kv_dtype: int = KV_BF16, max_seq_len: int = 0) -> int:
    """Decode workspace bytes; with the default kv_dtype this is the split-KV part alone."""
    if kv_dtype == KV_BF16:
        return int(lib().mla_decode_workspace_bytes(B, Sq, H, num_splits))
    return int(lib().mla_decode_workspace_bytes_kv(kv_dtype, B, Sq, H, num_splits, max_seq_len))


# ----------------------------------------------------------------------------- torch front end
def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def absorb_q(q_nope, q_pe, w_uk_t, out=None, stream=None):
    """q_nope [T,H,128] bf16 (any token/head strides, unit stride inside a head), q_pe [T,H,64]
    bf16 or None, W_UK_T [H,128,512] bf16 -> q [T,H,576] bf16."""
    import torch
    T, H = q_nope.shape[0], q_nope.shape[1]
    assert q_nope.stride(2) == 1 and w_uk_t.is_contiguous()
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.bfloat16, device=q_nope.device)
    spt, sph = (q_pe.stride(0), q_pe.stride(1)) if q_pe is not None else (0, 0)
    _check(lib().mla_absorb_q(_p(q_nope), q_nope.stride(0), q_nope.stride(1), _p(q_pe), spt, sph,
                              _p(w_uk_t), _p(out), T, H, _stream(stream)))
    return out


def _dt_code(buf, dt):
    """The output dtype code: `dt` when given, else the given buffer's dtype, else fp32."""
    import torch
    if dt is not None:
        return dt
    if buf is not None and buf.dtype == torch.bfloat16:
        return DT_BF16
    return DT_F32


def _out_buf(buf, shape, dt, device):
    """An output buffer of dtype code `dt` holding `shape`: made when not given; a given one must be
    contiguous, of that dtype and at least that large, since the kernels write through its pointer."""
    import torch
    tdt = torch.float32 if dt == DT_F32 else torch.bfloat16
    if buf is None:
        return torch.empty(shape, dtype=tdt, device=device)
    n = 1
    for d in shape:
        n *= int(d)
    if buf.dtype != tdt or buf.numel() < n or not buf.is_contiguous():
        raise ValueError(f"output buffer must be a contiguous {tdt} of at least {n} elements, "
                         f"got {buf.dtype} with {buf.numel()} (contiguous={buf.is_contiguous()})")
    return buf


def decode(q, kv_cache, block_table, seq_lens, max_seq_len, scale, kv_dtype=KV_BF16, num_splits=0,
           workspace=None, o_latent=None, o_dtype=None, lse=None, dev_status=None, stream=None,
           num_blocks=None):
    """q [B,Sq,H,576] bf16, kv_cache [num_blocks, 64*row_bytes] uint8 (or a bf16 view), block_table
    [B,max_blocks] int32, seq_lens [B] int32 -> (o_latent [B,Sq,H,512], lse [B,Sq,H])."""
    import torch
    B, Sq, H = q.shape[0], q.shape[1], q.shape[2]
    dev = q.device
    if num_blocks is None:
        num_blocks = kv_cache.numel() * kv_cache.element_size() // (PAGE * row_bytes(kv_dtype))
    S = resolve_num_splits(num_splits, B, Sq, H, max_seq_len)
    need = workspace_bytes(B, Sq, H, S, kv_dtype, max_seq_len)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    o_dtype = _dt_code(o_latent, o_dtype)
    o_latent = _out_buf(o_latent, (B, Sq, H, L), o_dtype, dev)
    lse = _out_buf(lse, (B, Sq, H), DT_F32, dev)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().mla_decode(_p(q), _p(kv_cache), kv_dtype, int(num_blocks), _p(block_table),
                            block_table.shape[1], _p(seq_lens), int(max_seq_len), B, Sq, H, float(scale),
                            int(S), _p(workspace), ws_bytes, _p(o_latent), o_dtype, _p(lse), _p(dev_status),
                            _stream(stream)))
    return o_latent, lse


def selftest_wait_timeout(dev_status, out, stream=None):
    """Run the bounded-wait self-test: dev_status int32 [1] and out int32 [2] on the device; after a
    synchronise dev_status has MLA_DEV_WAIT_TIMEOUT set, out[0] is the wait in ms, out[1] is 0."""
    _check(lib().mla_selftest_wait_timeout(_p(dev_status), _p(out), _stream(stream)))


def selftest_e4m3_widen(out, stream=None):
    """Run the FP8 widening self-test: out uint16/int16 [256] on the device receives, after a
    synchronise, the bf16 bits the FP8 decode kernel produces for e4m3 codes 0..255."""
    _check(lib().mla_selftest_e4m3_widen(_p(out), _stream(stream)))


def noalloc_max_workspace_bytes() -> int:
    return int(lib().mla_decode_noalloc_max_workspace_bytes())


def decode_noalloc(q, kv_cache, block_table, seq_lens, max_seq_len, scale, kv_dtype=KV_BF16, num_splits=0,
                   o_latent=None, o_dtype=None, lse=None, dev_status=None, stream=None, num_blocks=None):
    """decode() through mla_decode_noalloc: the split-KV scratch is the library's own fixed device
    array, so no workspace is passed (outputs are still made here when not given)."""
    import torch
    B, Sq, H = q.shape[0], q.shape[1], q.shape[2]
    dev = q.device
    if num_blocks is None:
        num_blocks = kv_cache.numel() * kv_cache.element_size() // (PAGE * row_bytes(kv_dtype))
    o_dtype = _dt_code(o_latent, o_dtype)
    o_latent = _out_buf(o_latent, (B, Sq, H, L), o_dtype, dev)
    lse = _out_buf(lse, (B, Sq, H), DT_F32, dev)
    _check(lib().mla_decode_noalloc(_p(q), _p(kv_cache), kv_dtype, int(num_blocks), _p(block_table),
                                    block_table.shape[1], _p(seq_lens), int(max_seq_len), B, Sq, H, float(scale),
                                    int(num_splits), _p(o_latent), o_dtype, _p(lse), _p(dev_status),
                                    _stream(stream)))
    return o_latent, lse


def decode_varlen(q, kv_cache, block_table, seq_lens, query_start_loc, max_seq_len, scale, kv_dtype=KV_BF16,
                  num_splits=0, workspace=None, o_latent=None, o_dtype=None, lse=None, dev_status=None, stream=None,
                  num_blocks=None):
    """q [total_q, H, 576] bf16 packed by query_start_loc [B + 1] int32 (device) ->
    (o_latent [total_q, H, 512], lse [total_q, H])."""
    import torch
    total_q, H = q.shape[0], q.shape[1]
    B = int(query_start_loc.shape[0]) - 1
    dev = q.device
    if num_blocks is None:
        num_blocks = kv_cache.numel() * kv_cache.element_size() // (PAGE * row_bytes(kv_dtype))
    S = resolve_num_splits(num_splits, max(total_q, 1), 1, H, max_seq_len)
    need = int(lib().mla_decode_varlen_workspace_bytes(kv_dtype, B, total_q, H, S, max_seq_len))
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    o_dtype = _dt_code(o_latent, o_dtype)
    o_latent = _out_buf(o_latent, (total_q, H, L), o_dtype, dev)
    lse = _out_buf(lse, (total_q, H), DT_F32, dev)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().mla_decode_varlen(_p(q), _p(kv_cache), kv_dtype, int(num_blocks), _p(block_table),
                                   block_table.shape[1], _p(seq_lens), _p(query_start_loc), int(max_seq_len), B,
                                   total_q, H, float(scale), int(S), _p(workspace), ws_bytes, _p(o_latent), o_dtype,
                                   _p(lse), _p(dev_status), _stream(stream)))
    return o_latent, lse


def cache_write(kv_c, k_pe, slot_mapping, kv_cache, kv_dtype=KV_BF16, kv_scale=0.0, dev_status=None, stream=None,
                num_blocks=None):
    """kv_c [T, 512] bf16 and k_pe [T, 64] bf16 (rows may be strided, unit inner stride),
    slot_mapping [T] int64 (< 0 = padding) -> rows written into kv_cache in place."""
    T = int(slot_mapping.shape[0])
    if num_blocks is None:
        num_blocks = kv_cache.numel() * kv_cache.element_size() // (PAGE * row_bytes(kv_dtype))
    _check(lib().mla_cache_write(_p(kv_c), kv_c.stride(0) if T else L, _p(k_pe), k_pe.stride(0) if T else R,
                                 _p(slot_mapping), T, _p(kv_cache), kv_dtype, int(num_blocks), float(kv_scale),
                                 _p(dev_status), _stream(stream)))
    return kv_cache


def out_proj(o_latent, w_uv, out=None, out_dtype=None, stream=None):
    """o_latent [T,H,512] fp32/bf16, W_UV [H,512,128] bf16 -> o [T,H,128] (fp32 unless out_dtype or
    a given `out` says bf16)."""
    import torch
    T, H = o_latent.shape[0], o_latent.shape[1]
    if o_latent.dtype not in (torch.float32, torch.bfloat16) or not o_latent.is_contiguous():
        raise ValueError(f"o_latent must be a contiguous fp32 or bf16 tensor, got {o_latent.dtype}")
    in_dtype = DT_F32 if o_latent.dtype == torch.float32 else DT_BF16
    out_dtype = _dt_code(out, out_dtype)
    out = _out_buf(out, (T, H, V), out_dtype, o_latent.device)
    _check(lib().mla_out_proj(_p(o_latent), in_dtype, _p(w_uv), _p(out), out_dtype, T, H, _stream(stream)))
    return out


def prefill_workspace_bytes(B: int, total_q: int, H: int, chunk_rows: int) -> int:
    return int(lib().mla_prefill_workspace_bytes(B, total_q, H, int(chunk_rows)))


def prefill_chunk_plan(ctx_lens, chunk_rows):
    """The context chunk plan for host context lengths: a list of (chunk, request, first
    position, tokens)."""
    import numpy as np
    cl = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    n = int(lib().mla_prefill_chunk_plan(cl.ctypes.data, cl.shape[0], int(chunk_rows), None, 0))
    if n < 0:
        raise MlaError(ERR_INVALID_ARG, "chunk_rows must hold at least one page")
    out = np.zeros((max(n, 1), 4), np.int64)
    lib().mla_prefill_chunk_plan(cl.ctypes.data, cl.shape[0], int(chunk_rows), out.ctypes.data, n)
    return out[:n]


def prefill(q, kv_c, k_pe, kv_cache, block_table, ctx_lens, query_start_loc, w_uk_t, w_uv, scale,
            kv_dtype=KV_BF16, chunk_rows=None, workspace=None, o=None, lse=None, dev_status=None, stream=None,
            num_blocks=None, ctx_lens_host=None, query_start_loc_host=None):
    """Prefill through the compute-friendly route. q [total_q, H, 192] bf16 (q_nope || q_pe),
    kv_c [total_q, 512] / k_pe [total_q, 64] bf16 (the new tokens' rows, row-strided allowed),
    ctx_lens [B] and query_start_loc [B + 1] int32 device tensors (read once on the host for the
    launch plan, unless host copies are passed as ctx_lens_host / query_start_loc_host int32 CPU
    tensors) -> (o [total_q, H, 128] fp32, lse [total_q, H] fp32)."""
    import torch
    total_q, H = q.shape[0], q.shape[1]
    B = int(query_start_loc.shape[0]) - 1
    dev = q.device
    ctx_host = ctx_lens.to("cpu", torch.int32).contiguous() if ctx_lens_host is None else ctx_lens_host
    qsl_host = query_start_loc.to("cpu", torch.int32).contiguous() if query_start_loc_host is None \
        else query_start_loc_host
    if num_blocks is None:
        num_blocks = kv_cache.numel() * kv_cache.element_size() // (PAGE * row_bytes(kv_dtype))
    if chunk_rows is None:  # the page's 64k-row budget, no larger than this batch's context needs
        chunk_rows = min(65536, max(PAGE, int(ctx_host.sum())))
    need = prefill_workspace_bytes(B, total_q, H, chunk_rows)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    if o is None:
        o = torch.empty((total_q, H, V), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((total_q, H), dtype=torch.float32, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().mla_prefill(_p(q), _p(kv_c), kv_c.stride(0) if total_q else L, _p(k_pe),
                             k_pe.stride(0) if total_q else R, _p(kv_cache), kv_dtype, int(num_blocks),
                             _p(block_table), block_table.shape[1], _p(ctx_lens), _p(query_start_loc),
                             ctypes.c_void_p(ctx_host.data_ptr()), ctypes.c_void_p(qsl_host.data_ptr()), B, H,
                             _p(w_uk_t), _p(w_uv), float(scale), int(chunk_rows), _p(workspace), ws_bytes, _p(o),
                             _p(lse), _p(dev_status), _stream(stream)))
    return o, lse
