"""Python binding of ``libattn_sink.so``: sink GQA attention for GB300.

Thin argument marshalling over the C ABI in ``include/attn_sink.h``.  Every
step of the computation runs in the library's CUDA kernels; this module only
checks tensors, allocates outputs/workspace with torch when the caller does
not pass them, and forwards device pointers plus the current torch stream.
There is no CPU fallback: if the library is missing, every call raises.

    import gqa_attention_sinks_gb300 as gas
    out, lse = gas.decode(q, k_cache, v_cache, kv_lens, block_table, sinks)
    out, lse = gas.prefill(q, k_cache, v_cache, cu_seqlens_q, kv_lens, block_table,
                           sinks, max_q_len=4096)
"""
import ctypes
import math
import os

import torch

__all__ = ["load", "prefill", "mixed", "decode", "decode_append", "merge", "decode_workspace_size",
           "prefill_workspace_size", "mixed_workspace_size", "status_string",
           "set_wait_limit_ns", "AttnSinkError", "LIB_PATH", "FLAG_BAD_PAGE", "FLAG_TIMEOUT",
           "SPLIT_PERSISTENT"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn_sink.so")
FLAG_BAD_PAGE, FLAG_TIMEOUT = 1, 2
SPLIT_PERSISTENT = -1
_BF16, _FP32 = 0, 1
_LIB = None

_vp, _i32, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t

# C-ABI signatures (argument types, return type), mirroring include/attn_sink.h.
SIGNATURES = {
    "attn_sink_prefill": ([_vp] * 10 + [_i32] * 8 + [_f32, _i32, _i32, _vp, _vp, _sz, _vp], _i32),
    "attn_sink_prefill_workspace_size": ([_i32] * 4, _sz),
    "attn_sink_mixed": ([_vp] * 6 + [_i32, _vp, _vp, _vp] + [_i32] * 9 + [_f32, _i32, _i32, _vp,
                                                                         _vp, _sz, _vp], _i32),
    "attn_sink_mixed_workspace_size": ([_i32] * 6, _sz),
    "attn_sink_decode": ([_vp] * 5 + [_i32, _vp, _vp, _vp] + [_i32] * 6 + [_f32, _i32, _i32, _vp,
                                                                         _vp, _sz, _vp], _i32),
    "attn_sink_decode_append": ([_vp] * 7 + [_i32, _vp, _vp, _vp] + [_i32] * 6 +
                                [_f32, _i32, _i32, _vp, _vp, _sz, _vp], _i32),
    "attn_sink_decode_workspace_size": ([_i32] * 7, _sz),
    "attn_sink_decode_static_scratch": ([_vp] * 5 + [_i32, _vp, _vp, _vp] + [_i32] * 6 +
                                        [_f32, _i32, _i32, _vp, _vp], _i32),
    "attn_sink_merge": ([_vp, _vp, _i32, _i32, _i32, _vp, _vp, _i32, _vp], _i32),
    "attn_sink_status_string": ([_i32], ctypes.c_char_p),
    "attn_sink_set_wait_limit_ns": ([ctypes.c_uint64], ctypes.c_uint64),
}


class AttnSinkError(RuntimeError):
    """A non-OK status returned by the C ABI."""

    def __init__(self, fn, status):
        super().__init__("%s failed: %s (status %d)" % (fn, status_string(status), status))
        self.status = status


def load(path=None):
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError("%s is missing: build it with gqa_attention_sinks_gb300.build.build()" % p)
        lib = ctypes.CDLL(p)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _LIB = lib
    return _LIB


def status_string(status):
    return load().attn_sink_status_string(int(status)).decode()


def set_wait_limit_ns(ns):
    """Test hook: limit of every pipeline wait for later calls (0 restores 1 s).
    Returns the previous limit."""
    return int(load().attn_sink_set_wait_limit_ns(int(ns)))


def _check(fn, status):
    if status != 0:
        raise AttnSinkError(fn, status)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return _BF16
    if t.dtype == torch.float32:
        return _FP32
    raise TypeError("q/k/v must be bfloat16 or float32, got %s" % t.dtype)


def _dev(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def decode_workspace_size(B, Hq, Hkv, D, block_table_stride, page_size, num_splits=0):
    """Bytes of scratch ``decode`` needs for these arguments."""
    return int(load().attn_sink_decode_workspace_size(B, Hq, Hkv, D, block_table_stride,
                                                      page_size, num_splits))


def prefill_workspace_size(B, Hq, D, max_q_len):
    """Bytes of scratch ``prefill`` needs for these arguments."""
    return int(load().attn_sink_prefill_workspace_size(B, Hq, D, max_q_len))


def decode(q, k_cache, v_cache, kv_lens, block_table, sinks, *, scale=None, num_splits=0,
           out=None, lse=None, workspace=None, err_flag=None, stream=None):
    """Paged decode with sinks.  q [B, Hq, D]; caches [pages, page_size, Hkv, D].

    num_splits: 0 automatic chunks, 1 no split, S > 1 that many page-aligned
    chunks, SPLIT_PERSISTENT (-1) persistent CTAs with equal shares of all keys.
    Returns (out [B, Hq, D] in q's dtype, lse [B, Hq] fp32).
    """
    lib = load()
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _dev(t, name, q.dtype)
    _dev(kv_lens, "kv_lens", torch.int32)
    _dev(block_table, "block_table", torch.int32)
    _dev(sinks, "sinks", torch.float32)
    B, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    bt_stride = block_table.shape[1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _dev(out, "out", q.dtype)
    _dev(lse, "lse", torch.float32)
    # (for fp32, num_splits=0 means one chunk; the size below then over-covers)
    need = decode_workspace_size(B, Hq, Hkv, D, bt_stride, page_size, num_splits)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.attn_sink_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(kv_lens),
                              _ptr(block_table), bt_stride, _ptr(sinks), _ptr(out), _ptr(lse),
                              B, Hq, Hkv, D, page_size, num_pages, scale, int(num_splits), dt,
                              _ptr(err_flag), _ptr(workspace), ws_bytes, _stream(stream))
    _check("attn_sink_decode", st)
    return out, lse


def decode_append(q, k_new, v_new, k_cache, v_cache, kv_lens, block_table, sinks, *, scale=None,
                  num_splits=0, out=None, lse=None, workspace=None, err_flag=None, stream=None):
    """One decode step that first writes k_new / v_new [B, Hkv, D] into the cache slot
    of position kv_lens[b] - 1, then attends over keys 0..kv_lens[b]-1 (the caches are
    updated in place).  Returns (out, lse) like ``decode``."""
    lib = load()
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache),
                    ("v_cache", v_cache)):
        _dev(t, name, q.dtype)
    _dev(kv_lens, "kv_lens", torch.int32)
    _dev(block_table, "block_table", torch.int32)
    _dev(sinks, "sinks", torch.float32)
    B, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D):
        raise ValueError("k_new / v_new must be [B, Hkv, D] = %s" % ((B, Hkv, D),))
    bt_stride = block_table.shape[1]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _dev(out, "out", q.dtype)
    _dev(lse, "lse", torch.float32)
    need = decode_workspace_size(B, Hq, Hkv, D, bt_stride, page_size, num_splits)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.attn_sink_decode_append(_ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(kv_lens), _ptr(block_table), bt_stride, _ptr(sinks),
                                     _ptr(out), _ptr(lse), B, Hq, Hkv, D, page_size, num_pages,
                                     scale, int(num_splits), dt, _ptr(err_flag), _ptr(workspace),
                                     ws_bytes, _stream(stream))
    _check("attn_sink_decode_append", st)
    return out, lse


def prefill(q, k_cache, v_cache, cu_seqlens_q, kv_lens, block_table, sinks, *, max_q_len,
            scale=None, causal=True, out=None, lse=None, workspace=None, err_flag=None,
            stream=None):
    """Ragged causal prefill with sinks.  q [total_q, Hq, D].

    max_q_len is a host int, an upper bound of every sequence's q_len (the
    caller knows it; reading it from cu_seqlens_q would synchronise).
    Returns (out [total_q, Hq, D] in q's dtype, lse [total_q, Hq] fp32).
    """
    lib = load()
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _dev(t, name, q.dtype)
    _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _dev(kv_lens, "kv_lens", torch.int32)
    _dev(block_table, "block_table", torch.int32)
    _dev(sinks, "sinks", torch.float32)
    total_q, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    B = kv_lens.shape[0]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    _dev(out, "out", q.dtype)
    _dev(lse, "lse", torch.float32)
    need = prefill_workspace_size(B, Hq, D, int(max_q_len))
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.attn_sink_prefill(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_q),
                               _ptr(kv_lens), _ptr(block_table), block_table.shape[1], _ptr(sinks),
                               _ptr(out), _ptr(lse), B, total_q, int(max_q_len), Hq, Hkv, D,
                               page_size, num_pages, scale, int(bool(causal)), dt, _ptr(err_flag),
                               _ptr(workspace), ws_bytes, _stream(stream))
    _check("attn_sink_prefill", st)
    return out, lse


def mixed_workspace_size(num_decode, Hq, Hkv, D, block_table_stride, page_size):
    """Bytes of scratch ``mixed`` needs for these arguments."""
    return int(load().attn_sink_mixed_workspace_size(num_decode, Hq, Hkv, D, block_table_stride,
                                                     page_size))


def mixed(q, k_cache, v_cache, cu_seqlens_q, kv_lens, block_table, sinks, *, num_decode,
          max_q_len, scale=None, causal=True, out=None, lse=None, workspace=None, err_flag=None,
          stream=None):
    """One launch for a ragged batch whose first num_decode sequences are
    single-query decode rows and whose others are prefill segments (q_len up
    to max_q_len).  q [total_q, Hq, D].  Returns (out, lse) like ``prefill``."""
    lib = load()
    dt = _dtype_code(q)
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _dev(t, name, q.dtype)
    _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _dev(kv_lens, "kv_lens", torch.int32)
    _dev(block_table, "block_table", torch.int32)
    _dev(sinks, "sinks", torch.float32)
    total_q, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    B = kv_lens.shape[0]
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((total_q, Hq), dtype=torch.float32, device=q.device)
    _dev(out, "out", q.dtype)
    _dev(lse, "lse", torch.float32)
    need = mixed_workspace_size(int(num_decode), Hq, Hkv, D, block_table.shape[1], page_size)
    if workspace is None and need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.attn_sink_mixed(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_q),
                             _ptr(kv_lens), _ptr(block_table), block_table.shape[1], _ptr(sinks),
                             _ptr(out), _ptr(lse), B, int(num_decode), total_q, int(max_q_len), Hq,
                             Hkv, D, page_size, num_pages, scale, int(bool(causal)), dt,
                             _ptr(err_flag), _ptr(workspace), ws_bytes, _stream(stream))
    _check("attn_sink_mixed", st)
    return out, lse


def merge(o_parts, lse_parts, *, out_dtype=torch.bfloat16, out=None, lse=None, stream=None):
    """LSE merge of partial states: o_parts [rows, S, D] fp32, lse_parts [rows, S] fp32."""
    lib = load()
    _dev(o_parts, "o_parts", torch.float32)
    _dev(lse_parts, "lse_parts", torch.float32)
    rows, S, D = o_parts.shape
    if out is None:
        out = torch.empty((rows, D), dtype=out_dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty(rows, dtype=torch.float32, device=o_parts.device)
    dt = _dtype_code(out)
    st = lib.attn_sink_merge(_ptr(o_parts), _ptr(lse_parts), rows, S, D, _ptr(out), _ptr(lse), dt,
                             _stream(stream))
    _check("attn_sink_merge", st)
    return out, lse
