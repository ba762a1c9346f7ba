"""fp64 CPU oracle for sink GQA attention (TEST INFRASTRUCTURE).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It never imports the CUDA library and
the CUDA library never imports it.

The arithmetic lives in ``attn_sink_oracle.c`` (plain C, double precision),
written from "GPT-OSS pada Hari ke-0", section "Atensi Sink": each head's sink
logit joins the softmax over the scaled query-key products and its column is
dropped from the output.  This module only marshals numpy arrays and states the
chunking rule used for split-KV decode.

Array conventions (numpy):
  q        [total_q, Hq, D]   float32, or uint16 holding bf16 bit patterns
  k_cache, v_cache [num_pages, page_size, Hkv, D]  same dtype as q
  cu_seqlens_q [B+1] int32, kv_lens [B] int32, block_table [B, stride] int32
  sinks    [Hq] float64 (may hold -inf)
"""
import ctypes
import math
import os

import numpy as np

from . import build as _build

_LIB = None
_F32, _BF16 = 0, 1


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        lib.oracle_partials.restype = ctypes.c_int64
        lib.oracle_partials.argtypes = [
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
            ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ]
        lib.oracle_merge.restype = None
        lib.oracle_merge.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.oracle_max_threads.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def max_threads() -> int:
    """OpenMP threads the oracle uses by default."""
    return int(_lib().oracle_max_threads())


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


class Problem:
    """Holds one batch's inputs in the layout the oracle reads."""

    def __init__(self, q, k_cache, v_cache, cu_seqlens_q, kv_lens, block_table, sinks,
                 scale, causal=True):
        if q.dtype == np.float32:
            self.dtype = _F32
        elif q.dtype == np.uint16:
            self.dtype = _BF16
        else:
            raise TypeError("q must be float32 or uint16 (bf16 bits)")
        for a in (k_cache, v_cache):
            if a.dtype != q.dtype:
                raise TypeError("q, k_cache and v_cache must share a dtype")
        self.q = np.ascontiguousarray(q)
        self.k = np.ascontiguousarray(k_cache)
        self.v = np.ascontiguousarray(v_cache)
        self.cu = np.ascontiguousarray(cu_seqlens_q, dtype=np.int32)
        self.kv_lens = np.ascontiguousarray(kv_lens, dtype=np.int32)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        if bt.ndim != 2:
            raise ValueError("block_table must be 2-D")
        self.bt = bt
        self.sinks = np.ascontiguousarray(sinks, dtype=np.float64)
        self.scale = float(scale)
        self.causal = bool(causal)
        self.total_q, self.Hq, self.D = self.q.shape
        self.num_pages, self.page_size, self.Hkv, d2 = self.k.shape
        self.B = len(self.kv_lens)
        if d2 != self.D or self.cu.shape != (self.B + 1,) or self.sinks.shape != (self.Hq,):
            raise ValueError("inconsistent shapes")

    # -- row bookkeeping ---------------------------------------------------
    def all_rows(self):
        return np.arange(self.total_q * self.Hq, dtype=np.int64)

    def row_seq(self, rows):
        """Sequence index of each flat row (token * Hq + head)."""
        tok = np.asarray(rows, dtype=np.int64) // self.Hq
        return np.searchsorted(self.cu, tok, side="right") - 1

    def partials(self, rows, bounds, sink_mask, threads=0):
        """Per-row partial (o, lse) over explicit key chunks.

        bounds: int64 [n_rows, S+1] chunk boundaries in key index space.
        sink_mask: bit c set means chunk c counts the sink.
        Returns (o [n_rows, S, D] float64, lse [n_rows, S] float64, n_invalid).
        """
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        bounds = np.ascontiguousarray(bounds, dtype=np.int64)
        n, s1 = bounds.shape
        S = s1 - 1
        if n != len(rows):
            raise ValueError("bounds must have one line per row")
        o = np.zeros((n, S, self.D), dtype=np.float64)
        lse = np.zeros((n, S), dtype=np.float64)
        bad = _lib().oracle_partials(
            _ptr(self.q), _ptr(self.k), _ptr(self.v), self.dtype, _ptr(self.cu),
            _ptr(self.kv_lens), _ptr(self.bt), self.bt.shape[1], _ptr(self.sinks),
            self.B, self.Hq, self.Hkv, self.D, self.page_size, self.num_pages, self.scale,
            int(self.causal), _ptr(rows), n, _ptr(bounds), S, int(sink_mask), _ptr(o), _ptr(lse),
            int(threads))
        if bad < 0:
            raise ValueError("oracle rejected its arguments")
        return o, lse, int(bad)

    def attention(self, rows=None, threads=0):
        """Unsplit sink attention: (out [n_rows, D], lse [n_rows], n_invalid)."""
        rows = self.all_rows() if rows is None else np.asarray(rows, dtype=np.int64)
        b = self.row_seq(rows)
        bounds = np.stack([np.zeros(len(rows), np.int64), self.kv_lens[b].astype(np.int64)], 1)
        o, lse, bad = self.partials(rows, bounds, 1, threads)
        return o[:, 0, :], lse[:, 0], bad

    def split_bounds(self, rows, num_splits):
        """Key boundaries of split-KV chunk c of S for each row's sequence.

        Chunk c covers whole pages [floor(c*P/S), floor((c+1)*P/S)) where
        P = ceil(kv_len / page_size), clipped to kv_len; chunk 0 holds key 0.
        """
        b = self.row_seq(rows)
        kv = self.kv_lens[b].astype(np.int64)
        P = (kv + self.page_size - 1) // self.page_size
        c = np.arange(num_splits + 1, dtype=np.int64)
        pages = (c[None, :] * P[:, None]) // num_splits
        return np.minimum(pages * self.page_size, kv[:, None])

    def attention_split(self, rows=None, num_splits=1, threads=0):
        """Split-KV sink attention: page-aligned chunks, sink in chunk 0, LSE merge."""
        rows = self.all_rows() if rows is None else np.asarray(rows, dtype=np.int64)
        bounds = self.split_bounds(rows, num_splits)
        o, lse, bad = self.partials(rows, bounds, 1, threads)
        out, l = merge(o, lse)
        return out, l, bad


def merge(o_parts, lse_parts):
    """LSE merge of partial states: o [n, S, D], lse [n, S] -> (out [n, D], lse [n])."""
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, S, D = o_parts.shape
    out = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    _lib().oracle_merge(_ptr(o_parts), _ptr(lse_parts), n, S, D, _ptr(out), _ptr(lse))
    return out, lse


def default_scale(head_dim: int) -> float:
    """Softmax scale 1/sqrt(head_dim) used by every configuration."""
    return 1.0 / math.sqrt(head_dim)


__all__ = ["Problem", "merge", "max_threads", "default_scale"]
os.environ.setdefault("OMP_WAIT_POLICY", "PASSIVE")
