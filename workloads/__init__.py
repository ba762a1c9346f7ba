"""Seeded synthetic inputs for sink GQA attention (shared by tests and bench).

This module draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path and the CPU oracle consume what it
returns, so neither depends on the other.

Every batch is a paged KV pool plus a ragged query batch:
  q            [total_q, Hq, D]          bf16 bit patterns (uint16) or float32
  k_cache/v_cache [num_pages, page_size, Hkv, D]  same dtype
  cu_seqlens_q [B+1] int32, kv_lens [B] int32
  block_table  [B, max_pages] int32      unused entries are -1
  sinks        [Hq] float32 (may hold -inf)

Pool recipe: exactly the pages the sequences need plus 10% spare pages; the
physical page of every logical page comes from a seeded permutation of the
pool; spare pages and the unused slots of each sequence's last page are filled
with NaN, so a kernel that reads past kv_len or through a stale table entry
produces NaN instead of a plausible number.
"""
from dataclasses import dataclass, field
import math

import numpy as np

BF16, FP32 = "bf16", "fp32"
_CHUNK = 1 << 24


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    xf, of = x.reshape(-1), out.reshape(-1)
    for s in range(0, xf.size, _CHUNK):
        u = xf[s:s + _CHUNK].view(np.uint32)
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
        r = r.astype(np.uint16)
        r[np.isnan(xf[s:s + _CHUNK])] = 0x7FC0
        of[s:s + _CHUNK] = r
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normals(rng, n, std=1.0):
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        rng.standard_normal(e - s, dtype=np.float32, out=out[s:e])
    if std != 1.0:
        out *= np.float32(std)
    return out


@dataclass
class Batch:
    """One ragged batch over a paged KV pool (host arrays)."""
    dtype: str
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    cu_seqlens_q: np.ndarray
    kv_lens: np.ndarray
    block_table: np.ndarray
    sinks: np.ndarray
    scale: float
    causal: bool = True
    meta: dict = field(default_factory=dict)

    @property
    def B(self):
        return len(self.kv_lens)

    @property
    def Hq(self):
        return self.q.shape[1]

    @property
    def D(self):
        return self.q.shape[2]

    @property
    def Hkv(self):
        return self.k_cache.shape[2]

    @property
    def page_size(self):
        return self.k_cache.shape[1]

    @property
    def num_pages(self):
        return self.k_cache.shape[0]

    @property
    def total_q(self):
        return self.q.shape[0]

    @property
    def q_lens(self):
        return np.diff(self.cu_seqlens_q)

    @property
    def max_q_len(self):
        return int(self.q_lens.max()) if self.B else 0

    def kv_tokens(self):
        return int(self.kv_lens.astype(np.int64).sum())


@dataclass
class Pool:
    """A paged KV pool shared by one or more batches."""
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_table: np.ndarray     # [num_seqs, max_pages]
    kv_lens: np.ndarray


def make_pool(rng, kv_lens, Hkv, D, page_size=16, dtype=BF16, spare_frac=0.10,
              outlier_frac=0.0, outlier_scale=20.0, shuffle=True, fill_len=None):
    """Allocate and fill a paged pool for sequences of the given KV lengths.

    fill_len (optional, per sequence, >= kv_len) fills that many keys, so a test
    can pre-place tokens that later steps append; pages are allocated for it.
    """
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    fill = kv_lens if fill_len is None else np.asarray(fill_len, dtype=np.int64)
    pages = (fill + page_size - 1) // page_size
    n_used = int(pages.sum())
    pool_pages = n_used + max(1, int(math.ceil(spare_frac * n_used)))
    perm = rng.permutation(pool_pages) if shuffle else np.arange(pool_pages)
    max_pages = max(1, int(pages.max()) if len(pages) else 1)
    bt = np.full((len(kv_lens), max_pages), -1, dtype=np.int32)
    cursor = 0
    for b, p in enumerate(pages):
        bt[b, :p] = perm[cursor:cursor + p]
        cursor += p

    row_elems = Hkv * D
    tokens = int(fill.sum())
    # flat pool row (physical page * page_size + slot) for every filled key
    seq_of = np.repeat(np.arange(len(fill)), fill)
    starts = np.concatenate([[0], np.cumsum(fill)[:-1]]).astype(np.int64)
    j = np.arange(tokens, dtype=np.int64) - starts[seq_of]
    dest = bt[seq_of, j // page_size].astype(np.int64) * page_size + j % page_size

    caches = []
    for which in ("k", "v"):
        vals = _normals(rng, tokens * row_elems).reshape(tokens, Hkv, D)
        if which == "k" and outlier_frac > 0:
            hit = rng.random((tokens, Hkv)) < outlier_frac
            vals[hit] *= np.float32(outlier_scale)
        if dtype == BF16:
            cache = np.full((pool_pages * page_size, Hkv, D), 0x7FC0, dtype=np.uint16)
            cache[dest] = to_bf16_bits(vals)
        else:
            cache = np.full((pool_pages * page_size, Hkv, D), np.nan, dtype=np.float32)
            cache[dest] = vals
        caches.append(cache.reshape(pool_pages, page_size, Hkv, D))
        del vals
    return Pool(caches[0], caches[1], bt, kv_lens.astype(np.int32))


def make_queries(rng, total_q, Hq, D, dtype=BF16):
    q = _normals(rng, total_q * Hq * D).reshape(total_q, Hq, D)
    return to_bf16_bits(q) if dtype == BF16 else q


def sinks_normal(rng, Hq, std):
    return (rng.standard_normal(Hq) * std).astype(np.float32)


def sinks_choice(rng, Hq, values=(-math.inf, -4.0, 0.0, 4.0, 8.0)):
    return np.asarray(values, dtype=np.float32)[rng.integers(0, len(values), Hq)]


def batch_from_pool(pool, seqs, q_lens, q, sinks, causal=True, dtype=BF16, meta=None):
    """Query batch over a subset of a pool's sequences (they keep their pages)."""
    seqs = np.asarray(seqs)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    bt = np.ascontiguousarray(pool.block_table[seqs])
    return Batch(dtype, q, pool.k_cache, pool.v_cache, cu, pool.kv_lens[seqs].copy(), bt,
                 sinks, 1.0 / math.sqrt(q.shape[2]), causal, dict(meta or {}))


# ---------------------------------------------------------------------------
# The workloads.  Seeds are 20260000 + workload index.
# ---------------------------------------------------------------------------

def tiny_prefill_decode(seed=20260001, num_seqs=2, Hq=8, Hkv=2, D=64, q_len=16, kv_len=64,
                        decode_steps=4, page_size=16):
    """Tiny fp32 case: causal prefill of q_len over kv_len, then decode steps.

    Pages are allocated for kv_len + decode_steps keys; the keys that the
    decode steps append are returned separately and their slots start as NaN.
    Returns dict(prefill=Batch, steps=[dict(q, new_k, new_v, kv_lens)]).
    """
    rng = np.random.default_rng(seed)
    total = kv_len + decode_steps
    pool = make_pool(rng, [kv_len] * num_seqs, Hkv, D, page_size, FP32,
                     fill_len=[total] * num_seqs)
    # hide the keys the decode steps will append: take them out of the pool
    appended = []
    for s in range(decode_steps):
        j = kv_len + s
        ks, vs = [], []
        for b in range(num_seqs):
            phys = pool.block_table[b, j // page_size]
            ks.append(pool.k_cache[phys, j % page_size].copy())
            vs.append(pool.v_cache[phys, j % page_size].copy())
            pool.k_cache[phys, j % page_size] = np.nan
            pool.v_cache[phys, j % page_size] = np.nan
        appended.append((np.stack(ks), np.stack(vs)))
    sinks = sinks_normal(rng, Hq, 1.0)
    q = make_queries(rng, num_seqs * q_len, Hq, D, FP32)
    prefill = batch_from_pool(pool, np.arange(num_seqs), [q_len] * num_seqs, q, sinks,
                              True, FP32, dict(workload="tiny prefill+decode"))
    steps = []
    for s in range(decode_steps):
        qd = make_queries(rng, num_seqs, Hq, D, FP32)
        steps.append(dict(q=qd, new_k=appended[s][0], new_v=appended[s][1],
                          kv_lens=np.full(num_seqs, kv_len + s + 1, dtype=np.int32),
                          positions=np.full(num_seqs, kv_len + s, dtype=np.int32)))
    return dict(prefill=prefill, steps=steps, pool=pool)


def gptoss_decode(seed=20260002, num_seqs=64, Hq=64, Hkv=8, D=64, kv_min=512, kv_max=8192,
                  page_size=16, sink_std=2.0, dtype=BF16):
    """Decode: one query token per sequence, KV lengths uniform in [kv_min, kv_max]."""
    rng = np.random.default_rng(seed)
    kv = rng.integers(kv_min, kv_max + 1, num_seqs)
    pool = make_pool(rng, kv, Hkv, D, page_size, dtype)
    sinks = sinks_normal(rng, Hq, sink_std)
    q = make_queries(rng, num_seqs, Hq, D, dtype)
    return batch_from_pool(pool, np.arange(num_seqs), np.ones(num_seqs, np.int64), q, sinks,
                           True, dtype, dict(workload="gpt-oss decode"))


def gptoss_prefill(seed=20260003, num_seqs=8, seq_len=4096, Hq=64, Hkv=8, D=64, page_size=16,
                   sink_std=2.0, dtype=BF16, q_lens=None):
    """Causal self-attention prefill: q_len == kv_len per sequence, ragged layout."""
    rng = np.random.default_rng(seed)
    lens = np.full(num_seqs, seq_len, np.int64) if q_lens is None else np.asarray(q_lens, np.int64)
    pool = make_pool(rng, lens, Hkv, D, page_size, dtype)
    sinks = sinks_normal(rng, Hq, sink_std)
    q = make_queries(rng, int(lens.sum()), Hq, D, dtype)
    return batch_from_pool(pool, np.arange(len(lens)), lens, q, sinks, True, dtype,
                           dict(workload="gpt-oss causal prefill"))


def long_split_decode(seed=20260004, num_seqs=4, kv_len=131072, Hq=64, Hkv=8, D=64,
                      page_size=16, num_splits=32, dtype=BF16):
    """Long-context decode with sinks drawn from {-inf, -4, 0, 4, 8}."""
    rng = np.random.default_rng(seed)
    pool = make_pool(rng, np.full(num_seqs, kv_len), Hkv, D, page_size, dtype)
    sinks = sinks_choice(rng, Hq)
    q = make_queries(rng, num_seqs, Hq, D, dtype)
    return batch_from_pool(pool, np.arange(num_seqs), np.ones(num_seqs, np.int64), q, sinks,
                           True, dtype, dict(workload="long split-KV decode",
                                             num_splits=num_splits))


def mixed_batch(seed=20260005, n_decode=48, decode_kv=(1024, 32768), n_prefill=4,
                prefill_new=512, prefix=(0, 16384), Hq=64, Hkv=8, D=64, page_size=16,
                sink_std=2.0, outlier_frac=0.01, dtype=BF16):
    """Decode sequences plus chunked-prefill segments sharing one page pool.

    1% of (token, kv-head) K rows are scaled by 20 before rounding (outlier
    logits).  Returns dict(decode=Batch, prefill=Batch, single=Batch), the last
    being both parts as one ragged batch (decode sequences as 1-token segments).
    """
    rng = np.random.default_rng(seed)
    kv_dec = rng.integers(decode_kv[0], decode_kv[1] + 1, n_decode)
    pre = rng.integers(prefix[0], prefix[1] + 1, n_prefill)
    kv_all = np.concatenate([kv_dec, pre + prefill_new])
    pool = make_pool(rng, kv_all, Hkv, D, page_size, dtype, outlier_frac=outlier_frac)
    sinks = sinks_normal(rng, Hq, sink_std)
    qd = make_queries(rng, n_decode, Hq, D, dtype)
    qp = make_queries(rng, n_prefill * prefill_new, Hq, D, dtype)
    dec = batch_from_pool(pool, np.arange(n_decode), np.ones(n_decode, np.int64), qd, sinks,
                          True, dtype, dict(workload="mixed batch: decode part"))
    prf = batch_from_pool(pool, np.arange(n_decode, n_decode + n_prefill),
                          np.full(n_prefill, prefill_new), qp, sinks, True, dtype,
                          dict(workload="mixed batch: chunked-prefill part", prefix=pre))
    # The whole batch as one ragged query batch: each decode sequence is a
    # one-token segment at its last position, then the chunked-prefill segments.
    one = batch_from_pool(pool, np.arange(n_decode + n_prefill),
                          np.concatenate([np.ones(n_decode, np.int64),
                                          np.full(n_prefill, prefill_new, np.int64)]),
                          np.concatenate([qd, qp]), sinks, True, dtype,
                          dict(workload="mixed batch as one ragged batch", n_decode=n_decode))
    return dict(decode=dec, prefill=prf, single=one)


def sample_rows(rng, batch, n):
    """Random flat rows (token * Hq + head) plus the first and last row."""
    total = batch.total_q * batch.Hq
    n = min(n, total)
    rows = rng.choice(total, size=n, replace=False)
    return np.unique(np.concatenate([rows, [0, total - 1]])).astype(np.int64)
