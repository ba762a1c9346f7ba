"""GPU parity of paged split-KV decode (and the merge) against the fp64 oracle."""
import math

import numpy as np
import pytest

import workloads as W
from _gpu import DeviceBatch, compare, oracle_problem

pytestmark = pytest.mark.gpu


def _decode(gas, db, num_splits=0, **kw):
    return gas.decode(db.q, db.k, db.v, db.kv_lens, db.bt, db.sinks, scale=db.b.scale,
                      num_splits=num_splits, err_flag=db.err, **kw)


def _small_decode(seed=5, num_seqs=7, kv=(1, 700), Hq=64, Hkv=8, sink_std=2.0, kv_lens=None):
    rng = np.random.default_rng(seed)
    lens = rng.integers(kv[0], kv[1] + 1, num_seqs) if kv_lens is None else np.asarray(kv_lens)
    pool = W.make_pool(rng, lens, Hkv, 64, 16, W.BF16)
    sinks = W.sinks_normal(rng, Hq, sink_std)
    q = W.make_queries(rng, len(lens), Hq, 64, W.BF16)
    return W.batch_from_pool(pool, np.arange(len(lens)), np.ones(len(lens), np.int64), q, sinks)


@pytest.mark.parametrize("num_splits", [0, 1, 2, 7, 32, -1])
def test_decode_parity_small(cuda_lib, num_splits):
    batch = _small_decode()
    db = DeviceBatch(batch)
    out, lse = _decode(cuda_lib, db, num_splits)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what="decode S=%d" % num_splits)
    assert db.err.item() == 0


@pytest.mark.parametrize("group,Hkv", [(1, 4), (2, 4), (4, 2), (16, 2)])
def test_decode_group_sizes(cuda_lib, group, Hkv):
    batch = _small_decode(seed=6, num_seqs=3, kv=(5, 300), Hq=group * Hkv, Hkv=Hkv)
    db = DeviceBatch(batch)
    for S in (0, 3, -1):
        out, lse = _decode(cuda_lib, db, S)
        ref, ref_lse, _ = oracle_problem(batch).attention()
        compare(out, lse, ref, ref_lse, what="group %d S=%d" % (group, S))


@pytest.mark.parametrize("Hq", [8, 16])
def test_decode_single_kv_head(cuda_lib, Hq):
    """Multi-query attention (Hkv = 1): the 4-head TMA box reaches past the tensor's
    head dimension, whose missing heads TMA fills with zeros."""
    batch = _small_decode(seed=12, num_seqs=5, kv=(1, 900), Hq=Hq, Hkv=1)
    db = DeviceBatch(batch)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    for S in (0, 3, -1):
        out, lse = _decode(cuda_lib, db, S)
        compare(out, lse, ref, ref_lse, what="MQA decode Hq %d S=%d" % (Hq, S))
    assert db.err.item() == 0


def test_decode_edge_lengths(cuda_lib):
    """kv_len 0 (out 0, lse = sink), 1, page boundaries and ragged tails."""
    lens = [0, 1, 15, 16, 17, 31, 32, 33, 63, 64, 65, 511, 512, 513]
    batch = _small_decode(seed=7, kv_lens=lens)
    batch.sinks[:4] = -math.inf                       # sink -inf with kv_len 0 -> lse -inf
    db = DeviceBatch(batch)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    for S in (0, 1, 4, 40, -1):
        out, lse = _decode(cuda_lib, db, S)
        compare(out, lse, ref, ref_lse, what="edge S=%d" % S)
        assert db.err.item() == 0


def test_decode_max_splits(cuda_lib):
    """num_splits = 256 (the maximum): most chunks of these sequences are empty pages
    ranges and only chunk 0 carries the sink."""
    batch = _small_decode(seed=9, num_seqs=4, kv=(1, 4100))
    db = DeviceBatch(batch)
    out, lse = _decode(cuda_lib, db, 256)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what="decode S=256")
    assert db.err.item() == 0


def test_decode_split_invariance_and_determinism(cuda_lib):
    batch = _small_decode(seed=8, num_seqs=5, kv=(200, 2000))
    db = DeviceBatch(batch)
    base, base_lse = _decode(cuda_lib, db, 1)
    for S in (2, 7, 32, 0):
        out, lse = _decode(cuda_lib, db, S)
        diff = (out.float() - base.float()).abs().max().item()
        assert diff <= 1e-2, (S, diff)
        assert (lse - base_lse).abs().max().item() <= 1e-3
        again, again_lse = _decode(cuda_lib, db, S)
        assert bool((again == out).all())
        assert bool((again_lse == lse).all())


def test_decode_page_table_bitwise(cuda_lib):
    """Same logical KV under a different physical placement: bitwise-equal output."""
    batch = _small_decode(seed=9, num_seqs=4, kv=(30, 900))
    rng = np.random.default_rng(9)
    perm = rng.permutation(batch.num_pages)
    inv = np.argsort(perm)
    moved = W.Batch(batch.dtype, batch.q, batch.k_cache[perm], batch.v_cache[perm],
                    batch.cu_seqlens_q, batch.kv_lens,
                    np.where(batch.block_table >= 0, inv[np.maximum(batch.block_table, 0)], -1).astype(np.int32),
                    batch.sinks, batch.scale)
    a, b = DeviceBatch(batch), DeviceBatch(moved)
    for S in (0, 3, -1):
        oa, la = _decode(cuda_lib, a, S)
        ob, lb = _decode(cuda_lib, b, S)
        assert bool((oa == ob).all()) and bool((la == lb).all())


def test_decode_bad_page_sets_flag(cuda_lib):
    batch = _small_decode(seed=10, num_seqs=3, kv_lens=[100, 200, 50])
    batch.block_table[1, 3] = batch.num_pages + 5       # out of the pool
    batch.block_table[2, 0] = -7
    db = DeviceBatch(batch)
    ref, ref_lse, bad = oracle_problem(batch).attention()
    assert bad > 0
    for S in (0, 1, 5, -1):
        db.err.zero_()
        out, lse = _decode(cuda_lib, db, S)
        assert db.err.item() & cuda_lib.FLAG_BAD_PAGE
        assert not db.err.item() & cuda_lib.FLAG_TIMEOUT
        compare(out, lse, ref, ref_lse, what="bad page S=%d" % S)


def test_merge_entry_point(cuda_lib):
    """attn_sink_merge on oracle partials equals the oracle's unsplit result."""
    import torch
    batch = _small_decode(seed=11, num_seqs=3, kv=(40, 400), Hq=16, Hkv=2)
    prob = oracle_problem(batch)
    rows = prob.all_rows()
    S = 5
    bounds = prob.split_bounds(rows, S)
    o, l, _ = prob.partials(rows, bounds, 1)
    ref, ref_lse, _ = prob.attention()
    op = torch.from_numpy(o.astype(np.float32)).cuda()
    lp = torch.from_numpy(l.astype(np.float32)).cuda()
    for dt in (torch.bfloat16, torch.float32):
        out, lse = cuda_lib.merge(op, lp, out_dtype=dt)
        compare(out, lse, ref, ref_lse, what="merge %s" % dt)
    # all partials at -inf: out 0 and lse -inf
    out, lse = cuda_lib.merge(torch.zeros(2, 3, 64, device="cuda"),
                              torch.full((2, 3), -math.inf, device="cuda"))
    assert bool((out.float() == 0).all()) and bool(torch.isneginf(lse).all())


def test_decode_fp32_tiny_steps(cuda_lib):
    """Tiny fp32 workload: 4 decode steps, each appending one K/V row first."""
    import torch
    t = W.tiny_prefill_decode()
    batch = t["prefill"]
    db = DeviceBatch(batch)
    for step in t["steps"]:
        for b in range(batch.B):
            j = int(step["positions"][b])
            phys = int(batch.block_table[b, j // batch.page_size])
            batch.k_cache[phys, j % batch.page_size] = step["new_k"][b]
            batch.v_cache[phys, j % batch.page_size] = step["new_v"][b]
            db.k[phys, j % batch.page_size] = torch.from_numpy(step["new_k"][b]).cuda()
            db.v[phys, j % batch.page_size] = torch.from_numpy(step["new_v"][b]).cuda()
        dec = W.Batch(W.FP32, step["q"], batch.k_cache, batch.v_cache,
                      np.arange(batch.B + 1, dtype=np.int32), step["kv_lens"], batch.block_table,
                      batch.sinks, batch.scale)
        ref, ref_lse, _ = oracle_problem(dec).attention()
        q = torch.from_numpy(step["q"]).cuda()
        kvl = torch.from_numpy(step["kv_lens"]).cuda()
        for S in (0, 2):
            out, lse = cuda_lib.decode(q, db.k, db.v, kvl, db.bt, db.sinks, num_splits=S,
                                       err_flag=db.err)
            compare(out, lse, ref, ref_lse, what="fp32 decode S=%d" % S)
        assert db.err.item() == 0


def test_decode_gptoss_full(cuda_lib):
    """64 seqs, KV 512..8192, Hq 64 / Hkv 8: every row against the oracle."""
    batch = W.gptoss_decode()
    db = DeviceBatch(batch)
    out, lse = _decode(cuda_lib, db, 0)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what="gpt-oss decode")
    out_p, lse_p = _decode(cuda_lib, db, -1)         # the persistent split
    compare(out_p, lse_p, ref, ref_lse, what="gpt-oss decode, persistent split")
    assert db.err.item() == 0


def test_decode_long_split_full(cuda_lib):
    """4 seqs x 131072 keys split into 32 chunks; sinks from {-inf,-4,0,4,8}."""
    batch = W.long_split_decode()
    db = DeviceBatch(batch)
    out, lse = _decode(cuda_lib, db, 32)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what="long split decode")
    out0, lse0 = _decode(cuda_lib, db, 0)
    compare(out0, lse0, ref, ref_lse, what="long decode auto split")
    assert db.err.item() == 0


def test_decode_mixed_part_full(cuda_lib):
    """Decode half of the mixed batch (KV 1k..32k, 1% outlier keys), as the bench
    runs it: every row."""
    m = W.mixed_batch()
    batch = m["decode"]
    db = DeviceBatch(batch)
    out, lse = _decode(cuda_lib, db, 0)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what="mixed decode, every row")
    assert db.err.item() == 0
