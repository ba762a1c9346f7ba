"""GPU parity of attn_sink_mixed (decode rows and prefill segments in one
persistent launch) against the oracle."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from _gpu import DeviceBatch, compare, oracle_problem

pytestmark = pytest.mark.gpu


def _mixed(gas, db, num_decode, **kw):
    b = db.b
    max_q = int(b.q_lens[num_decode:].max()) if num_decode < b.B else 1
    return gas.mixed(db.q, db.k, db.v, db.cu, db.kv_lens, db.bt, db.sinks, num_decode=num_decode,
                     max_q_len=max_q, scale=b.scale, causal=b.causal, err_flag=db.err, **kw)


def _batch(seed, dec_kv, pre_q, pre_prefix, Hq=64, Hkv=8, sinks=None, outlier_frac=0.0):
    """num_decode one-token sequences over dec_kv keys, then prefill segments of
    pre_q new tokens over pre_prefix earlier keys, in one pool."""
    rng = np.random.default_rng(seed)
    dec_kv = np.asarray(dec_kv, np.int64)
    pre_q = np.asarray(pre_q, np.int64)
    kv = np.concatenate([dec_kv, pre_q + np.asarray(pre_prefix, np.int64)])
    pool = W.make_pool(rng, np.maximum(kv, 1), Hkv, 64, 16, W.BF16, outlier_frac=outlier_frac)
    pool.kv_lens[:] = kv                      # kv_len 0 rows keep one (unread) page
    s = W.sinks_normal(rng, Hq, 2.0) if sinks is None else np.asarray(sinks, np.float32)
    q_lens = np.concatenate([np.ones(len(dec_kv), np.int64), pre_q])
    q = W.make_queries(rng, int(q_lens.sum()), Hq, 64, W.BF16)
    return W.batch_from_pool(pool, np.arange(len(kv)), q_lens, q, s)


def _check(gas, batch, num_decode, what):
    db = DeviceBatch(batch)
    out, lse = _mixed(gas, db, num_decode)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what=what)
    assert db.err.item() == 0, db.err.item()
    return db, out, lse


def test_mixed_small_edges(cuda_lib):
    """Decode rows with kv_len 0, 1, 15, 16, 17, 1024, 1025 (one past a chunk)
    and 3000 (three chunks), next to prefill segments with and without a prefix."""
    _check(cuda_lib, _batch(61, [0, 1, 15, 16, 17, 1024, 1025, 3000], [40, 200, 7], [0, 333, 2000]),
           8, "mixed edges")


@pytest.mark.parametrize("group,Hkv", [(8, 2), (16, 2), (1, 8), (4, 18)])
def test_mixed_head_layouts(cuda_lib, group, Hkv):
    """KV heads not a multiple of the 8-head decode box (the box's extra heads
    are zero-filled and skipped), group sizes 1..16."""
    _check(cuda_lib, _batch(62, [900, 2100, 40], [33, 150], [60, 500], Hq=group * Hkv, Hkv=Hkv),
           3, "mixed group %d Hkv %d" % (group, Hkv))


def test_mixed_sink_extremes(cuda_lib):
    sinks = np.array([-math.inf, -4, 0, 4, 8, 20, -math.inf, 8] * 8, np.float32)
    _check(cuda_lib, _batch(63, [700, 5000], [90], [100], sinks=sinks), 2, "mixed sinks")


def test_mixed_all_decode_and_no_decode(cuda_lib):
    """num_decode = B (only decode items) and num_decode = 0 (only query tiles)."""
    _check(cuda_lib, _batch(64, [100, 2048, 4097, 1], [], []), 4, "mixed all decode")
    _check(cuda_lib, _batch(65, [], [64, 300], [0, 1000]), 0, "mixed no decode")


def test_mixed_matches_prefill_of_the_same_batch(cuda_lib):
    """attn_sink_mixed and attn_sink_prefill over one batch agree (the decode rows
    differ only in fp32 summation order)."""
    batch = _batch(66, [1500, 70, 4000], [128, 20], [256, 0])
    db = DeviceBatch(batch)
    om, lm = _mixed(cuda_lib, db, 3)
    op, lp = cuda_lib.prefill(db.q, db.k, db.v, db.cu, db.kv_lens, db.bt, db.sinks,
                              max_q_len=batch.max_q_len, scale=batch.scale, err_flag=db.err)
    assert (om.float() - op.float()).abs().max().item() <= 1e-2
    assert (lm - lp).abs().max().item() <= 1e-3
    # the prefill segments' rows run the same query tiles: bitwise equal
    first = int(batch.cu_seqlens_q[3])
    assert torch.equal(om[first:], op[first:]) and torch.equal(lm[first:], lp[first:])
    assert db.err.item() == 0


def test_mixed_bad_page_in_a_decode_row(cuda_lib):
    batch = _batch(67, [2000, 300], [50], [10])
    batch.block_table[0, 5] = batch.num_pages + 3
    db = DeviceBatch(batch)
    out, lse = _mixed(cuda_lib, db, 2)
    assert db.err.item() & cuda_lib.FLAG_BAD_PAGE
    ref, ref_lse, bad = oracle_problem(batch).attention()
    assert bad > 0
    compare(out, lse, ref, ref_lse, what="mixed bad page")


def test_mixed_deterministic_and_workspace_reuse(cuda_lib):
    batch = _batch(68, [3000, 123, 9000], [64, 256], [512, 4000])
    db = DeviceBatch(batch)
    need = cuda_lib.mixed_workspace_size(3, batch.Hq, batch.Hkv, 64, batch.block_table.shape[1], 16)
    wsb = torch.empty(need, dtype=torch.uint8, device="cuda")
    o1, l1 = _mixed(cuda_lib, db, 3, workspace=wsb)
    o2, l2 = _mixed(cuda_lib, db, 3, workspace=wsb)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_mixed_gptoss_full(cuda_lib):
    """The mixed workload as one launch: 48 decode rows over 1k..32k keys and four
    512-token chunks over prefixes up to 16k, 1% outlier keys: every row."""
    batch = W.mixed_batch()["single"]
    _check(cuda_lib, batch, batch.meta["n_decode"], "mixed batch, one launch, every row")


def test_mixed_fp32(cuda_lib):
    """fp32 inputs run the whole mixed batch on the fp32 path (decode rows included)."""
    rng = np.random.default_rng(69)
    dec_kv, pre_q, pre_prefix = np.array([40, 90]), np.array([16, 5]), np.array([48, 0])
    kv = np.concatenate([dec_kv, pre_q + pre_prefix])
    pool = W.make_pool(rng, kv, 2, 64, 16, W.FP32)
    sinks = W.sinks_normal(rng, 8, 1.0)
    q_lens = np.concatenate([np.ones(2, np.int64), pre_q])
    q = W.make_queries(rng, int(q_lens.sum()), 8, 64, W.FP32)
    batch = W.batch_from_pool(pool, np.arange(4), q_lens, q, sinks, True, W.FP32)
    _check(cuda_lib, batch, 2, "mixed fp32")
