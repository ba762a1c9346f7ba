"""GPU parity of the causal ragged prefill (tcgen05 / TMEM / TMA) against the oracle."""
import math

import numpy as np
import pytest

import workloads as W
from _gpu import DeviceBatch, compare, oracle_problem

pytestmark = pytest.mark.gpu


def _prefill(gas, db, causal=None, **kw):
    b = db.b
    return gas.prefill(db.q, db.k, db.v, db.cu, db.kv_lens, db.bt, db.sinks,
                       max_q_len=b.max_q_len, scale=b.scale,
                       causal=b.causal if causal is None else causal, err_flag=db.err, **kw)


def _batch(seed, q_lens, prefix=None, Hq=64, Hkv=8, sink_std=2.0, causal=True, dtype=W.BF16,
           sinks=None):
    rng = np.random.default_rng(seed)
    q_lens = np.asarray(q_lens, np.int64)
    pre = np.zeros_like(q_lens) if prefix is None else np.asarray(prefix, np.int64)
    pool = W.make_pool(rng, q_lens + pre, Hkv, 64, 16, dtype)
    s = W.sinks_normal(rng, Hq, sink_std) if sinks is None else np.asarray(sinks, np.float32)
    q = W.make_queries(rng, int(q_lens.sum()), Hq, 64, dtype)
    return W.batch_from_pool(pool, np.arange(len(q_lens)), q_lens, q, s, causal, dtype)


def _check_all(gas, batch, what):
    db = DeviceBatch(batch)
    out, lse = _prefill(gas, db)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what=what)
    assert db.err.item() == 0, db.err.item()
    return out, lse


def test_prefill_ragged_self_attention(cuda_lib):
    """Ragged lengths spanning several tiles plus short tails (1, 16, 33 tokens)."""
    _check_all(cuda_lib, _batch(21, [200, 77, 1, 16, 33, 300]), "ragged causal")


def test_prefill_empty_segment_and_loose_max_q_len(cuda_lib):
    """A sequence with no new tokens between two that have some (its KV prefix is
    never read), and max_q_len given as a loose upper bound: the grid then holds
    work tiles past every sequence's end, which must do nothing."""
    batch = _batch(23, [40, 0, 25], prefix=[0, 100, 50])
    db = DeviceBatch(batch)
    out, lse = cuda_lib.prefill(db.q, db.k, db.v, db.cu, db.kv_lens, db.bt, db.sinks,
                                max_q_len=batch.max_q_len + 200, scale=batch.scale,
                                causal=True, err_flag=db.err)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what="empty segment")
    assert db.err.item() == 0, db.err.item()


def test_prefill_with_prefix(cuda_lib):
    """Chunked prefill: new tokens appended to an existing KV prefix (bottom-right causal)."""
    _check_all(cuda_lib, _batch(22, [64, 100, 5, 130], prefix=[0, 300, 17, 1000]), "prefix")


def test_prefill_many_sequences_global_metadata(cuda_lib):
    """1100 short sequences: more than the kernel keeps in shared memory, so work
    tiles are decoded from the global length arrays (and a few with long prefixes)."""
    rng = np.random.default_rng(31)
    q_lens = rng.integers(1, 6, 1100)
    prefix = rng.integers(0, 40, 1100)
    prefix[::97] = 300
    _check_all(cuda_lib, _batch(31, q_lens, prefix=prefix, Hq=16, Hkv=2), "1100 sequences")


def test_prefill_many_heads_global_sinks(cuda_lib):
    """Hq = 288 query heads (group 16 over 18 KV heads): more sinks than the
    kernel keeps in shared memory."""
    _check_all(cuda_lib, _batch(32, [40, 9], prefix=[0, 20], Hq=288, Hkv=18), "288 heads")


def test_prefill_multi_token_verify(cuda_lib):
    """Speculative-decoding verification: 2..5 new tokens per sequence over prefixes of
    1k..5k keys (bottom-right causal), 24 sequences, Hq 64 / Hkv 8."""
    rng = np.random.default_rng(33)
    q_lens = rng.integers(2, 6, 24)
    prefix = rng.integers(1000, 5000, 24)
    _check_all(cuda_lib, _batch(33, q_lens, prefix=prefix), "multi-token verify")


def test_prefill_one_long_sequence_sampled(cuda_lib):
    """One 16384-token causal prefill (rows see up to 128 key tiles), Hq 64 / Hkv 8:
    sampled rows plus both ends of the sequence."""
    batch = _batch(34, [16384])
    db = DeviceBatch(batch)
    out, lse = _prefill(cuda_lib, db)
    rows = W.sample_rows(np.random.default_rng(34), batch, 768)
    ends = np.concatenate([np.arange(t * 64, (t + 1) * 64) for t in (0, 1, 16382, 16383)])
    rows = np.unique(np.concatenate([rows, ends]))
    ref, ref_lse, _ = oracle_problem(batch).attention(rows)
    compare(out, lse, ref, ref_lse, rows=rows, what="one long prefill")
    assert db.err.item() == 0


def test_prefill_rows_before_first_key(cuda_lib):
    """Causal with kv_len < q_len: bottom-right aligned, the first q_len - kv_len rows
    of a sequence see no key at all (out 0, lse = sink), including a whole tile."""
    rng = np.random.default_rng(35)
    q_lens = np.array([40, 10, 20, 300])
    kv = np.array([30, 3, 20, 100])
    pool = W.make_pool(rng, kv, 8, 64, 16, W.BF16)
    sinks = W.sinks_normal(rng, 64, 2.0)
    q = W.make_queries(rng, int(q_lens.sum()), 64, 64, W.BF16)
    _check_all(cuda_lib, W.batch_from_pool(pool, np.arange(4), q_lens, q, sinks),
               "rows before the first key")


def test_prefill_non_causal(cuda_lib):
    batch = _batch(23, [50, 129], prefix=[10, 60], causal=False)
    _check_all(cuda_lib, batch, "non-causal")


@pytest.mark.parametrize("group,Hkv", [(1, 4), (2, 4), (4, 2), (16, 2)])
def test_prefill_group_sizes(cuda_lib, group, Hkv):
    _check_all(cuda_lib, _batch(24, [70, 200], prefix=[0, 33], Hq=group * Hkv, Hkv=Hkv),
               "group %d" % group)


def test_prefill_single_kv_head(cuda_lib):
    """Multi-query attention: one KV head, 16 query heads (group 16)."""
    _check_all(cuda_lib, _batch(36, [90, 33], prefix=[0, 200], Hq=16, Hkv=1), "MQA prefill")


def test_prefill_sink_extremes(cuda_lib):
    """Sinks -inf, -4, 0, 4, 8 and large: sink=-inf is plain attention, large sinks
    push the output toward 0."""
    sinks = np.array([-math.inf, -4, 0, 4, 8, 20, -math.inf, 8] * 8, np.float32)
    _check_all(cuda_lib, _batch(25, [150, 40], prefix=[20, 0], sinks=sinks), "sink extremes")


def test_prefill_outlier_keys(cuda_lib):
    """1% of K rows scaled by 20 (logits in the hundreds): rescaling must stay exact."""
    m = W.mixed_batch(seed=26, n_decode=1, decode_kv=(16, 16), n_prefill=3, prefill_new=160,
                      prefix=(0, 700))
    _check_all(cuda_lib, m["prefill"], "outliers")


def test_prefill_fp32_tiny(cuda_lib):
    """Tiny fp32 case: 2 seqs, Hq 8 / Hkv 2, q_len 16 over kv_len 64 (SIMT fp32 path)."""
    t = W.tiny_prefill_decode()
    _check_all(cuda_lib, t["prefill"], "fp32 tiny prefill")


def test_prefill_page_table_bitwise_and_deterministic(cuda_lib):
    batch = _batch(27, [130, 90], prefix=[40, 0])
    rng = np.random.default_rng(27)
    perm = rng.permutation(batch.num_pages)
    inv = np.argsort(perm)
    moved = W.Batch(batch.dtype, batch.q, batch.k_cache[perm], batch.v_cache[perm],
                    batch.cu_seqlens_q, batch.kv_lens,
                    np.where(batch.block_table >= 0, inv[np.maximum(batch.block_table, 0)],
                             -1).astype(np.int32), batch.sinks, batch.scale)
    a, b = DeviceBatch(batch), DeviceBatch(moved)
    oa, la = _prefill(cuda_lib, a)
    ob, lb = _prefill(cuda_lib, b)
    oc, lc = _prefill(cuda_lib, a)
    assert bool((oa == ob).all()) and bool((la == lb).all())
    assert bool((oa == oc).all()) and bool((la == lc).all())


def test_prefill_bad_page_sets_flag(cuda_lib):
    batch = _batch(28, [100, 60], prefix=[50, 0])
    batch.block_table[0, 2] = batch.num_pages + 1
    db = DeviceBatch(batch)
    out, lse = _prefill(cuda_lib, db)
    assert db.err.item() & cuda_lib.FLAG_BAD_PAGE
    assert not db.err.item() & cuda_lib.FLAG_TIMEOUT
    ref, ref_lse, bad = oracle_problem(batch).attention()
    assert bad > 0
    compare(out, lse, ref, ref_lse, what="bad page")


def test_prefill_gptoss_full(cuda_lib):
    """8 x 4096 causal prefill, Hq 64 / Hkv 8, as the bench runs it: every row
    (2.1 M rows, about 4.3 G query-key pairs for the oracle)."""
    batch = W.gptoss_prefill()
    db = DeviceBatch(batch)
    out, lse = _prefill(cuda_lib, db)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what="gpt-oss prefill, every row")
    assert db.err.item() == 0


def test_prefill_mixed_part_full(cuda_lib):
    """Chunked-prefill half of the mixed batch (4 x 512 new tokens over prefixes up
    to 16k, 1% outlier keys), as the bench runs it: every row."""
    m = W.mixed_batch()
    batch = m["prefill"]
    db = DeviceBatch(batch)
    out, lse = _prefill(cuda_lib, db)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what="mixed prefill, every row")
    assert db.err.item() == 0


def test_prefill_mixed_batch_as_one_launch(cuda_lib):
    """The whole mixed batch (48 decode sequences as one-token segments at their
    last position, then four 512-token chunks over long prefixes, 1% outlier
    keys) as a single prefill launch from one work list: every decode row and a
    sample of the chunk rows against the oracle."""
    batch = W.mixed_batch()["single"]
    db = DeviceBatch(batch)
    out, lse = _prefill(cuda_lib, db)
    n_dec = batch.meta["n_decode"]
    rows = np.unique(np.concatenate([np.arange(n_dec * batch.Hq),
                                     W.sample_rows(np.random.default_rng(41), batch, 400)]))
    ref, ref_lse, _ = oracle_problem(batch).attention(rows)
    compare(out, lse, ref, ref_lse, rows=rows, what="mixed batch as one launch")
    assert db.err.item() == 0, db.err.item()



def test_prefill_workspace_reused_back_to_back(cuda_lib):
    """One workspace for two different calls enqueued back to back (no host sync in
    between): each call restarts the tile-claim counter, so both cover every tile."""
    import torch
    a = _batch(51, [300, 5, 77], prefix=[0, 900, 40])
    b = _batch(52, [1, 1, 1, 700], prefix=[4000, 30, 0, 10])
    da, dbb = DeviceBatch(a), DeviceBatch(b)
    need = max(cuda_lib.prefill_workspace_size(x.B, x.Hq, x.D, x.max_q_len) for x in (a, b))
    wsb = torch.empty(need, dtype=torch.uint8, device="cuda")
    oa, la = _prefill(cuda_lib, da, workspace=wsb)
    ob, lb = _prefill(cuda_lib, dbb, workspace=wsb)
    oa2, la2 = _prefill(cuda_lib, da, workspace=wsb)
    for batch, db, o, l in ((a, da, oa, la), (b, dbb, ob, lb)):
        ref, ref_lse, _ = oracle_problem(batch).attention()
        compare(o, l, ref, ref_lse, what="reused workspace")
        assert db.err.item() == 0
    assert torch.equal(oa, oa2) and torch.equal(la, la2)
