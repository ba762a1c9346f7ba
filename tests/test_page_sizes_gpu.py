"""Page sizes other than 16 (any multiple of 16 up to 256): prefill, split decode and
the appending decode step against the oracle.  A page then holds several 16-key
units, so the in-page row offsets and the decode's (dim, token in page, head, page)
tensor-map coordinates are exercised."""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu import DeviceBatch, compare, oracle_problem, to_device

pytestmark = pytest.mark.gpu


def _batch(seed, q_lens, prefix, page_size, Hq=32, Hkv=4, decode=False):
    rng = np.random.default_rng(seed)
    q_lens = np.asarray(q_lens, np.int64)
    kv = q_lens + np.asarray(prefix, np.int64)
    pool = W.make_pool(rng, kv, Hkv, 64, page_size, W.BF16)
    sinks = W.sinks_normal(rng, Hq, 2.0)
    nq = len(kv) if decode else int(q_lens.sum())
    q = W.make_queries(rng, nq, Hq, 64, W.BF16)
    return W.batch_from_pool(pool, np.arange(len(kv)), np.ones(len(kv), np.int64) if decode else q_lens,
                             q, sinks)


@pytest.mark.parametrize("page_size", [32, 64, 256])
def test_prefill_page_sizes(cuda_lib, page_size):
    batch = _batch(60 + page_size, [150, 33, 7], [0, 300, 1000], page_size)
    db = DeviceBatch(batch)
    out, lse = cuda_lib.prefill(db.q, db.k, db.v, db.cu, db.kv_lens, db.bt, db.sinks,
                                max_q_len=batch.max_q_len, scale=batch.scale, err_flag=db.err)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what="prefill page %d" % page_size)
    assert db.err.item() == 0


@pytest.mark.parametrize("page_size,num_splits", [(32, 0), (64, 0), (64, 3), (256, 0), (256, 2), (64, -1)])
def test_decode_page_sizes(cuda_lib, page_size, num_splits):
    batch = _batch(70 + page_size, [1] * 6, [0, 15, 200, 1023, 3000, 512], page_size, decode=True)
    db = DeviceBatch(batch)
    out, lse = cuda_lib.decode(db.q, db.k, db.v, db.kv_lens, db.bt, db.sinks, scale=batch.scale,
                               num_splits=num_splits, err_flag=db.err)
    ref, ref_lse, _ = oracle_problem(batch).attention()
    compare(out, lse, ref, ref_lse, what="decode page %d S=%d" % (page_size, num_splits))
    assert db.err.item() == 0


@pytest.mark.parametrize("page_size", [32, 256])
def test_decode_append_page_sizes(cuda_lib, page_size):
    full = _batch(80 + page_size, [1] * 5, [0, 40, 255, 256, 700], page_size, decode=True)
    k_hidden, v_hidden = full.k_cache.copy(), full.v_cache.copy()
    Hkv = full.k_cache.shape[2]
    k_new = np.empty((full.B, Hkv, 64), np.uint16)
    v_new = np.empty_like(k_new)
    for b, kv in enumerate(full.kv_lens):
        pos = int(kv) - 1
        phys, row = full.block_table[b, pos // page_size], pos % page_size
        k_new[b], v_new[b] = full.k_cache[phys, row], full.v_cache[phys, row]
        k_hidden[phys, row] = 0x7FC0
        v_hidden[phys, row] = 0x7FC0
    hidden = W.Batch(full.dtype, full.q, k_hidden, v_hidden, full.cu_seqlens_q, full.kv_lens,
                     full.block_table, full.sinks, full.scale)
    db = DeviceBatch(hidden)
    out, lse = cuda_lib.decode_append(db.q, to_device(k_new, None), to_device(v_new, None), db.k,
                                      db.v, db.kv_lens, db.bt, db.sinks, scale=full.scale,
                                      err_flag=db.err)
    torch.cuda.synchronize()
    assert torch.equal(db.k.view(torch.int16), to_device(full.k_cache, None).view(torch.int16))
    ref, ref_lse, _ = oracle_problem(full).attention()
    compare(out, lse, ref, ref_lse, what="decode+append page %d" % page_size)
    assert db.err.item() == 0
