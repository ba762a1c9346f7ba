"""GPU parity of the decode step that appends its own key and value first
(attn_sink_decode_append): the appended slots hold k_new / v_new bit for bit, the
outputs match the oracle over the completed cache, and they equal an explicit
write followed by attn_sink_decode bit for bit."""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu import DeviceBatch, compare, oracle_problem, to_device

pytestmark = pytest.mark.gpu


def _same_bits(a, b):
    """Bitwise equality (NaN-poisoned slots compare equal to themselves)."""
    it = torch.int16 if a.element_size() == 2 else torch.int32
    return torch.equal(a.view(it), b.view(it))


def _hidden_last(seed, lens, Hq=64, Hkv=8):
    """Batch whose last key of every sequence is taken out of the cache (NaN there)
    and returned as the step's k_new / v_new [B, Hkv, 64]."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, np.int64)
    pool = W.make_pool(rng, lens, Hkv, 64, 16, W.BF16)
    sinks = W.sinks_normal(rng, Hq, 2.0)
    q = W.make_queries(rng, len(lens), Hq, 64, W.BF16)
    full = W.batch_from_pool(pool, np.arange(len(lens)), np.ones(len(lens), np.int64), q, sinks)
    k_hidden, v_hidden = full.k_cache.copy(), full.v_cache.copy()
    k_new = np.empty((len(lens), Hkv, 64), np.uint16)
    v_new = np.empty_like(k_new)
    for b, kv in enumerate(lens):
        pos = kv - 1
        phys, row = full.block_table[b, pos // 16], pos % 16
        k_new[b], v_new[b] = full.k_cache[phys, row], full.v_cache[phys, row]
        k_hidden[phys, row] = 0x7FC0  # bf16 NaN
        v_hidden[phys, row] = 0x7FC0
    hidden = W.Batch(full.dtype, full.q, k_hidden, v_hidden, full.cu_seqlens_q, full.kv_lens,
                     full.block_table, full.sinks, full.scale)
    return full, hidden, k_new, v_new


@pytest.mark.parametrize("Hkv,num_splits", [(8, 0), (8, 7), (2, 0), (6, 3), (8, -1), (6, -1)])
def test_decode_append_bf16(cuda_lib, Hkv, num_splits):
    lens = [1, 16, 17, 300, 1000, 2049, 64, 5]
    full, hidden, k_new, v_new = _hidden_last(50 + Hkv, lens, Hq=8 * Hkv, Hkv=Hkv)
    db = DeviceBatch(hidden)
    kn, vn = to_device(k_new, None), to_device(v_new, None)
    out, lse = cuda_lib.decode_append(db.q, kn, vn, db.k, db.v, db.kv_lens, db.bt, db.sinks,
                                      scale=full.scale, num_splits=num_splits, err_flag=db.err)
    torch.cuda.synchronize()
    # the appended slots now hold exactly k_new / v_new, and nothing else changed
    assert _same_bits(db.k, to_device(full.k_cache, None))
    assert _same_bits(db.v, to_device(full.v_cache, None))
    ref, ref_lse, _ = oracle_problem(full).attention()
    compare(out, lse, ref, ref_lse, what="decode+append Hkv %d S=%d" % (Hkv, num_splits))
    # the same as writing first and decoding
    o2, l2 = cuda_lib.decode(db.q, db.k, db.v, db.kv_lens, db.bt, db.sinks, scale=full.scale,
                             num_splits=num_splits, err_flag=db.err)
    assert torch.equal(out, o2) and torch.equal(lse, l2)
    assert db.err.item() == 0


def test_decode_append_bad_page_sets_flag(cuda_lib):
    full, hidden, k_new, v_new = _hidden_last(58, [40, 70])
    bt = hidden.block_table.copy()
    bt[1, 69 // 16] = hidden.k_cache.shape[0] + 5  # the appended slot's page is out of range
    bad = W.Batch(hidden.dtype, hidden.q, hidden.k_cache, hidden.v_cache, hidden.cu_seqlens_q,
                  hidden.kv_lens, bt, hidden.sinks, hidden.scale)
    db = DeviceBatch(bad)
    cuda_lib.decode_append(db.q, to_device(k_new, None), to_device(v_new, None), db.k, db.v,
                           db.kv_lens, db.bt, db.sinks, err_flag=db.err)
    torch.cuda.synchronize()
    assert db.err.item() & 1
    expect = hidden.k_cache.copy()
    expect[full.block_table[0, 39 // 16], 39 % 16] = k_new[0]  # sequence 0 was appended
    assert _same_bits(db.k, to_device(expect, None))


def test_decode_append_fp32_tiny_steps(cuda_lib):
    """Tiny fp32 workload: 4 decode steps, each appending its K/V row in the call."""
    t = W.tiny_prefill_decode()
    batch = t["prefill"]
    db = DeviceBatch(batch)
    for step in t["steps"]:
        for b in range(batch.B):
            j = int(step["positions"][b])
            phys = int(batch.block_table[b, j // batch.page_size])
            batch.k_cache[phys, j % batch.page_size] = step["new_k"][b]
            batch.v_cache[phys, j % batch.page_size] = step["new_v"][b]
        dec = W.Batch(W.FP32, step["q"], batch.k_cache, batch.v_cache,
                      np.arange(batch.B + 1, dtype=np.int32), step["kv_lens"], batch.block_table,
                      batch.sinks, batch.scale)
        ref, ref_lse, _ = oracle_problem(dec).attention()
        out, lse = cuda_lib.decode_append(torch.from_numpy(step["q"]).cuda(),
                                          torch.from_numpy(step["new_k"]).cuda(),
                                          torch.from_numpy(step["new_v"]).cuda(), db.k, db.v,
                                          torch.from_numpy(step["kv_lens"]).cuda(), db.bt, db.sinks,
                                          err_flag=db.err)
        compare(out, lse, ref, ref_lse, what="fp32 decode+append")
        assert _same_bits(db.k, torch.from_numpy(batch.k_cache).cuda())
    assert db.err.item() == 0
