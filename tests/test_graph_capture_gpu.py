"""The C-ABI calls read no device memory from the host and allocate nothing, so a
CUDA graph can capture them.  Replays with new inputs written in place must equal
eager calls bit for bit, and agree with the oracle."""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu import DeviceBatch, compare, oracle_problem

pytestmark = pytest.mark.gpu


def _decode_batch(seed, lens):
    rng = np.random.default_rng(seed)
    pool = W.make_pool(rng, lens, 8, 64, 16, W.BF16, fill_len=np.full(len(lens), 900))
    sinks = W.sinks_normal(rng, 64, 2.0)
    q = W.make_queries(rng, len(lens), 64, 64, W.BF16)
    return W.batch_from_pool(pool, np.arange(len(lens)), np.ones(len(lens), np.int64), q, sinks)


@pytest.mark.parametrize("num_splits", [0, -1])
def test_decode_graph_replay_matches_eager(cuda_lib, num_splits):
    """Decode captured once and replayed while the KV lengths change: the split
    plan (automatic chunks, or the persistent split's shares) is derived on the
    device at every replay."""
    gas = cuda_lib
    lens0 = np.array([700, 33, 512, 900, 1, 257], np.int64)
    batch = _decode_batch(40, lens0)
    db = DeviceBatch(batch)
    B, Hq, D = db.q.shape
    Hkv, ps = db.k.shape[2], db.k.shape[1]
    ws = torch.empty(max(256, gas.decode_workspace_size(B, Hq, Hkv, D, db.bt.shape[1], ps, num_splits)),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty_like(db.q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")

    def call():
        gas.decode(db.q, db.k, db.v, db.kv_lens, db.bt, db.sinks, scale=batch.scale, out=out,
                   lse=lse, workspace=ws, num_splits=num_splits, err_flag=db.err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # warm-up outside capture (module load, kernel attributes)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()

    rng = np.random.default_rng(41)
    for step in range(3):
        # new queries and new lengths (the pages already hold 900 keys per sequence)
        lens = rng.integers(1, 901, len(lens0))
        q = W.make_queries(rng, B, Hq, D, W.BF16)
        db.q.copy_(torch.from_numpy(q.view(np.int16)).view(torch.bfloat16).cuda())
        db.kv_lens.copy_(torch.from_numpy(lens.astype(np.int32)))
        g.replay()
        torch.cuda.synchronize()
        o_graph, l_graph = out.clone(), lse.clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(o_graph, out) and torch.equal(l_graph, lse), "replay %d differs" % step
        ref_batch = W.Batch(batch.dtype, q, batch.k_cache, batch.v_cache, batch.cu_seqlens_q,
                            lens.astype(np.int32), batch.block_table, batch.sinks, batch.scale)
        ref, ref_lse, _ = oracle_problem(ref_batch).attention()
        compare(o_graph, l_graph, ref, ref_lse, what="graph replay %d" % step)
    assert db.err.item() == 0


def test_prefill_graph_replay_matches_eager(cuda_lib):
    gas = cuda_lib
    rng = np.random.default_rng(42)
    q_lens = np.array([130, 17, 64], np.int64)
    prefix = np.array([40, 300, 0], np.int64)
    pool = W.make_pool(rng, q_lens + prefix, 8, 64, 16, W.BF16)
    sinks = W.sinks_normal(rng, 64, 2.0)
    q = W.make_queries(rng, int(q_lens.sum()), 64, 64, W.BF16)
    batch = W.batch_from_pool(pool, np.arange(3), q_lens, q, sinks)
    db = DeviceBatch(batch)
    out = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device="cuda")
    # One workspace for the eager calls and the replays: the call's memset node
    # restarts the tile-claim counter on every replay.
    wsb = torch.empty(gas.prefill_workspace_size(batch.B, batch.Hq, batch.D, int(q_lens.max())),
                      dtype=torch.uint8, device="cuda")

    def call():
        gas.prefill(db.q, db.k, db.v, db.cu, db.kv_lens, db.bt, db.sinks, max_q_len=int(q_lens.max()),
                    scale=batch.scale, out=out, lse=lse, workspace=wsb, err_flag=db.err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for step in range(2):
        q2 = W.make_queries(rng, int(q_lens.sum()), 64, 64, W.BF16)
        db.q.copy_(torch.from_numpy(q2.view(np.int16)).view(torch.bfloat16).cuda())
        g.replay()
        torch.cuda.synchronize()
        o_graph, l_graph = out.clone(), lse.clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(o_graph, out) and torch.equal(l_graph, lse), "replay %d differs" % step
        ref_batch = W.Batch(batch.dtype, q2, batch.k_cache, batch.v_cache, batch.cu_seqlens_q,
                            batch.kv_lens, batch.block_table, batch.sinks, batch.scale)
        ref, ref_lse, _ = oracle_problem(ref_batch).attention()
        compare(o_graph, l_graph, ref, ref_lse, what="prefill graph replay %d" % step)
    assert db.err.item() == 0


def test_mixed_graph_replay_matches_eager(cuda_lib):
    """attn_sink_mixed captured in a CUDA graph: its memset node restarts both claim
    counters, so replays with new queries equal eager calls bitwise."""
    gas = cuda_lib
    rng = np.random.default_rng(43)
    dec_kv = np.array([1500, 40, 3000], np.int64)
    pre_q, pre_prefix = np.array([100, 33], np.int64), np.array([200, 0], np.int64)
    kv = np.concatenate([dec_kv, pre_q + pre_prefix])
    pool = W.make_pool(rng, kv, 8, 64, 16, W.BF16)
    sinks = W.sinks_normal(rng, 64, 2.0)
    q_lens = np.concatenate([np.ones(3, np.int64), pre_q])
    q = W.make_queries(rng, int(q_lens.sum()), 64, 64, W.BF16)
    batch = W.batch_from_pool(pool, np.arange(5), q_lens, q, sinks)
    db = DeviceBatch(batch)
    out = torch.empty_like(db.q)
    lse = torch.empty(db.q.shape[:2], dtype=torch.float32, device="cuda")
    wsb = torch.empty(gas.mixed_workspace_size(3, 64, 8, 64, batch.block_table.shape[1], 16),
                      dtype=torch.uint8, device="cuda")

    def call():
        gas.mixed(db.q, db.k, db.v, db.cu, db.kv_lens, db.bt, db.sinks, num_decode=3, max_q_len=100,
                  scale=batch.scale, out=out, lse=lse, workspace=wsb, err_flag=db.err)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    for step in range(2):
        q2 = W.make_queries(rng, int(q_lens.sum()), 64, 64, W.BF16)
        db.q.copy_(torch.from_numpy(q2.view(np.int16)).view(torch.bfloat16).cuda())
        g.replay()
        torch.cuda.synchronize()
        o_graph, l_graph = out.clone(), lse.clone()
        call()
        torch.cuda.synchronize()
        assert torch.equal(o_graph, out) and torch.equal(l_graph, lse), "replay %d differs" % step
        ref_batch = W.Batch(batch.dtype, q2, batch.k_cache, batch.v_cache, batch.cu_seqlens_q,
                            batch.kv_lens, batch.block_table, batch.sinks, batch.scale)
        ref, ref_lse, _ = oracle_problem(ref_batch).attention()
        compare(o_graph, l_graph, ref, ref_lse, what="mixed graph replay %d" % step)
    assert db.err.item() == 0
