"""The failure path of the bounded pipeline waits, exercised on the GPU without
a fault: with the wait limit lowered to 1 ns the kernels' first pending waits
give up, so a correct call must come back with ATTN_SINK_FLAG_TIMEOUT set; the
context must then still run the same call correctly once the limit is back."""
import numpy as np
import pytest
import torch

import workloads as W
from _gpu import DeviceBatch, compare, oracle_problem

pytestmark = pytest.mark.gpu


def _prefill(gas, db):
    b = db.b
    return gas.prefill(db.q, db.k, db.v, db.cu, db.kv_lens, db.bt, db.sinks,
                       max_q_len=b.max_q_len, scale=b.scale, causal=True, err_flag=db.err)


def _decode(gas, db):
    return gas.decode(db.q, db.k, db.v, db.kv_lens, db.bt, db.sinks, scale=db.b.scale,
                      num_splits=4, err_flag=db.err)


def _decode_persistent(gas, db):
    return gas.decode(db.q, db.k, db.v, db.kv_lens, db.bt, db.sinks, scale=db.b.scale,
                      num_splits=gas.SPLIT_PERSISTENT, err_flag=db.err)


def _mixed(gas, db):
    b = db.b
    nd = b.meta["n_decode"]
    return gas.mixed(db.q, db.k, db.v, db.cu, db.kv_lens, db.bt, db.sinks, num_decode=nd,
                     max_q_len=int(b.q_lens[nd:].max()), scale=b.scale, err_flag=db.err)


@pytest.mark.parametrize("kind", ["prefill", "decode", "decode_persistent", "mixed"])
def test_timeout_flag_then_context_still_usable(cuda_lib, kind):
    if kind == "prefill":
        batch = W.gptoss_prefill(seed=20260103, num_seqs=2, seq_len=1024)
        run = _prefill
    elif kind == "mixed":
        batch = W.mixed_batch(seed=20260105, n_decode=6, decode_kv=(1000, 3000), n_prefill=2,
                              prefill_new=100, prefix=(0, 500))["single"]
        run = _mixed
    else:
        batch = W.gptoss_decode(seed=20260102, num_seqs=16)
        run = _decode if kind == "decode" else _decode_persistent
    db = DeviceBatch(batch)
    previous = cuda_lib.set_wait_limit_ns(1)
    try:
        run(cuda_lib, db)
        torch.cuda.synchronize()
        flags = db.err.item()
    finally:
        cuda_lib.set_wait_limit_ns(previous)
    assert flags & cuda_lib.FLAG_TIMEOUT, flags
    assert not flags & cuda_lib.FLAG_BAD_PAGE, flags

    db.err.zero_()
    out, lse = run(cuda_lib, db)
    torch.cuda.synchronize()
    assert db.err.item() == 0, db.err.item()
    if kind == "prefill":
        rows = W.sample_rows(np.random.default_rng(5), batch, 256)
        ref, ref_lse, _ = oracle_problem(batch).attention(rows)
        compare(out, lse, ref, ref_lse, rows=rows, what="prefill after a timed-out call")
    else:
        ref, ref_lse, _ = oracle_problem(batch).attention()
        compare(out, lse, ref, ref_lse, what="%s after a timed-out call" % kind)
