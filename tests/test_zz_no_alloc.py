"""attn_sink_decode_static_scratch: the decode entry point for callers that
cannot allocate device memory (their allocator owns all device memory, or
cudaMalloc's implicit synchronisation is not acceptable on their path).

It must give the same result as attn_sink_decode with a caller-provided
workspace, call after call, using only its library-owned static scratch.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from _gpu import DeviceBatch, MAX_ABS, MEAN_ABS, LSE_ABS

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 32 << 20  # ATTN_SINK_STATIC_SCRATCH_BYTES in include/attn_sink.h


def _static_decode(lib, db, num_splits, out, lse):
    b = db.b
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.attn_sink_decode_static_scratch(
        p(db.q), p(db.k), p(db.v), p(db.kv_lens), p(db.bt), db.bt.shape[1], p(db.sinks), p(out),
        p(lse), b.B, b.Hq, b.Hkv, b.D, b.page_size, b.num_pages, b.scale, num_splits, 0,
        p(db.err), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("num_splits", [0, 32])
def test_static_scratch_matches_workspace_decode(cuda_lib, num_splits):
    lib = cuda_lib.load()
    batch = W.gptoss_decode(num_seqs=12, kv_min=300, kv_max=5000)
    db = DeviceBatch(batch)
    need = cuda_lib.decode_workspace_size(batch.B, batch.Hq, batch.Hkv, batch.D,
                                          batch.block_table.shape[1], batch.page_size, num_splits)
    assert 0 < need <= STATIC_SCRATCH_BYTES            # the split path really uses scratch
    ref, ref_lse = cuda_lib.decode(db.q, db.k, db.v, db.kv_lens, db.bt, db.sinks,
                                   scale=batch.scale, num_splits=num_splits, err_flag=db.err)
    torch.cuda.synchronize()
    for call in range(2):                              # two calls in a row share the scratch
        out = torch.full_like(ref, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = _static_decode(lib, db, num_splits, out, lse)
        torch.cuda.synchronize()
        assert st == 0, cuda_lib.status_string(st)
        err = (out.float() - ref.float()).abs()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, call
        assert (lse - ref_lse).abs().max().item() <= LSE_ABS, call
    assert db.err.item() == 0


def test_static_scratch_rejects_oversize(cuda_lib):
    """A call whose partials exceed the static array is refused before any launch."""
    lib = cuda_lib.load()
    B, Hq, Hkv, stride = 512, 64, 8, 4096          # 512*64 rows x 128 chunks of fp32 partials
    need = cuda_lib.decode_workspace_size(B, Hq, Hkv, 64, stride, 16, 0)
    assert need > STATIC_SCRATCH_BYTES
    # Real buffers with every kv_len = 0, so even a launch would read no keys.
    q = torch.zeros((B, Hq, 64), dtype=torch.bfloat16, device="cuda")
    cache = torch.zeros((1, 16, Hkv, 64), dtype=torch.bfloat16, device="cuda")
    kv_lens = torch.zeros(B, dtype=torch.int32, device="cuda")
    bt = torch.zeros((B, stride), dtype=torch.int32, device="cuda")
    sinks = torch.zeros(Hq, dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.attn_sink_decode_static_scratch(
        p(q), p(cache), p(cache), p(kv_lens), p(bt), stride, p(sinks), p(out), None, B, Hq, Hkv,
        64, 16, 1, 0.125, 0, 0, None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 3                                     # ATTN_SINK_ERR_WORKSPACE
