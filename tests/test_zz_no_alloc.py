"""attn_sink_decode_static_scratch: the decode entry point for callers that
cannot allocate device memory (their allocator owns all device memory, or
cudaMalloc's implicit synchronisation is not acceptable on their path).

It must give exactly the result of attn_sink_decode with a caller-provided
workspace (the same kernels on the same inputs), call after call, using only
its library-owned static scratch, which keeps the previous call's contents.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W
from _gpu import DeviceBatch

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 32 << 20  # ATTN_SINK_STATIC_SCRATCH_BYTES in include/attn_sink.h


def _static_decode(lib, db, num_splits, out, lse, dtype_code):
    b = db.b
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.attn_sink_decode_static_scratch(
        p(db.q), p(db.k), p(db.v), p(db.kv_lens), p(db.bt), db.bt.shape[1], p(db.sinks), p(out),
        p(lse), b.B, b.Hq, b.Hkv, b.D, b.page_size, b.num_pages, b.scale, num_splits, dtype_code,
        p(db.err), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _check_same_as_workspace_decode(gas, db, num_splits, dtype_code):
    """One static-scratch call against attn_sink_decode with a fresh workspace:
    bitwise equal outputs and lse."""
    lib = gas.load()
    ref, ref_lse = gas.decode(db.q, db.k, db.v, db.kv_lens, db.bt, db.sinks, scale=db.b.scale,
                              num_splits=num_splits, err_flag=db.err)
    out = torch.full_like(ref, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    st = _static_decode(lib, db, num_splits, out, lse, dtype_code)
    torch.cuda.synchronize()
    assert st == 0, gas.status_string(st)
    assert torch.equal(out, ref), (out.float() - ref.float()).abs().max().item()
    assert torch.equal(lse, ref_lse)
    assert db.err.item() == 0


@pytest.mark.parametrize("num_splits", [0, 32])
def test_static_scratch_matches_workspace_decode(cuda_lib, num_splits):
    """A large call, then a smaller, different one: the second call's partials
    land over the first call's leftovers in the shared array and must still
    give exactly the workspace result (its rows include kv_len 0 and 1, an
    exact page boundary and a -inf sink)."""
    big = W.gptoss_decode(num_seqs=12, kv_min=300, kv_max=5000)
    need = cuda_lib.decode_workspace_size(big.B, big.Hq, big.Hkv, big.D,
                                          big.block_table.shape[1], big.page_size, num_splits)
    assert 0 < need <= STATIC_SCRATCH_BYTES            # the split path really uses scratch
    small = W.gptoss_decode(seed=77, num_seqs=5, kv_min=100, kv_max=900)
    small.kv_lens[:3] = [0, 1, 256]
    small.sinks[:8] = -np.inf
    for batch in (big, small, big):
        _check_same_as_workspace_decode(cuda_lib, DeviceBatch(batch), num_splits, 0)


@pytest.mark.parametrize("num_splits", [0, 8])
def test_static_scratch_fp32(cuda_lib, num_splits):
    """The fp32 path: num_splits 0 runs unsplit (no scratch), 8 writes fp32
    partials to the static array."""
    t = W.tiny_prefill_decode()
    pre = t["prefill"]
    step = t["steps"][0]
    pre.kv_lens[:] = 64
    dec = W.Batch(W.FP32, step["q"], pre.k_cache, pre.v_cache,
                  np.arange(pre.B + 1, dtype=np.int32), pre.kv_lens.copy(), pre.block_table,
                  pre.sinks, pre.scale)
    for _ in range(2):
        _check_same_as_workspace_decode(cuda_lib, DeviceBatch(dec), num_splits, 1)


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
