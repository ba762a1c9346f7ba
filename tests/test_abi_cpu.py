"""The C-ABI library builds, loads without a GPU and exports every symbol that
include/attn_sink.h declares; host-side argument checks reject bad calls before
any CUDA work (no GPU needed, no compute call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "attn_sink.h")).read()
    return sorted(set(re.findall(r"ATTN_SINK_API\s+[\w\s\*]+?\b(attn_sink_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from gqa_attention_sinks_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_entry_points():
    names = _declared()
    for n in ("attn_sink_prefill", "attn_sink_decode", "attn_sink_merge",
              "attn_sink_decode_workspace_size", "attn_sink_prefill_workspace_size",
              "attn_sink_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_signatures_cover_header():
    import gqa_attention_sinks_gb300 as gas
    assert sorted(gas.SIGNATURES) == _declared()


def test_wait_limit_hook_is_host_only(lib):
    """The test hook for the timeout path only stores a value: it returns the
    previous limit, and 0 restores the default of one second."""
    f = lib.attn_sink_set_wait_limit_ns
    f.argtypes = [ctypes.c_uint64]
    f.restype = ctypes.c_uint64
    first = f(12345)
    try:
        assert f(0) == 12345
        assert f(0) == 1_000_000_000
    finally:
        f(first)


def test_status_strings(lib):
    f = lib.attn_sink_status_string
    f.restype = ctypes.c_char_p
    assert f(0) == b"ok"
    assert b"invalid" in f(1) and b"unsupported" in f(2) and b"workspace" in f(3)


def test_workspace_size_is_host_only(lib):
    f = lib.attn_sink_decode_workspace_size
    f.restype = ctypes.c_size_t
    # fixed split: rows * S * 64 fp32 + rows * S fp32, each rounded up to 256 B
    rows, S = 4 * 64, 32
    expect = -(-rows * S * 64 * 4 // 256) * 256 + -(-rows * S * 4 // 256) * 256
    assert f(4, 64, 8, 64, 8192, 16, S) == expect
    assert f(4, 64, 8, 64, 8192, 16, 1) == 0
    assert f(4, 64, 8, 64, 8192, 16, 0) > 0
    assert f(4, 64, 8, 32, 8192, 16, 0) == 0       # unsupported head dim


def _call_decode(lib, **kw):
    # Fake, 256-aligned addresses: every call below is rejected by the host
    # checks before anything touches them.
    args = dict(q=256, k=512, v=768, kv=1024, bt=1280, stride=4, sinks=1536, out=1792, lse=None, B=2, Hq=8,
                Hkv=2, D=64, ps=16, pages=8, scale=0.125, S=0, dt=0, err=None, ws=None, wsb=0,
                stream=None)
    args.update(kw)
    f = lib.attn_sink_decode
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [vp] * 5 + [i32, vp, vp, vp] + [i32] * 6 + [ctypes.c_float, i32, i32, vp, vp,
                                                            ctypes.c_size_t, vp]
    f.restype = i32
    a = args
    return f(a["q"], a["k"], a["v"], a["kv"], a["bt"], a["stride"], a["sinks"], a["out"], a["lse"],
             a["B"], a["Hq"], a["Hkv"], a["D"], a["ps"], a["pages"], a["scale"], a["S"], a["dt"],
             a["err"], a["ws"], a["wsb"], a["stream"])


def test_host_validation_rejects_before_launch(lib):
    # Only argument checks run for these calls; the pointers are never dereferenced.
    assert _call_decode(lib, q=None) == 1                      # null pointer
    assert _call_decode(lib, Hq=6, Hkv=4) == 1                 # Hq % Hkv != 0
    assert _call_decode(lib, D=128) == 2                       # unsupported head dim
    assert _call_decode(lib, ps=8) == 2                        # bf16 needs page_size % 16 == 0
    assert _call_decode(lib, Hq=64, Hkv=2) == 2                # group 32 unsupported
    assert _call_decode(lib, q=256 + 4) == 1                   # misaligned q
    assert _call_decode(lib, S=300) == 1                       # too many splits
    assert _call_decode(lib, S=-2) == 1                        # (-1 is the persistent split)
    assert _call_decode(lib, scale=float("nan")) == 1
    assert _call_decode(lib, S=4, ws=None, wsb=0) == 3         # missing workspace
    assert _call_decode(lib, S=4, ws=256 + 16, wsb=1 << 20) == 3   # misaligned workspace
    assert _call_decode(lib, B=0) == 0                         # empty batch is a no-op


def test_prefill_workspace_size_is_host_only(lib):
    f = lib.attn_sink_prefill_workspace_size
    f.argtypes = [ctypes.c_int32] * 4
    f.restype = ctypes.c_size_t
    assert f(8, 64, 64, 4096) == 256          # the work-tile claim counter
    assert f(0, 64, 64, 4096) == 0            # nothing to do
    assert f(8, 64, 64, 0) == 0
    assert f(8, 64, 128, 4096) == 0           # unsupported head dim


def _call_prefill(lib, **kw):
    # Fake, 256-aligned addresses: every call below is rejected by the host
    # checks before anything touches them.
    args = dict(q=256, k=512, v=768, cu=1024, kv=1280, bt=1536, stride=4, sinks=1792, out=2048,
                lse=None, B=2, total_q=8, max_q=4, Hq=8, Hkv=2, D=64, ps=16, pages=8, scale=0.125,
                causal=1, dt=0, err=None, ws=4096, wsb=256, stream=None)
    args.update(kw)
    f = lib.attn_sink_prefill
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [vp] * 6 + [i32, vp, vp, vp] + [i32] * 8 + [ctypes.c_float, i32, i32, vp, vp,
                                                              ctypes.c_size_t, vp]
    f.restype = i32
    a = args
    return f(a["q"], a["k"], a["v"], a["cu"], a["kv"], a["bt"], a["stride"], a["sinks"], a["out"],
             a["lse"], a["B"], a["total_q"], a["max_q"], a["Hq"], a["Hkv"], a["D"], a["ps"],
             a["pages"], a["scale"], a["causal"], a["dt"], a["err"], a["ws"], a["wsb"], a["stream"])


def test_prefill_host_validation_rejects_before_launch(lib):
    assert _call_prefill(lib, q=None) == 1                     # null pointer
    assert _call_prefill(lib, causal=2) == 1
    assert _call_prefill(lib, D=128) == 2                      # unsupported head dim
    assert _call_prefill(lib, ws=None, wsb=0) == 3             # bf16 needs the workspace
    assert _call_prefill(lib, wsb=128) == 3                    # too small
    assert _call_prefill(lib, ws=4096 + 64) == 3               # misaligned
    assert _call_prefill(lib, B=0) == 0                        # empty batch is a no-op
    assert _call_prefill(lib, max_q=0, ws=None, wsb=0) == 0    # no rows: nothing to do


def test_static_scratch_checks_arguments_like_decode(lib):
    """Bad calls get the same status from the static-scratch entry point as from
    attn_sink_decode: argument errors come before the scratch-size check."""
    f = lib.attn_sink_decode_static_scratch
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [vp] * 5 + [i32, vp, vp, vp] + [i32] * 6 + [ctypes.c_float, i32, i32, vp, vp]
    f.restype = i32

    def call(**kw):
        a = dict(q=256, k=512, v=768, kv=1024, bt=1280, stride=4096, sinks=1536, out=1792,
                 lse=None, B=512, Hq=64, Hkv=8, D=64, ps=16, pages=8, scale=0.125, S=0, dt=0,
                 err=None, stream=None)
        a.update(kw)
        return f(a["q"], a["k"], a["v"], a["kv"], a["bt"], a["stride"], a["sinks"], a["out"],
                 a["lse"], a["B"], a["Hq"], a["Hkv"], a["D"], a["ps"], a["pages"], a["scale"],
                 a["S"], a["dt"], a["err"], a["stream"])

    same = dict(B=512, Hq=64, Hkv=8, stride=4096)
    for kw in (dict(S=300), dict(Hq=60), dict(q=None), dict(D=128), dict(scale=float("inf"))):
        args = dict(same, **kw)
        assert call(**args) == _call_decode(lib, **args), kw
    assert call(S=300) == 1 and call(D=128) == 2
    assert call() == 3                    # valid, but its partials exceed the static array
    assert call(B=0) == 0


def _call_mixed(lib, **kw):
    # Fake, 256-aligned addresses: every call below is rejected by the host
    # checks before anything touches them.
    args = dict(q=256, k=512, v=768, cu=1024, kv=1280, bt=1536, stride=4, sinks=1792, out=2048,
                lse=None, B=4, nd=2, total_q=8, max_q=4, Hq=8, Hkv=2, D=64, ps=16, pages=8,
                scale=0.125, causal=1, dt=0, err=None, ws=4096, wsb=1 << 20, stream=None)
    args.update(kw)
    f = lib.attn_sink_mixed
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    f.argtypes = [vp] * 6 + [i32, vp, vp, vp] + [i32] * 9 + [ctypes.c_float, i32, i32, vp, vp,
                                                              ctypes.c_size_t, vp]
    f.restype = i32
    a = args
    return f(a["q"], a["k"], a["v"], a["cu"], a["kv"], a["bt"], a["stride"], a["sinks"], a["out"],
             a["lse"], a["B"], a["nd"], a["total_q"], a["max_q"], a["Hq"], a["Hkv"], a["D"],
             a["ps"], a["pages"], a["scale"], a["causal"], a["dt"], a["err"], a["ws"], a["wsb"],
             a["stream"])


def test_mixed_host_validation_and_workspace_size(lib):
    size = lib.attn_sink_mixed_workspace_size
    size.argtypes = [ctypes.c_int32] * 6
    size.restype = ctypes.c_size_t
    # counters, plus num_decode * Hq rows of partials when a row can span several
    # 1024-key items (8192-key table rows: 8 slots)
    rows, slots = 48 * 64, 8
    parts = -(-rows * slots * 64 * 4 // 256) * 256 + -(-rows * slots * 4 // 256) * 256
    assert size(48, 64, 8, 64, 512, 16) == 256 + parts
    assert size(48, 64, 8, 64, 64, 16) == 256          # one item per row: no partials
    assert size(48, 64, 8, 128, 512, 16) == 0          # unsupported head dim
    assert _call_mixed(lib, nd=5) == 1                 # num_decode > B
    assert _call_mixed(lib, nd=-1) == 1
    assert _call_mixed(lib, q=None) == 1
    assert _call_mixed(lib, D=128) == 2
    assert _call_mixed(lib, B=1025, nd=0) == 2         # bf16: the sequences must fit shared memory
    assert _call_mixed(lib, Hq=512, Hkv=32) == 2
    assert _call_mixed(lib, ws=None, wsb=0) == 3       # bf16 needs the workspace
    assert _call_mixed(lib, ws=4096 + 64) == 3         # misaligned
    assert _call_mixed(lib, B=0, nd=0) == 0            # empty batch is a no-op
