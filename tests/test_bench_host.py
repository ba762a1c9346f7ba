"""Host logic of bench.py: work formulas and the multi-rank (gloo, CPU) path."""
import json
import os
import subprocess
import sys

import numpy as np

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_prefill_flops_matches_causal_pair_count():
    b = W.gptoss_prefill(num_seqs=2, q_lens=[5, 3], Hq=2, Hkv=1)
    # brute-force count of visible (query, key) pairs
    pairs = 0
    for ql, kl in zip(b.q_lens, b.kv_lens):
        for i in range(ql):
            pairs += kl - ql + i + 1
    assert bench.prefill_flops(b) == 4 * b.D * b.Hq * pairs
    # the headline prefill workload: 8 x 4096, Hq 64, D 64 -> 1.0998 TFLOP
    big = W.Batch(W.BF16, np.zeros((1, 64, 64), np.uint16), np.zeros((1, 16, 8, 64), np.uint16),
                  np.zeros((1, 16, 8, 64), np.uint16),
                  np.arange(0, 8 * 4096 + 1, 4096, dtype=np.int32), np.full(8, 4096, np.int32),
                  np.zeros((8, 256), np.int32), np.zeros(64, np.float32), 0.125)
    assert abs(bench.prefill_flops(big) / 1e12 - 1.0998) < 1e-3


def test_decode_bytes():
    b = W.gptoss_decode(num_seqs=3, kv_min=20, kv_max=40)
    kv = int(b.kv_lens.sum()) * b.Hkv * b.D * 4
    assert bench.decode_bytes(b) >= kv
    assert bench.decode_bytes(b) - kv < 3 * b.Hq * b.D * 8


def test_reference_arm_two_ranks_gloo():
    """torchrun with two CPU ranks: only rank 0 prints one JSON line."""
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=29533", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["impl"] == "reference" and res["n_gpus"] == 2 and res["value"] > 0
    assert res["cpu_baseline"]["kind"] == "oracle"


def _timing_rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import time

        def clock():
            return time.perf_counter, lambda t0: (time.perf_counter() - t0) * 1e3
        delay = 0.02 * (rank + 1)                   # rank 1 is the slow one
        calls = []

        def step():
            calls.append(1)
            time.sleep(delay)
        ms = bench.time_region(step, 3, 2, sync=lambda: None, barrier=dist.barrier,
                               reduce_max=bench.make_reduce_max(world, "cpu"), clock=clock)
        q.put((rank, ms, len(calls)))
    finally:
        dist.destroy_process_group()


def test_timed_region_max_over_two_gloo_ranks():
    """The timed region of the GPU arm (barrier on both sides, max over ranks) run
    by two CPU ranks over gloo: both ranks report the slower rank's time, and
    exactly warmup + steps calls happen per rank."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_timing_rank, args=(r, 2, 29541, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, n0), (r1, ms1, n1) = res
    assert n0 == n1 == 5
    assert ms0 == ms1                                  # the same maximum on both ranks
    assert 3 * 40 <= ms0 < 3 * 40 + 200                # rank 1's three 40 ms steps


def test_traffic_is_reported_only_for_the_captured_sources(monkeypatch):
    """A pinned ncu traffic figure holds for the kernel sources it was captured
    with: a different source hash makes the roofline report no traffic."""
    for kind, e in bench.NCU_TRAFFIC.items():
        assert e["files"] and all(f.startswith(bench.CSRC) for f in e["files"]), kind
        got = bench.ncu_traffic(kind)
        if e["sha256"] == bench.sources_sha256(e["files"]) and e["bytes"]:
            assert got == e["bytes"]
        else:
            assert got is None
    monkeypatch.setattr(bench, "sources_sha256", lambda files: "0" * 64)
    assert all(bench.ncu_traffic(k) is None for k in bench.NCU_TRAFFIC)
    assert bench.ncu_traffic("no such workload") is None
