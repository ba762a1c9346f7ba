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
