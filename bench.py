"""Benchmark: sink GQA attention on GB300 (decode HBM GB/s, prefill TFLOP/s).

Default (N=1): one JSON line.  Its headline workload is gpt-oss-shaped paged
decode (64 seqs, Hq 64, Hkv 8, D 64, KV lengths uniform in [512, 8192], page
size 16, bf16).  A step is one decode call: the split-KV kernel plus the LSE
merge, through the C ABI; value = algorithmic K/V bytes per step / device
time per step.  The other workloads are timed the same way and reported as
sub-objects, each with its own roofline and CPU-oracle baseline:
  "prefill"  8 x 4096 causal prefill, ragged layout (TFLOP/s of the causal half)
  "long"     4 x 131072-key decode split into 32 chunks (GB/s)
  "mixed"    48 decode seqs (KV 1k..32k) + 4 x 512-token chunked prefills over
             prefixes up to 16k, 1% outlier keys: the decode part (GB/s) and the
             chunked-prefill part (TFLOP/s), each against its own roofline, and
             the whole batch as one attn_sink_mixed launch ("one_launch")

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload all|decode|prefill|long|mixed] [--no-cpu-baseline]

Multi-GPU (torchrun): every rank runs its own replica of the workload with a
rank-specific seed (weak scaling, no collective on the data path); timing is
the max over ranks.  --impl reference times the fp64 CPU oracle on the host
cores over a bounded sample of the headline workload.
"""
import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "sink-GQA attn: decode HBM GB/s & prefill TFLOP/s, % of GB300 roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of the
# dominant kernel of a workload, from the ncu captures summarised in profiles/.  A
# value holds only for the kernel sources it was captured with (sha256 over the
# listed files); after any change to them the roofline reports traffic = null.
CSRC = "gqa_attention_sinks_gb300/csrc/"
PREFILL_SOURCES = [CSRC + f for f in ("prefill_bf16.cu", "tcgen05.cuh", "ptx.cuh", "kernels.h",
                                      "decode_unit.cuh")]
DECODE_SOURCES = [CSRC + f for f in ("decode_bf16.cu", "ptx.cuh", "kernels.h", "api.cu",
                                     "decode_unit.cuh")]
NCU_TRAFFIC = {
    # prefill_kernel, 8 x 4096 causal prefill
    "prefill": {"files": PREFILL_SOURCES,
                "sha256": "dc6ed89ce508011f2a9b1d313a3cd31b0af19e29b2627eed5da828007bf18104", "bytes": 557558272},
    # decode_split_kernel, gpt-oss decode (64 seqs)
    "decode": {"files": DECODE_SOURCES,
               "sha256": "d5359e965e705dc861d4b523f8eb32a6d2cb78e9cb8da3267774bc3ca019f032", "bytes": 582872832},
    # decode_split_kernel, long split decode (4 x 131072 keys, 32 chunks)
    "long": {"files": DECODE_SOURCES, "sha256": "d5359e965e705dc861d4b523f8eb32a6d2cb78e9cb8da3267774bc3ca019f032", "bytes": 1074084864},
    # decode_split_kernel, the mixed batch's decode part
    "mixed_decode": {"files": DECODE_SOURCES, "sha256": "d5359e965e705dc861d4b523f8eb32a6d2cb78e9cb8da3267774bc3ca019f032", "bytes": 1647429376},
    # prefill_kernel, the mixed batch's chunked-prefill part
    "mixed_prefill": {"files": PREFILL_SOURCES, "sha256": "dc6ed89ce508011f2a9b1d313a3cd31b0af19e29b2627eed5da828007bf18104", "bytes": 69377024},
}


def sources_sha256(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def ncu_traffic(kind):
    e = NCU_TRAFFIC.get(kind)
    if not e or not e["bytes"] or sources_sha256(e["files"]) != e["sha256"]:
        return None
    return e["bytes"]


# ----------------------------------------------------------------- helpers
def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def decode_bytes(batch):
    """Algorithmic HBM bytes of one decode step: every K and V row once per KV head,
    plus q, out (bf16), lse (fp32) and the block table entries read."""
    kv = batch.kv_tokens() * batch.Hkv * batch.D * 2 * 2
    io = batch.B * batch.Hq * batch.D * 2 * 2 + batch.B * batch.Hq * 4
    pages = int(np.sum((batch.kv_lens.astype(np.int64) + batch.page_size - 1) // batch.page_size)) * 4
    return kv + io + pages


def visible_pairs(batch, rows=None):
    """(query row, key) pairs the rows see (all rows of the batch when rows is None)."""
    q = batch.q_lens.astype(np.int64)
    kv = batch.kv_lens.astype(np.int64)
    if rows is None:
        pairs = 0
        for ql, kl in zip(q, kv):
            if batch.causal:
                first = kl - ql + 1                   # keys seen by the first query
                pairs += ql * first + ql * (ql - 1) // 2
            else:
                pairs += ql * kl
        return int(pairs) * batch.Hq
    tok = np.asarray(rows, np.int64) // batch.Hq
    seq = np.searchsorted(batch.cu_seqlens_q, tok, side="right") - 1
    i = tok - batch.cu_seqlens_q[seq]
    pos = kv[seq] - q[seq] + i
    seen = np.clip(pos + 1, 0, kv[seq]) if batch.causal else kv[seq]
    return int(seen.sum())


def prefill_flops(batch):
    """Algorithmic FLOPs of causal prefill: 4*D per visible (query row, key) pair."""
    return 4 * batch.D * visible_pairs(batch)


def time_region(fn, steps, warmup, *, sync, barrier, reduce_max, clock):
    """Runs `warmup` untimed steps, then times exactly `steps` steps bracketed by
    sync + barrier + sync on both sides; returns the maximum over ranks (ms).
    clock() returns (start, stop) callables; stop(start_token) gives ms."""
    for _ in range(warmup):
        fn()
    sync()
    barrier()
    sync()
    start, stop = clock()
    tok = start()
    for _ in range(steps):
        fn()
    ms = stop(tok)
    sync()
    barrier()
    return reduce_max(ms)


def make_reduce_max(ws, device):
    """Max of a float over the ranks of the default process group (identity at N=1)."""
    def reduce_max(x):
        if ws == 1:
            return float(x)
        import torch
        import torch.distributed as dist
        t = torch.tensor([float(x)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return reduce_max


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while work runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), "attn_sink_bench_clocks_%d.csv" % os.getpid())

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 7:
                try:
                    rows.append((float(parts[0]), float(parts[1]), parts[2:]))
                except ValueError:
                    pass
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i in range(4) if r[i + 1] == "Active"})
        sm = [r[0] for r in rows]
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r[1] for r in rows),
                "samples": len(rows), "reasons": reasons}


# ----------------------------------------------------------------- CPU oracle
def cpu_oracle_rate(batch, seconds, unit, rng_seed=7):
    """Time the fp64 oracle on the host cores over a bounded sample of the batch.

    Decode-like batches (one query per sequence) are sampled by whole sequences,
    in order, and rated in GB/s of algorithmic K/V bytes; prefill batches by
    random query tokens (all heads) in groups of 64, rated in TFLOP/s of the
    algorithmic 4*D FLOPs per visible (row, key) pair.  Runs about `seconds`."""
    import oracle
    prob = oracle.Problem(batch.q, batch.k_cache, batch.v_cache, batch.cu_seqlens_q,
                          batch.kv_lens, batch.block_table, batch.sinks, batch.scale, batch.causal)
    rng = np.random.default_rng(rng_seed)
    work, elapsed, units = 0, 0.0, 0
    b = 0
    while elapsed < seconds and units < 100000:
        if unit == "GB/s":
            rows = np.arange(batch.cu_seqlens_q[b] * batch.Hq, batch.cu_seqlens_q[b + 1] * batch.Hq)
            w = visible_pairs(batch, rows) * batch.D * 2 * 2 // (batch.Hq // batch.Hkv)
            b = (b + 1) % batch.B
            units += 1
        else:
            toks = rng.choice(batch.total_q, size=min(64, batch.total_q), replace=False)
            rows = (toks[:, None] * batch.Hq + np.arange(batch.Hq)[None, :]).reshape(-1)
            w = 4 * batch.D * visible_pairs(batch, rows)
            units += len(toks)
        t0 = time.perf_counter()
        prob.attention(rows)
        elapsed += time.perf_counter() - t0
        work += w
    value = work / elapsed / (1e9 if unit == "GB/s" else 1e12)
    what = ("%d whole sequences (all heads)" % units if unit == "GB/s"
            else "%d random query tokens (all heads)" % units)
    return {"value": round(value, 4), "unit": unit, "cores": oracle.max_threads(),
            "kind": "oracle", "sample": "%s, %.1f s of fp64 oracle time" % (what, elapsed)}


# ----------------------------------------------------------------- GPU arm
class GpuArm:
    def __init__(self, args, ws, rank, local):
        import torch
        import gqa_attention_sinks_gb300 as gas
        self.torch, self.gas = torch, gas
        self.args, self.ws, self.rank, self.local = args, ws, rank, local
        torch.cuda.set_device(local)
        gas.load()
        self.dev = torch.device("cuda", local)
        self.stream = torch.cuda.current_stream()
        self.pk, self.pk_kind = peaks()
        self.reduce_max = make_reduce_max(ws, self.dev)
        self.seed_off = 1000 * rank

    # -- plumbing
    def to_dev(self, a):
        torch = self.torch
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(self.dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def pinned(self, a):
        torch = self.torch
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                             else np.ascontiguousarray(a))
        t = t.pin_memory()
        return t.view(torch.bfloat16) if a.dtype == np.uint16 else t

    def barrier(self):
        if self.ws > 1:
            self.torch.distributed.barrier()

    def event_clock(self):
        torch, stream = self.torch, self.stream

        def start():
            e = torch.cuda.Event(enable_timing=True)
            e.record(stream)
            return e

        def stop(e0):
            e1 = torch.cuda.Event(enable_timing=True)
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)
        return start, stop

    def timed(self, fn, steps, warmup):
        """Total ms of `steps` back-to-back calls (max over ranks)."""
        return time_region(fn, steps, warmup, sync=self.torch.cuda.synchronize,
                           barrier=self.barrier, reduce_max=self.reduce_max,
                           clock=self.event_clock)

    def per_call(self, fn, steps):
        """Mean device time of one call, each call bracketed by its own events."""
        torch, stream = self.torch, self.stream
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in evs:
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs]))

    def with_clocks(self, run):
        sampler = ClockSampler(self.local)
        sampler.start()
        try:
            out = run()
        finally:
            clocks = sampler.stop()
        return out, clocks

    def warm_clock(self, fn):
        t_end = time.time() + self.args.clock_window   # load the GPU while sampling starts
        while time.time() < t_end:
            fn()
            self.torch.cuda.synchronize()

    # -- the calls
    def decode_step(self, batch, splits):
        torch, gas = self.torch, self.gas
        d = dict(q=self.to_dev(batch.q), k=self.to_dev(batch.k_cache), v=self.to_dev(batch.v_cache),
                 kvl=self.to_dev(batch.kv_lens), bt=self.to_dev(batch.block_table),
                 sinks=self.to_dev(batch.sinks))
        d["out"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=self.dev)
        need = gas.decode_workspace_size(batch.B, batch.Hq, batch.Hkv, batch.D,
                                         batch.block_table.shape[1], batch.page_size, splits)
        d["ws"] = torch.empty(max(need, 256), dtype=torch.uint8, device=self.dev)
        d["launches"] = 2 if need > 0 else 1

        def step():
            gas.decode(d["q"], d["k"], d["v"], d["kvl"], d["bt"], d["sinks"], scale=batch.scale,
                       num_splits=splits, out=d["out"], lse=d["lse"], workspace=d["ws"])
        return step, d

    def prefill_step(self, batch):
        torch, gas = self.torch, self.gas
        d = dict(q=self.to_dev(batch.q), k=self.to_dev(batch.k_cache), v=self.to_dev(batch.v_cache),
                 cu=self.to_dev(batch.cu_seqlens_q), kvl=self.to_dev(batch.kv_lens),
                 bt=self.to_dev(batch.block_table), sinks=self.to_dev(batch.sinks))
        d["out"] = torch.empty_like(d["q"])
        d["lse"] = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=self.dev)
        need = gas.prefill_workspace_size(batch.B, batch.Hq, batch.D, batch.max_q_len)
        d["ws"] = torch.empty(max(need, 256), dtype=torch.uint8, device=self.dev)

        def step():
            gas.prefill(d["q"], d["k"], d["v"], d["cu"], d["kvl"], d["bt"], d["sinks"],
                        max_q_len=batch.max_q_len, scale=batch.scale, out=d["out"], lse=d["lse"],
                        workspace=d["ws"])
        return step, d

    # -- parts
    def hbm_roofline(self, nbytes, call_ms, traffic_kind, kernel):
        ach = nbytes / (call_ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": self.pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / self.pk["hbm_gbs"], 4),
                "traffic": ncu_traffic(traffic_kind) if traffic_kind else None,
                "peak_source": self.pk_kind, "kernel": kernel}

    def tensor_roofline(self, flops, call_ms, traffic_kind):
        ach = flops / (call_ms * 1e-3) / 1e12
        peak = self.pk["bf16_tflops"]
        return {"bound": "tensor", "achieved": round(ach, 2), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4),
                "traffic": ncu_traffic(traffic_kind) if traffic_kind else None,
                "peak_source": self.pk_kind, "kernel": "prefill_kernel (tcgen05, one launch)"}

    def decode_part(self, batch, splits, name, steps, traffic_kind):
        step, d = self.decode_step(batch, splits)
        nbytes = decode_bytes(batch)

        def run():
            self.warm_clock(step)
            total = self.timed(step, steps, self.args.warmup)
            return total, self.per_call(step, steps)
        (total_ms, call_ms), clocks = self.with_clocks(run)
        ms = total_ms / steps
        part = {"workload": name, "value": round(self.ws * nbytes / (ms * 1e-3) / 1e9, 1),
                "unit": "GB/s", "ms_per_step": round(ms, 5), "steps": steps,
                "num_splits": splits, "bytes_per_step": nbytes,
                "roofline": self.hbm_roofline(nbytes, call_ms, traffic_kind,
                                              "decode split kernel + LSE merge (one C-ABI call)"),
                "gpu_launches": d["launches"] * steps, "clocks": clocks}
        return part, step, d

    def prefill_part(self, batch, name, steps, traffic_kind):
        step, d = self.prefill_step(batch)
        flops = prefill_flops(batch)

        def run():
            self.warm_clock(step)
            total = self.timed(step, steps, self.args.warmup)
            return total, self.per_call(step, steps)
        (total_ms, call_ms), clocks = self.with_clocks(run)
        ms = total_ms / steps
        part = {"workload": name, "value": round(self.ws * flops / (ms * 1e-3) / 1e12, 2),
                "unit": "TFLOP/s", "ms_per_step": round(ms, 5), "steps": steps,
                "flops_per_step": flops, "roofline": self.tensor_roofline(flops, call_ms, traffic_kind),
                "gpu_launches": steps, "clocks": clocks}
        return part, step

    def mixed_one_launch(self, batch, num_decode, steps, dec_bytes, pre_flops):
        """The whole mixed batch through attn_sink_mixed: decode rows and prefill
        segments in one persistent launch (plus the merge of split decode rows)."""
        torch, gas = self.torch, self.gas
        d = dict(q=self.to_dev(batch.q), k=self.to_dev(batch.k_cache), v=self.to_dev(batch.v_cache),
                 cu=self.to_dev(batch.cu_seqlens_q), kvl=self.to_dev(batch.kv_lens),
                 bt=self.to_dev(batch.block_table), sinks=self.to_dev(batch.sinks))
        out = torch.empty_like(d["q"])
        lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=self.dev)
        need = gas.mixed_workspace_size(num_decode, batch.Hq, batch.Hkv, batch.D,
                                        batch.block_table.shape[1], batch.page_size)
        ws = torch.empty(max(need, 256), dtype=torch.uint8, device=self.dev)
        max_q = int(batch.q_lens[num_decode:].max())

        def step():
            gas.mixed(d["q"], d["k"], d["v"], d["cu"], d["kvl"], d["bt"], d["sinks"],
                      num_decode=num_decode, max_q_len=max_q, scale=batch.scale, out=out, lse=lse,
                      workspace=ws)

        def run():
            self.warm_clock(step)
            total = self.timed(step, steps, self.args.warmup)
            return total, self.per_call(step, steps)
        (total_ms, call_ms), clocks = self.with_clocks(run)
        # lower bound with perfect overlap: the decode bytes at the HBM peak and
        # the prefill FLOPs at the bf16 peak run side by side
        bound_ms = max(dec_bytes / (self.pk["hbm_gbs"] * 1e9), pre_flops / (self.pk["bf16_tflops"] * 1e12)) * 1e3
        sum_ms = (dec_bytes / (self.pk["hbm_gbs"] * 1e9) + pre_flops / (self.pk["bf16_tflops"] * 1e12)) * 1e3
        self.release(d)
        return {"workload": "the whole mixed batch through attn_sink_mixed (one persistent launch "
                            "+ merge)", "ms_per_step": round(total_ms / steps, 5), "steps": steps,
                "call_ms": round(call_ms, 5), "overlap_bound_ms": round(bound_ms, 5),
                "serial_bound_ms": round(sum_ms, 5),
                "frac_of_overlap_bound": round(bound_ms / call_ms, 4), "gpu_launches": 2 * steps,
                "clocks": clocks}

    def e2e_decode(self, batch, splits, d):
        """End to end through the C ABI: every step copies all its inputs from pinned
        host memory and reads its result back.  Two device input sets alternate, so
        the copy of step i+1 (on a copy stream) overlaps the decode of step i; the
        decode of a set waits for that set's copy, and a set is refilled only after
        the decode that read it has finished."""
        torch, gas, stream = self.torch, self.gas, self.stream
        h_in = [self.pinned(a) for a in (batch.q, batch.k_cache, batch.v_cache, batch.kv_lens,
                                         batch.block_table, batch.sinks)]
        first = [d["q"], d["k"], d["v"], d["kvl"], d["bt"], d["sinks"]]
        sets = [first, [torch.empty_like(t) for t in first]]
        outs = [(d["out"], d["lse"]), (torch.empty_like(d["out"]), torch.empty_like(d["lse"]))]
        wss = [d["ws"], torch.empty_like(d["ws"])]
        h_out = torch.empty(d["out"].shape, dtype=d["out"].dtype).pin_memory()
        h_lse = torch.empty(d["lse"].shape, dtype=d["lse"].dtype).pin_memory()
        copy_stream = torch.cuda.Stream(device=self.dev)
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        freed = [torch.cuda.Event(), torch.cuda.Event()]

        def e2e_step(i):
            st = i % 2
            d_in, (o_d, l_d) = sets[st], outs[st]
            copy_stream.wait_event(freed[st])
            with torch.cuda.stream(copy_stream):
                for h, dv in zip(h_in, d_in):
                    dv.copy_(h, non_blocking=True)
                copied[st].record(copy_stream)
            stream.wait_event(copied[st])
            gas.decode(d_in[0], d_in[1], d_in[2], d_in[3], d_in[4], d_in[5], scale=batch.scale,
                       num_splits=splits, out=o_d, lse=l_d, workspace=wss[st])
            freed[st].record(stream)
            h_out.copy_(o_d, non_blocking=True)
            h_lse.copy_(l_d, non_blocking=True)

        for st in range(2):                        # both sets' events exist before timing
            freed[st].record(stream)
        steps = max(4, min(self.args.steps, 20))
        for i in range(2):                         # warm-up
            e2e_step(i)
        torch.cuda.synchronize()
        self.barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        copy_stream.wait_stream(stream)            # the first copy starts after t0
        for i in range(steps):
            e2e_step(i)
        t1.record(stream)                          # after the last decode and read-back
        torch.cuda.synchronize()
        self.barrier()
        ms = self.reduce_max(t0.elapsed_time(t1)) / steps
        h2d = sum(t.numel() * t.element_size() for t in h_in)
        d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
        nbytes = decode_bytes(batch)
        return {"value": round(self.ws * nbytes / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h}

    def release(self, *objs):
        for o in objs:
            if isinstance(o, dict):
                o.clear()
        self.torch.cuda.synchronize()
        self.torch.cuda.empty_cache()


def cpu_baselines_wanted(args, ws, rank):
    return rank == 0 and ws == 1 and not args.no_cpu_baseline


def run_ours(args, ws, rank, local):
    arm = GpuArm(args, ws, rank, local)
    so = arm.seed_off
    steps = args.steps
    want_cpu = cpu_baselines_wanted(args, ws, rank)
    sub = {}
    head = None

    if args.workload in ("all", "decode"):
        batch = W.gptoss_decode(seed=20260002 + so)
        name = ("gpt-oss decode: 64 seqs, Hq 64, Hkv 8, D 64, KV lengths U[512, 8192], page 16, "
                "shuffled page table, bf16")
        part, step, d = arm.decode_part(batch, 0, name, steps, "decode")
        part["e2e"] = arm.e2e_decode(batch, 0, d)
        if want_cpu:
            part["cpu_baseline"] = cpu_oracle_rate(batch, args.cpu_seconds, "GB/s")
        arm.release(d)
        head = part

    if args.workload in ("all", "prefill"):
        batch = W.gptoss_prefill(seed=20260003 + so)
        name = ("gpt-oss causal prefill: 8 seqs x 4096, Hq 64, Hkv 8, D 64, bf16, ragged "
                "cu_seqlens, paged K/V, out bf16 + fp32 lse")
        part, _ = arm.prefill_part(batch, name, max(3, min(steps, 50)), "prefill")
        if want_cpu:
            part["cpu_baseline"] = cpu_oracle_rate(batch, args.cpu_seconds, "TFLOP/s")
        arm.release()
        sub["prefill"] = part
        del batch

    if args.workload in ("all", "long"):
        batch = W.long_split_decode(seed=20260004 + so)
        name = "long split-KV decode: 4 seqs x 131072 keys, 32 chunks, Hq 64, Hkv 8, D 64, bf16"
        part, _, d = arm.decode_part(batch, 32, name, max(3, min(steps, 100)), "long")
        if want_cpu:
            part["cpu_baseline"] = cpu_oracle_rate(batch, args.cpu_seconds, "GB/s")
        arm.release(d)
        sub["long"] = part
        del batch

    if args.workload in ("all", "mixed"):
        m = W.mixed_batch(seed=20260005 + so)
        k = max(3, min(steps, 100))
        dpart, dstep, d = arm.decode_part(
            m["decode"], 0, "mixed batch, decode part: 48 seqs, KV U[1024, 32768], Hq 64, Hkv 8, "
            "D 64, bf16, 1% outlier keys", k, "mixed_decode")
        ppart, pstep = arm.prefill_part(
            m["prefill"], "mixed batch, chunked-prefill part: 4 x 512 new tokens over prefixes "
            "U[0, 16384], Hq 64, Hkv 8, D 64, bf16, 1% outlier keys", k, "mixed_prefill")

        def both():
            dstep()
            pstep()
        total = arm.timed(both, k, args.warmup)
        one = arm.mixed_one_launch(m["single"], m["single"].meta["n_decode"], k,
                                   dpart["bytes_per_step"], ppart["flops_per_step"])
        if want_cpu:
            dpart["cpu_baseline"] = cpu_oracle_rate(m["decode"], args.cpu_seconds / 2, "GB/s")
            ppart["cpu_baseline"] = cpu_oracle_rate(m["prefill"], args.cpu_seconds / 2, "TFLOP/s")
        arm.release(d)
        sub["mixed"] = {"workload": "mixed batch: decode part then chunked-prefill part, two "
                                    "launches on one stream",
                        "ms_per_step": round(total / k, 5), "decode": dpart, "prefill": ppart,
                        "one_launch": one}
        one["vs_two_launches"] = round((total / k) / one["ms_per_step"], 3)
        del m

    if head is None:
        # a single non-headline workload: its own numbers head the line
        key = next(iter(sub))
        p = sub.pop(key)
        if key == "mixed":
            p = dict(p["decode"], mixed_prefill=p["prefill"], ms_both=p["ms_per_step"])
        head = p
    res = {"metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": ws,
           "steps": head["steps"], "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded normal q/k/v, shuffled page table)",
           "config": {"workload": head["workload"],
                      "l2": "inputs larger than L2 (129 MB): no flush between steps"},
           "roofline": head["roofline"], "gpu_launches": head["gpu_launches"],
           "clocks": head["clocks"]}
    for k in ("e2e", "cpu_baseline", "num_splits", "bytes_per_step", "flops_per_step"):
        if k in head:
            (res["config"] if k in ("num_splits", "bytes_per_step", "flops_per_step")
             else res)[k] = head[k]
    for k, v in head.items():
        if k in ("mixed_prefill", "ms_both"):
            res[k] = v
    res.update(sub)
    return res


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    batch = W.gptoss_decode()
    import oracle
    oracle.max_threads()
    steps, warm = args.steps, args.warmup
    per_step_seqs = 2
    times, nbytes = [], 0
    b = 0
    prob = oracle.Problem(batch.q, batch.k_cache, batch.v_cache, batch.cu_seqlens_q,
                          batch.kv_lens, batch.block_table, batch.sinks, batch.scale, True)
    for i in range(warm + steps):
        seqs = [(b + j) % batch.B for j in range(per_step_seqs)]
        b = (b + per_step_seqs) % batch.B
        rows = np.concatenate([np.arange(s * batch.Hq, (s + 1) * batch.Hq) for s in seqs])
        t0 = time.perf_counter()
        prob.attention(rows)
        dt = time.perf_counter() - t0
        if i >= warm:
            times.append(dt)
            nbytes += sum(int(batch.kv_lens[s]) for s in seqs) * batch.Hkv * batch.D * 4
    total = sum(times)
    value = nbytes / total / 1e9
    threads = oracle.max_threads()
    sample = "%d decode sequences (all 64 heads) per step of the 64-sequence batch" % per_step_seqs
    return {"metric": METRIC, "impl": "reference", "value": round(value, 3), "unit": "GB/s",
            "n_gpus": ws, "steps": steps, "warmup": warm,
            "ms_per_step": round(1e3 * total / steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "gpt-oss decode: 64 seqs, Hq 64, Hkv 8, D 64, KV U[512, 8192], "
                                   "page 16 (fp64 CPU oracle, bounded sample)"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["all", "decode", "prefill", "long", "mixed"],
                    default="all")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=6.0,
                    help="seconds of fp64 oracle time per workload for the CPU baselines")
    ap.add_argument("--clock-window", type=float, default=1.0,
                    help="seconds of untimed steps run while clock sampling starts")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend)

    if args.impl == "reference":
        res = run_reference(args, ws, rank)
    else:
        res = run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
