"""Benchmark: sink GQA attention on GB300 (decode HBM GB/s, prefill TFLOP/s).

Default (N=1): one JSON line whose headline workload is gpt-oss-shaped paged
decode (64 seqs, Hq 64, Hkv 8, D 64, KV lengths uniform in [512, 8192], page
size 16, bf16).  A step is one decode call: the split-KV kernel plus the LSE
merge, through the C ABI.  value = algorithmic K/V bytes per step / device
time per step.  The prefill workload (8 x 4096 causal, ragged layout) is timed
the same way and reported under "prefill" in TFLOP/s of the causal half.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill|long|mixed] [--no-cpu-baseline]

Multi-GPU (torchrun): every rank runs its own replica of the workload with a
rank-specific seed (weak scaling, no collective on the data path); timing is
the max over ranks.  --impl reference times the fp64 CPU oracle on the host
cores over a bounded sample of the same workload.
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
# dominant kernel, from the ncu captures summarised in profiles/.  A value holds
# only for the kernel sources it was captured with (sha256 over the listed files);
# after any change to them the roofline reports traffic = null.
CSRC = "gqa_attention_sinks_gb300/csrc/"
NCU_TRAFFIC = {
    "prefill": {"files": [CSRC + f for f in ("prefill_bf16.cu", "tcgen05.cuh", "ptx.cuh",
                                               "exp2_poly.cuh", "kernels.h")],
                "sha256": "78c8244eec28bb38175d335bca1f4cf8fba4d82f72883e9421ff3d381b62a7c1",
                "bytes": 812987136},
    "decode": {"files": [CSRC + f for f in ("decode_bf16.cu", "ptx.cuh", "kernels.h", "api.cu")],
               "sha256": "bb0a99524c531ef95cb63a834ce534f3e6b7126f07678c6335e654ce193ce02a",
               "bytes": 583148800},
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


def prefill_flops(batch):
    """Algorithmic FLOPs of causal prefill: 4*D per visible (query row, key) pair."""
    q = batch.q_lens.astype(np.int64)
    kv = batch.kv_lens.astype(np.int64)
    pairs = 0
    for ql, kl in zip(q, kv):
        first = kl - ql + 1                       # keys seen by the first query
        pairs += ql * first + ql * (ql - 1) // 2 if batch.causal else ql * kl
    return 4 * batch.D * batch.Hq * int(pairs)


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


# ----------------------------------------------------------------- GPU arm
def run_ours(args, ws, rank, local):
    import torch
    import gqa_attention_sinks_gb300 as gas

    torch.cuda.set_device(local)
    gas.load()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    pk, pk_kind = peaks()

    def to_dev(a):
        if a.dtype == np.uint16:
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    def pinned(a):
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16
                             else np.ascontiguousarray(a))
        t = t.pin_memory()
        return t.view(torch.bfloat16) if a.dtype == np.uint16 else t

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    def max_over_ranks(x):
        if ws == 1:
            return x
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())

    def timed(fn, steps, warmup, per_call=False):
        """Device time of `steps` calls after `warmup` calls (ms total, per-call list)."""
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        per = []
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        if per_call:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(steps)]
        t0.record(stream)
        for i in range(steps):
            if per_call:
                evs[i][0].record(stream)
            fn()
            if per_call:
                evs[i][1].record(stream)
        t1.record(stream)
        torch.cuda.synchronize()
        barrier()
        total = t0.elapsed_time(t1)
        if per_call:
            per = [a.elapsed_time(b) for a, b in evs]
        return max_over_ranks(total), per

    seed_off = 1000 * rank
    result = {}

    # ---------------------------------------------------------- decode
    if args.workload in ("decode", "long", "mixed"):
        if args.workload == "decode":
            batch = W.gptoss_decode(seed=20260002 + seed_off)
            splits = 0
            wl = ("gpt-oss decode: 64 seqs, Hq 64, Hkv 8, D 64, KV lengths U[512, 8192], "
                  "page 16, shuffled page table, bf16")
        elif args.workload == "long":
            batch = W.long_split_decode(seed=20260004 + seed_off)
            splits = 32
            wl = "long split-KV decode: 4 seqs x 131072 keys, 32 chunks, Hq 64, Hkv 8, D 64, bf16"
        else:
            batch = W.mixed_batch(seed=20260005 + seed_off)["decode"]
            splits = 0
            wl = "mixed batch, decode part: 48 seqs, KV U[1024, 32768], Hq 64, Hkv 8, bf16"
        q, k, v = to_dev(batch.q), to_dev(batch.k_cache), to_dev(batch.v_cache)
        kvl, bt, sinks = to_dev(batch.kv_lens), to_dev(batch.block_table), to_dev(batch.sinks)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        need = gas.decode_workspace_size(batch.B, batch.Hq, batch.Hkv, batch.D,
                                         batch.block_table.shape[1], batch.page_size, splits)
        wsbuf = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)

        def step():
            gas.decode(q, k, v, kvl, bt, sinks, scale=batch.scale, num_splits=splits, out=out,
                       lse=lse, workspace=wsbuf)

        nbytes = decode_bytes(batch)
        sampler = ClockSampler(local)
        sampler.start()
        t_end = time.time() + args.clock_window
        while time.time() < t_end:                 # clock window: load the GPU for sampling
            step()
            torch.cuda.synchronize()
        total_ms, _ = timed(step, args.steps, args.warmup)
        _, per = timed(step, args.steps, 0, per_call=True)
        clocks = sampler.stop()
        ms = total_ms / args.steps
        call_ms = float(np.mean(per))
        value = ws * nbytes / (ms * 1e-3) / 1e9
        achieved = nbytes / (call_ms * 1e-3) / 1e9
        launches_per_step = 2 if need > 0 else 1

        # End to end through the C ABI: every step copies all its inputs from pinned
        # host memory and reads its result back.  Two device input sets alternate, so
        # the copy of step i+1 (on a copy stream) overlaps the decode of step i; the
        # decode of a set waits for that set's copy, and a set is refilled only after
        # the decode that read it has finished.
        h_in = [pinned(a) for a in (batch.q, batch.k_cache, batch.v_cache, batch.kv_lens,
                                    batch.block_table, batch.sinks)]
        sets = [[q, k, v, kvl, bt, sinks], [torch.empty_like(t) for t in (q, k, v, kvl, bt, sinks)]]
        outs = [(out, lse), (torch.empty_like(out), torch.empty_like(lse))]
        wss = [wsbuf, torch.empty_like(wsbuf)]
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        copy_stream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        freed = [torch.cuda.Event(), torch.cuda.Event()]

        def e2e_step(i):
            st = i % 2
            d_in, (o_d, l_d) = sets[st], outs[st]
            copy_stream.wait_event(freed[st])
            with torch.cuda.stream(copy_stream):
                for h, d in zip(h_in, d_in):
                    d.copy_(h, non_blocking=True)
                copied[st].record(copy_stream)
            stream.wait_event(copied[st])
            gas.decode(d_in[0], d_in[1], d_in[2], d_in[3], d_in[4], d_in[5], scale=batch.scale,
                       num_splits=splits, out=o_d, lse=l_d, workspace=wss[st])
            freed[st].record(stream)
            h_out.copy_(o_d, non_blocking=True)
            h_lse.copy_(l_d, non_blocking=True)

        for st in range(2):                        # both sets' events exist before timing
            freed[st].record(stream)
        e2e_steps = max(4, min(args.steps, 20))
        for i in range(2):                         # warm-up
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        copy_stream.wait_stream(stream)            # the first copy starts after t0
        for i in range(e2e_steps):
            e2e_step(i)
        t1.record(stream)                          # after the last decode and read-back
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(t0.elapsed_time(t1)) / e2e_steps
        h2d = sum(t.numel() * t.element_size() for t in h_in)
        d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()

        result = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded normal q/k/v, shuffled page table)",
            "config": {"workload": wl, "num_splits": splits,
                       "l2": "inputs larger than L2: %.0f MB of K/V per step" % (nbytes / 1e6),
                       "bytes_per_step": nbytes},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / pk["hbm_gbs"], 4),
                         "traffic": ncu_traffic("decode") if args.workload == "decode" else None,
                         "peak_source": pk_kind,
                         "kernel": "decode split kernel + LSE merge (one C-ABI call)"},
            "e2e": {"value": round(ws * nbytes / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                    "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }

    # ---------------------------------------------------------- prefill
    if (args.workload in ("decode", "prefill", "mixed")) and not args.no_prefill:
        if args.workload == "mixed":
            pre = W.mixed_batch(seed=20260005 + seed_off)["prefill"]
            pre_name = ("mixed batch, chunked-prefill part: 4 x 512 new tokens over prefixes "
                        "U[0, 16384], Hq 64, Hkv 8, D 64, bf16, paged K/V, 1% outlier keys")
        else:
            pre = W.gptoss_prefill(seed=20260003 + seed_off)
            pre_name = ("gpt-oss causal prefill: 8 seqs x 4096, Hq 64, Hkv 8, D 64, bf16, "
                        "ragged cu_seqlens, paged K/V")
        q, k, v = to_dev(pre.q), to_dev(pre.k_cache), to_dev(pre.v_cache)
        cu, kvl = to_dev(pre.cu_seqlens_q), to_dev(pre.kv_lens)
        bt, sinks = to_dev(pre.block_table), to_dev(pre.sinks)
        out = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)

        def pstep():
            gas.prefill(q, k, v, cu, kvl, bt, sinks, max_q_len=pre.max_q_len, scale=pre.scale,
                        out=out, lse=lse)

        flops = prefill_flops(pre)
        part = {"workload": pre_name, "flops_per_step": flops}
        try:
            pstep()
            torch.cuda.synchronize()
            psteps = max(3, min(args.steps, 50))
            sampler = ClockSampler(local)
            sampler.start()
            t_end = time.time() + args.clock_window
            while time.time() < t_end:
                pstep()
                torch.cuda.synchronize()
            total_ms, per = timed(pstep, psteps, args.warmup, per_call=True)
            pclocks = sampler.stop()
            pms = total_ms / psteps
            call_ms = float(np.mean(per))
            ach = flops / (call_ms * 1e-3) / 1e12
            peak = pk["bf16_tflops"]
            part.update({"value": round(ws * flops / (pms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                         "ms_per_step": round(pms, 4), "steps": psteps, "clocks": pclocks,
                         "roofline": {"bound": "tensor", "achieved": round(ach, 2), "peak": peak,
                                      "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                                      "traffic": (ncu_traffic("prefill") if args.workload != "mixed"
                                                  else None),
                                      "peak_source": pk_kind}})
        except gas.AttnSinkError as e:
            part.update({"unavailable": str(e)})
        if result:
            result["prefill"] = part
        else:
            result = {"metric": METRIC, "value": part.get("value"), "unit": "TFLOP/s",
                      "n_gpus": ws, "steps": part.get("steps", args.steps), "warmup": args.warmup,
                      "ms_per_step": part.get("ms_per_step"), "higher_is_better": True,
                      "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                      "data": "synthetic (seeded normal q/k/v)",
                      "config": {"workload": part["workload"]},
                      "roofline": part.get("roofline"), "gpu_launches": part.get("steps", 0),
                      "clocks": part.get("clocks")}
    return result


# ----------------------------------------------------------------- CPU oracle
def cpu_oracle_rate(batch, seconds, max_seqs=None, rows_per_seq=None):
    """Time the fp64 oracle on the host cores over whole sequences of the batch.

    Returns (GB/s of algorithmic K/V bytes, threads, sample description, steps)."""
    import oracle
    prob = oracle.Problem(batch.q, batch.k_cache, batch.v_cache, batch.cu_seqlens_q,
                          batch.kv_lens, batch.block_table, batch.sinks, batch.scale, batch.causal)
    n = batch.B if max_seqs is None else min(max_seqs, batch.B)
    done_bytes, elapsed, seqs = 0, 0.0, 0
    b = 0
    while elapsed < seconds and seqs < 1000 * batch.B:  # about `seconds` of oracle work
        rows = np.arange(batch.cu_seqlens_q[b] * batch.Hq, batch.cu_seqlens_q[b + 1] * batch.Hq)
        t0 = time.perf_counter()
        prob.attention(rows)
        elapsed += time.perf_counter() - t0
        done_bytes += int(batch.kv_lens[b]) * batch.Hkv * batch.D * 4
        seqs += 1
        b = (b + 1) % n
    return done_bytes / elapsed / 1e9, oracle.max_threads(), "%d whole sequences" % seqs, elapsed


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
    ap.add_argument("--workload", choices=["decode", "prefill", "long", "mixed"], default="decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--clock-window", type=float, default=2.0,
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
        if rank == 0 and ws == 1 and not args.no_cpu_baseline and args.workload in ("decode",):
            batch = W.gptoss_decode()
            rate, threads, sample, secs = cpu_oracle_rate(batch, args.cpu_seconds)
            res["cpu_baseline"] = {"value": round(rate, 3), "unit": "GB/s", "cores": threads,
                                   "kind": "oracle", "sample": sample + " (%.1f s)" % secs}
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
