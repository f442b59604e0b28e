"""Benchmark of the paged KV attention path on one GB300 (or N replicas).

Default workload: the batch-decode configuration (64 requests, kv_len
~ U[512, 4096], page size 16, 32 qo / 8 kv heads, head_dim 128, bf16 NHD,
split-KV with LSE merge).  A step is one run() of the plan (decode kernel +
merge kernel) with every input resident in HBM; the metric is algorithmic
KV bytes (+ Q, O, LSE) per second.  When the tensor-core path is built the
append-prefill workload (16 requests, append_paged_kv_cache then causal
attention) is measured the same way and reported under "prefill".

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode KV GB/s vs HBM peak; append-prefill TFLOP/s vs bf16 TC peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        p["source"] = "measured"
        return p
    p = dict(FALLBACK_PEAKS)
    p["source"] = "fallback"
    return p


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, x in enumerate(r) if x == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": rows[0][1],
                "reasons": reasons, "samples": len(rows)}


def flush_l2(buf):
    buf.add_(1)


def time_steps(fn, steps, warmup, stream, l2_buf=None):
    """Per-step CUDA-event durations (ms) on the launching stream."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        if l2_buf is not None:
            flush_l2(l2_buf)
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


# ---------------------------------------------------------------------------
# Workloads
# ---------------------------------------------------------------------------

def decode_setup(device):
    import paged_kv_attention_plan_gb300 as pka
    from paged_kv_attention_plan_gb300 import workloads as W
    from tests.gpu_util import bf16, i32

    b = W.batch_decode(seed=1001)
    d = dict(batch=b, q=bf16(b.q, device), k=bf16(b.k_pool, device), v=bf16(b.v_pool, device),
             idx=i32(b.kv_indices, device))
    attn = pka.BatchAttention(device=device)
    info = attn.plan(None, b.kv_indptr, b.last_page_len, num_qo_heads=32, num_kv_heads=8,
                     head_dim=128, page_size=16, split_mode="auto")
    d["attn"], d["info"] = attn, info
    d["o"] = torch.empty_like(d["q"])
    d["lse"] = torch.empty(b.nnz_q, 32, dtype=torch.float32, device=device)
    kv_tokens = int(np.sum(b.kv_lens))
    d["kv_bytes"] = kv_tokens * 8 * 128 * 2 * 2
    d["bytes"] = d["kv_bytes"] + 2 * d["q"].numel() * 2 + d["lse"].numel() * 4
    d["launches"] = int(info.num_decode_items > 0) + int(info.num_prefill_items > 0) + \
        int(info.num_merge_tasks > 0)
    return d


def decode_step(d):
    d["attn"].run(d["q"], d["k"], d["v"], d["idx"], out=d["o"], lse=d["lse"])


def e2e_decode(d, steps, warmup, stream, device):
    """Through the public API with host buffers: H2D of this step's inputs
    (q, kv_indices and the plan built from host metadata), run, D2H of O/LSE."""
    import paged_kv_attention_plan_gb300 as pka
    b = d["batch"]
    q_h = d["q"].cpu().pin_memory()
    idx_h = torch.from_numpy(b.kv_indices).pin_memory()
    o_h = torch.empty(d["o"].shape, dtype=d["o"].dtype).pin_memory()
    lse_h = torch.empty(d["lse"].shape, dtype=torch.float32).pin_memory()
    q_d, idx_d = torch.empty_like(d["q"]), torch.empty_like(d["idx"])
    attn = pka.BatchAttention(device=device)

    def step():
        q_d.copy_(q_h, non_blocking=True)
        idx_d.copy_(idx_h, non_blocking=True)
        attn.plan(None, b.kv_indptr, b.last_page_len, num_qo_heads=32, num_kv_heads=8,
                  head_dim=128, page_size=16, split_mode="auto")
        attn.run(q_d, d["k"], d["v"], idx_d, out=d["o"], lse=d["lse"])
        o_h.copy_(d["o"], non_blocking=True)
        lse_h.copy_(d["lse"], non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = max(ev0.elapsed_time(ev1), wall * 1e3) / steps
    h2d = q_h.numel() * 2 + idx_h.numel() * 4 + int(attn.info.int_ws_bytes)
    d2h = o_h.numel() * 2 + lse_h.numel() * 4
    return {"value": d["bytes"] / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms}


def oracle_sample(seconds_budget=20.0, max_requests=None):
    """CPU oracle on the first requests of the batch-decode workload."""
    from oracle import ref
    from paged_kv_attention_plan_gb300 import workloads as W
    b = W.batch_decode(seed=1001)
    done_bytes, t_used, r = 0, 0.0, 0
    limit = max_requests or b.batch_size
    while t_used < seconds_budget and r < limit:
        t0 = time.perf_counter()
        ref.batch_attention(b.q, b.k_pool, b.v_pool, qo_indptr=b.qo_indptr,
                            kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                            last_page_len=b.last_page_len, page_size=16, num_qo_heads=32,
                            num_kv_heads=8, requests=[r])
        t_used += time.perf_counter() - t0
        done_bytes += int(b.kv_lens[r]) * 8 * 128 * 2 * 2 + 2 * 32 * 128 * 2 + 32 * 4
        r += 1
    return done_bytes / t_used / 1e9, r, t_used


def cpu_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        if info:
            return max(i.get("num_threads", 1) for i in info)
    except Exception:
        pass
    return os.cpu_count()


# ---------------------------------------------------------------------------

def reference_arm(args, rank):
    if rank != 0:
        return
    vals = []
    for _ in range(args.warmup):
        oracle_sample(seconds_budget=0.0, max_requests=1)
    for _ in range(args.steps):
        v, nreq, secs = oracle_sample(seconds_budget=2.0, max_requests=2)
        vals.append(v)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "batch_decode: 64 req, kv_len U[512,4096], page 16, 32/8 "
                                   "heads, D 128, NHD; CPU oracle on the first 2 requests "
                                   "per step"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cpu_threads(),
                             "kind": "oracle",
                             "sample": "first 2 requests of the batch-decode workload per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pka", choices=["pka", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    device = f"cuda:{local}"
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(device))
    stream = torch.cuda.current_stream()

    d = decode_setup(device)
    pk = peaks()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]
                    if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit()
                    else local)
    with ClockSampler(gpu_index) as clocks:
        barrier()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(args.warmup):
            decode_step(d)
        barrier()
        ev0.record(stream)
        for _ in range(args.steps):
            decode_step(d)
        ev1.record(stream)
        barrier()
    total_ms = ev0.elapsed_time(ev1)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([total_ms], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms = total_ms / args.steps
    value = world * d["bytes"] / (ms * 1e-3) / 1e9

    # per-launch duration of the decode step (inputs > L2, so no flush is needed)
    per = time_steps(lambda: decode_step(d), 200, 5, stream)
    step_ms = statistics.median(per)
    achieved = d["bytes"] / (step_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": None,
            "kernel": "decode_kernel<128,4> + merge_kernel<128> (one run())",
            "peak_source": pk["source"]}

    e2e = e2e_decode(d, min(args.steps, 500), 5, stream, device)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([e2e["ms_per_step"]], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e["value"] = world * d["bytes"] / (float(t.item()) * 1e-3) / 1e9
    e2e.pop("ms_per_step")

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "batch_decode: 64 req, kv_len U[512,4096] (seed 1001), page 16, "
                                   "32/8 heads, D 128, bf16 NHD, split-KV auto + LSE merge",
                       "kv_bytes_per_step": d["kv_bytes"], "bytes_per_step": d["bytes"],
                       "l2": "inputs (604 MB of K/V) larger than L2; no flush",
                       "parallelism": f"replicas x{world}"},
            "roofline": roof, "e2e": e2e, "gpu_launches": d["launches"] * args.steps,
            "clocks": clocks.summary(), "plan": d["info"].as_dict()}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, nreq, secs = oracle_sample(seconds_budget=15.0)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": cpu_threads(),
                                "kind": "oracle",
                                "sample": f"first {nreq} requests of the batch-decode workload "
                                          f"({secs:.1f} s of CPU work)"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
