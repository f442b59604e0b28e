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


def recorded_traffic(kernel):
    """DRAM bytes per launch of `kernel` from its committed ncu capture
    (profiles/traffic.json), or None when the kernel's sources changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    h = hashlib.sha256()
    for name in rec["sources"]:
        with open(os.path.join(ROOT, "paged_kv_attention_plan_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return rec["dram_bytes_per_launch"] if h.hexdigest() == rec["source_sha256"] else None


def flush_l2(buf):
    buf.add_(1)


def max_over_ranks(x: float, world: int, device="cpu") -> float:
    """The largest value of x over all ranks (x itself when world == 1)."""
    if world <= 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, ms_per_step: float, world: int) -> float:
    """Whole-job throughput: units of all ranks per second of the slowest rank."""
    return world * units_per_rank / (ms_per_step * 1e-3)


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

def bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """bf16 bit patterns (uint16) as a bf16 device tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def i32(a, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def kv_tensor(pool: np.ndarray, device="cuda") -> torch.Tensor:
    """A K/V pool on the device: bf16 from bit patterns, or uint8 e4m3 codes."""
    if pool.dtype == np.uint8:
        return torch.from_numpy(np.ascontiguousarray(pool)).to(device)
    return bf16(pool, device)


def decode_setup(device, kv_dtype="bf16", on_tensor_cores=False):
    """Batch-decode workload; kv_dtype "e4m3" stores K/V as 8-bit codes (one
    scale per pool), halving the K/V bytes per key."""
    import paged_kv_attention_plan_gb300 as pka
    from inputs import workloads as W

    b = W.batch_decode(seed=1001, kv_dtype=kv_dtype, k_scale=0.5, v_scale=2.0)
    d = dict(batch=b, q=bf16(b.q, device), k=kv_tensor(b.k_pool, device),
             v=kv_tensor(b.v_pool, device), idx=i32(b.kv_indices, device))
    attn = pka.BatchAttention(device=device)
    kw = dict(num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, split_mode="auto",
              kv_dtype=kv_dtype, k_scale=b.k_scale, v_scale=b.v_scale,
              decode_on_tensor_cores=on_tensor_cores)
    info = attn.plan(None, b.kv_indptr, b.last_page_len, **kw)
    d["attn"], d["info"] = attn, info
    t = []
    for _ in range(20):  # host time of one plan() (validation, planning, image, async copy)
        t0 = time.perf_counter()
        attn.plan(None, b.kv_indptr, b.last_page_len, **kw)
        t.append(time.perf_counter() - t0)
    d["plan_us"] = statistics.median(t) * 1e6
    d["o"] = torch.empty_like(d["q"])
    d["lse"] = torch.empty(b.nnz_q, 32, dtype=torch.float32, device=device)
    kv_tokens = int(np.sum(b.kv_lens))
    d["kv_tokens"] = kv_tokens
    d["kv_bytes"] = kv_tokens * 8 * 128 * (1 if kv_dtype == "e4m3" else 2) * 2
    d["bytes"] = d["kv_bytes"] + 2 * d["q"].numel() * 2 + d["lse"].numel() * 4
    # split decode rows are merged inside the decode kernel; the merge kernel
    # only runs for states it does not cover
    d["launches"] = int(info.num_decode_items > 0) + int(info.num_prefill_items > 0) + \
        int(info.num_merge_tasks > info.num_decode_joins * (32 // 8))
    return d


def decode_step(d):
    d["attn"].run(d["q"], d["k"], d["v"], d["idx"], out=d["o"], lse=d["lse"])


def e2e_decode(d, steps, warmup, stream, device):
    """Through the public API with host buffers: every step copies its inputs
    (q, kv_indices and the plan built from host metadata) from pinned host
    memory, runs, and reads O/LSE back to pinned host memory.  Steps are
    pipelined as a serving loop runs them: step i+1's copies and plan() go on
    a copy stream while step i computes, and step i's result is read back on
    a third stream; device buffers and plans are double-buffered, ordered by
    events, and all copies of all steps sit inside the timed region.  Q and
    kv_indices share one staging buffer (one copy in), O and LSE one output
    buffer (one copy out)."""
    import paged_kv_attention_plan_gb300 as pka
    b = d["batch"]
    q_bytes = d["q"].numel() * 2
    idx_bytes = b.kv_indices.size * 4
    o_bytes, lse_bytes = d["o"].numel() * 2, d["lse"].numel() * 4
    in_h = torch.empty(q_bytes + idx_bytes, dtype=torch.uint8).pin_memory()
    in_h[:q_bytes].view(torch.bfloat16).view(d["q"].shape).copy_(d["q"].cpu())
    in_h[q_bytes:].view(torch.int32).copy_(torch.from_numpy(b.kv_indices))
    out_h = [torch.empty(o_bytes + lse_bytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    in_d = [torch.empty(q_bytes + idx_bytes, dtype=torch.uint8, device=device) for _ in range(2)]
    out_d = [torch.empty(o_bytes + lse_bytes, dtype=torch.uint8, device=device) for _ in range(2)]
    q_d = [t[:q_bytes].view(torch.bfloat16).view(d["q"].shape) for t in in_d]
    idx_d = [t[q_bytes:].view(torch.int32) for t in in_d]
    o_d = [t[:o_bytes].view(torch.bfloat16).view(d["o"].shape) for t in out_d]
    lse_d = [t[o_bytes:].view(torch.float32).view(d["lse"].shape) for t in out_d]
    attn = [pka.BatchAttention(device=device) for _ in range(2)]
    h2d_s, d2h_s = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    ready, done, read = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e in done + read:
        e.record(stream)
    kw = dict(num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16, split_mode="auto")

    # (torch.cuda.set_stream rather than the stream context manager: the
    # manager costs 6-10 us of host time per use on the Grace host)
    def step(i):
        s = i & 1
        h2d_s.wait_event(done[s])  # step i-2 no longer reads slot s
        torch.cuda.set_stream(h2d_s)
        in_d[s].copy_(in_h, non_blocking=True)
        torch.cuda.set_stream(stream)
        attn[s].plan(None, b.kv_indptr, b.last_page_len, stream=h2d_s, **kw)
        ready[s].record(h2d_s)
        stream.wait_event(ready[s])
        stream.wait_event(read[s])  # step i-2's output has been read back
        attn[s].run(q_d[s], d["k"], d["v"], idx_d[s], out=o_d[s], lse=lse_d[s], stream=stream)
        done[s].record(stream)
        d2h_s.wait_event(done[s])
        torch.cuda.set_stream(d2h_s)
        out_h[s].copy_(out_d[s], non_blocking=True)
        torch.cuda.set_stream(stream)
        read[s].record(d2h_s)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        step(i)
    stream.wait_event(read[(steps - 1) & 1])
    ev1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ms = max(ev0.elapsed_time(ev1), wall * 1e3) / steps
    h2d = q_bytes + idx_bytes + int(attn[0].info.int_ws_bytes)
    d2h = o_bytes + lse_bytes
    # the last step's read-back against an output of the device-only loop
    decode_step(d)
    torch.cuda.synchronize()
    o_last = out_h[(steps - 1) & 1][:o_bytes].view(torch.bfloat16).view(d["o"].shape).float()
    diff = float((o_last - d["o"].cpu().float()).abs().max())
    return {"value": d["bytes"] / (ms * 1e-3) / 1e9, "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "max_abs_diff_vs_device_loop": diff,
            "pipeline": "Q + kv_indices copied in (one copy) and plan() on a copy stream, run on the "
                        "compute stream, O + LSE read back (one copy) on a third; double-buffered, "
                        "all inside the timed region"}


def prefill_flops(b):
    """Algorithmic FLOPs of attention over visible (query, key) pairs:
    4 * D * Hq per pair (QK^T and PV, 2 FLOPs per multiply-add)."""
    pairs = 0
    for q, k in zip(b.qo_lens, b.kv_lens):
        q, k = int(q), int(k)
        if b.mask_mode == "causal":
            pairs += q * (k - q) + q * (q + 1) // 2
        else:
            pairs += q * k
    return 4 * b.head_dim * b.num_qo_heads * pairs


def prefill_setup(device):
    """Append-prefill workload: append_paged_kv_cache writes the new rows,
    then causal attention of the new rows against their whole history."""
    import paged_kv_attention_plan_gb300 as pka
    from inputs import workloads as W

    b = W.append_prefill(seed=1002)
    d = dict(batch=b, q=bf16(b.q, device), k=bf16(b.k_pool, device), v=bf16(b.v_pool, device),
             k_new=bf16(b.k_new, device), v_new=bf16(b.v_new, device),
             idx=i32(b.kv_indices, device), qo=i32(b.qo_indptr, device),
             kvp=i32(b.kv_indptr, device), last=i32(b.last_page_len, device))
    d["params"] = pka.make_params(32, 8, 128, 16)
    attn = pka.BatchAttention(device=device)
    d["info"] = attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, num_qo_heads=32,
                          num_kv_heads=8, head_dim=128, page_size=16, split_mode="auto")
    d["attn"] = attn
    d["o"] = torch.empty_like(d["q"])
    d["lse"] = torch.empty(b.nnz_q, 32, dtype=torch.float32, device=device)
    d["flops"] = prefill_flops(b)
    d["append_bytes"] = 2 * 2 * b.nnz_q * 8 * 128 * 2
    return d


def prefill_fp8_setup(device):
    """The append-prefill workload over e4m3 pools (HND, page 16, k_scale 0.5,
    v_scale 2): append_paged_kv_cache quantizes the new rows into the pools,
    then attention (the tensor-core rows' keys decoded to a bf16 scratch)."""
    import paged_kv_attention_plan_gb300 as pka
    from inputs import workloads as W

    b = W.append_prefill(seed=1002, layout="HND", kv_dtype="e4m3", k_scale=0.5, v_scale=2.0)
    d = dict(batch=b, q=bf16(b.q, device), k=kv_tensor(b.k_pool, device),
             v=kv_tensor(b.v_pool, device), k_new=bf16(b.k_new, device),
             v_new=bf16(b.v_new, device), idx=i32(b.kv_indices, device),
             qo=i32(b.qo_indptr, device), kvp=i32(b.kv_indptr, device),
             last=i32(b.last_page_len, device))
    kw = dict(layout="HND", kv_dtype="e4m3", k_scale=0.5, v_scale=2.0)
    d["params"] = pka.make_params(32, 8, 128, 16, **kw)
    attn = pka.BatchAttention(device=device)
    d["info"] = attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, num_qo_heads=32,
                          num_kv_heads=8, head_dim=128, page_size=16, split_mode="auto", **kw)
    d["attn"] = attn
    d["o"] = torch.empty_like(d["q"])
    d["lse"] = torch.empty(b.nnz_q, 32, dtype=torch.float32, device=device)
    d["flops"] = prefill_flops(b)
    return d


def prefill_append(d):
    import paged_kv_attention_plan_gb300 as pka
    pka.pka_append_paged_kv_cache(d["params"], d["k_new"], d["v_new"], d["qo"], d["kvp"], d["idx"],
                                  d["last"], d["k"], d["v"], d["k"].stride(0))


def prefill_attn(d):
    d["attn"].run(d["q"], d["k"], d["v"], d["idx"], out=d["o"], lse=d["lse"])


def ragged_setup(device):
    """Ragged prefill with a custom mask: packbits of the boolean mask, then
    attention over ragged K/V (8 requests, 32/32 heads)."""
    import paged_kv_attention_plan_gb300 as pka
    from inputs import workloads as W

    b = W.ragged_custom_mask(seed=1004)
    d = dict(batch=b, q=bf16(b.q, device), k=bf16(b.k_pool, device), v=bf16(b.v_pool, device))
    d["bools"] = torch.from_numpy(b.mask_bool).to(device)
    d["packed"] = torch.empty((b.mask_bool.size + 7) // 8, dtype=torch.uint8, device=device)
    attn = pka.BatchAttention(device=device)
    d["info"] = attn.plan(b.qo_indptr, b.kv_indptr, None, num_qo_heads=32, num_kv_heads=32,
                          head_dim=128, mask_mode="custom", kv_ragged=True, split_mode="auto")
    d["attn"] = attn
    d["o"] = torch.empty_like(d["q"])
    d["lse"] = torch.empty(b.nnz_q, 32, dtype=torch.float32, device=device)
    d["flops_visible"] = 4 * 128 * 32 * int(b.mask_bool.sum())
    tiles = sum(((int(n) + 127) // 128) ** 2 for n in b.kv_lens)
    d["flops_tiles"] = 4 * 128 * 32 * tiles * 128 * 128
    d["flops_all"] = 4 * 128 * 32 * sum(int(n) ** 2 for n in b.kv_lens)
    return d


def ragged_step(d):
    import paged_kv_attention_plan_gb300 as pka
    pka.pka_packbits(d["bools"], d["packed"])
    d["attn"].run(d["q"], d["k"], d["v"], None, d["packed"], out=d["o"], lse=d["lse"])


def mixed_setup(device, page_size, layout):
    """Mixed serving step: 8 long + 120 short decodes and 4 prefill chunks of
    512 tokens in one plan (decode kernel, tensor-core kernel, merge)."""
    import paged_kv_attention_plan_gb300 as pka
    from inputs import workloads as W

    b = W.mixed_step(seed=1003, page_size=page_size, layout=layout, with_payload=False)
    pool = int(b.extra["pool_pages"])
    shape = (pool, page_size, 8, 128) if layout == "NHD" else (pool, 8, page_size, 128)
    g = torch.Generator(device=device).manual_seed(1003)
    d = dict(batch=b)
    d["k"] = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
    d["v"] = torch.randn(shape, generator=g, device=device).to(torch.bfloat16)
    d["q"] = torch.randn((b.nnz_q, 32, 128), generator=g, device=device).to(torch.bfloat16)
    d["idx"] = i32(b.kv_indices, device)
    attn = pka.BatchAttention(device=device)
    d["info"] = attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, num_qo_heads=32,
                          num_kv_heads=8, head_dim=128, page_size=page_size, layout=layout)
    d["attn"] = attn
    d["o"] = torch.empty_like(d["q"])
    d["lse"] = torch.empty(b.nnz_q, 32, dtype=torch.float32, device=device)
    dec = np.asarray(b.qo_lens) == 1
    d["decode_bytes"] = int(np.sum(np.asarray(b.kv_lens)[dec])) * 8 * 128 * 2 * 2
    pairs = 0
    for q_, k_ in zip(np.asarray(b.qo_lens)[~dec], np.asarray(b.kv_lens)[~dec]):
        pairs += int(q_) * (int(k_) - int(q_)) + int(q_) * (int(q_) + 1) // 2
    d["prefill_flops"] = 4 * 128 * 32 * pairs
    return d


def mixed_step(d):
    d["attn"].run(d["q"], d["k"], d["v"], d["idx"], out=d["o"], lse=d["lse"])


def cascade_setup(device):
    """64 decode rows sharing a 32768-token prompt (own suffixes U[512,2048]),
    planned as a two-level cascade and, for comparison, as a flat batch whose
    page tables each list the prompt's pages."""
    import paged_kv_attention_plan_gb300 as pka
    from inputs import workloads as W

    c = W.shared_prompt_decode(with_payload=False)
    root, own = c.levels
    pages = int(c.kv_indices.size)
    g = torch.Generator(device=device).manual_seed(1005)
    d = {}
    d["k"] = torch.randn((pages, 16, 8, 128), generator=g, device=device).to(torch.bfloat16)
    d["v"] = torch.randn((pages, 16, 8, 128), generator=g, device=device).to(torch.bfloat16)
    d["q"] = torch.randn((c.nnz_q, 32, 128), generator=g, device=device).to(torch.bfloat16)
    d["o"] = torch.empty_like(d["q"])
    d["lse"] = torch.empty(c.nnz_q, 32, dtype=torch.float32, device=device)
    d["idx"] = i32(c.kv_indices, device)
    casc = pka.BatchAttention(device=device)
    levels = [(lv["qo_indptr"], lv["kv_indptr"], lv["last_page_len"]) for lv in c.levels]
    kw = dict(num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    d["info"] = casc.plan_cascade(levels, **kw)
    d["casc"] = casc
    t = []
    for _ in range(5):
        t0 = time.perf_counter()
        casc.plan_cascade(levels, **kw)
        t.append(time.perf_counter() - t0)
    d["plan_us"] = statistics.median(t) * 1e6
    kv_indptr, flat = [0], []
    for r in range(len(own["kv_lens"])):
        flat += list(root["kv_indices"]) + list(own["kv_indices"][own["kv_indptr"][r]:
                                                                  own["kv_indptr"][r + 1]])
        kv_indptr.append(len(flat))
    flat_attn = pka.BatchAttention(device=device)
    flat_attn.plan(None, np.asarray(kv_indptr, np.int32), own["last_page_len"], **kw)
    d["flat"] = flat_attn
    d["flat_idx"] = i32(np.asarray(flat, np.int32), device)
    n, prompt = len(own["kv_lens"]), int(root["kv_lens"][0])
    own_tokens = int(np.sum(own["kv_lens"]))
    d["unique_bytes"] = (prompt + own_tokens) * 8 * 128 * 2 * 2
    d["flat_bytes"] = (n * prompt + own_tokens) * 8 * 128 * 2 * 2
    d["shared_flops"] = 4 * 128 * 32 * n * prompt
    d["own_bytes"] = own_tokens * 8 * 128 * 2 * 2
    d["prompt_bytes"] = prompt * 8 * 128 * 2 * 2
    return d


def cascade_step(d):
    d["casc"].run(d["q"], d["k"], d["v"], d["idx"], out=d["o"], lse=d["lse"])


def cascade_flat_step(d):
    d["flat"].run(d["q"], d["k"], d["v"], d["flat_idx"], out=d["o"], lse=d["lse"])


def oracle_sample(seconds_budget=20.0, max_requests=None):
    """CPU oracle on the requests of the batch-decode workload, taken in
    order (wrapping around after the last) until the time budget is spent or
    max_requests have run."""
    from oracle import ref
    from inputs import workloads as W
    b = W.batch_decode(seed=1001)
    done_bytes, t_used, r = 0, 0.0, 0
    limit = max_requests or 1 << 30
    while (r == 0 or t_used < seconds_budget) and r < limit:
        x = r % b.batch_size
        t0 = time.perf_counter()
        ref.batch_attention(b.q, b.k_pool, b.v_pool, qo_indptr=b.qo_indptr,
                            kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                            last_page_len=b.last_page_len, page_size=16, num_qo_heads=32,
                            num_kv_heads=8, requests=[x])
        t_used += time.perf_counter() - t0
        done_bytes += int(b.kv_lens[x]) * 8 * 128 * 2 * 2 + 2 * 32 * 128 * 2 + 32 * 4
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


def profile_one(name, device, stream, steps, warmup, pk):
    """Run one workload's steps only (used under ncu); prints its timings."""
    if name in ("decode", "decode_fp8", "decode_tc"):
        d = decode_setup(device, "e4m3" if name == "decode_fp8" else "bf16",
                         on_tensor_cores=name == "decode_tc")
        ms = time_steps(lambda: decode_step(d), steps, warmup, stream)
        out = {"workload": "batch_decode", "ms": statistics.median(ms),
               "GB/s": d["bytes"] / (statistics.median(ms) * 1e-3) / 1e9}
    elif name in ("prefill", "prefill_fp8"):
        d = prefill_setup(device) if name == "prefill" else prefill_fp8_setup(device)
        ms = time_steps(lambda: (prefill_append(d), prefill_attn(d)), steps, warmup, stream)
        out = {"workload": "append_prefill", "ms": statistics.median(ms),
               "TFLOP/s": d["flops"] / (statistics.median(ms) * 1e-3) / 1e12}
    elif name.startswith("mixed"):
        P = 1 if name == "mixed1" else 16
        d = mixed_setup(device, P, "NHD" if P == 1 else "HND")
        ms = time_steps(lambda: mixed_step(d), steps, warmup, stream)
        out = {"workload": f"mixed_step_page{P}", "ms": statistics.median(ms)}
    elif name == "cascade":
        d = cascade_setup(device)
        ms = time_steps(lambda: cascade_step(d), steps, warmup, stream)
        out = {"workload": "shared_prompt_decode (cascade)", "ms": statistics.median(ms)}
    else:
        d = ragged_setup(device)
        ms = time_steps(lambda: ragged_step(d), steps, warmup, stream)
        out = {"workload": "ragged_custom_mask", "ms": statistics.median(ms),
               "TFLOP/s(all pairs)": d["flops_all"] / (statistics.median(ms) * 1e-3) / 1e12}
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="pka", choices=["pka", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="all",
                    choices=["all", "decode", "decode_fp8", "decode_tc", "prefill", "prefill_fp8",
                             "ragged", "mixed1", "mixed16", "cascade"],
                    help="all (default) prints the benchmark line; a single workload only runs "
                         "that workload's kernels (for profiling) and prints its numbers")
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

    pk = peaks()
    if args.workload != "all":
        profile_one(args.workload, device, stream, args.steps, args.warmup, pk)
        return
    d = decode_setup(device)

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
    total_ms = max_over_ranks(ev0.elapsed_time(ev1), world, device)
    decode_ms = total_ms / args.steps
    value = job_throughput(d["bytes"], decode_ms, world) / 1e9

    # per-launch duration of the decode step (inputs > L2, so no flush is needed)
    per = time_steps(lambda: decode_step(d), 200, 5, stream)
    step_ms = statistics.median(per)
    achieved = d["bytes"] / (step_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / pk["hbm_gbs"], "traffic": recorded_traffic("decode_kernel<128>"),
            "algorithmic_bytes": d["bytes"],
            "kernel": "decode_kernel<128> (one run(); split states merged in-kernel)",
            "peak_source": pk["source"]}

    # ---- the same decode batch over e4m3 K/V (half the bytes per key)
    d8 = decode_setup(device, "e4m3")
    f8_ms = statistics.median(time_steps(lambda: decode_step(d8), 200, 5, stream))
    fp8_decode = {"workload": "batch_decode over e4m3 K/V (k_scale 0.5, v_scale 2): same requests "
                              "and heads as the bf16 line",
                  "ms_per_step": f8_ms, "GB/s": d8["bytes"] / (f8_ms * 1e-3) / 1e9,
                  "kv_tokens_per_s": d8["kv_tokens"] / (f8_ms * 1e-3),
                  "bf16_kv_tokens_per_s": d["kv_tokens"] / (step_ms * 1e-3),
                  "roofline": {"bound": "hbm", "achieved": d8["bytes"] / (f8_ms * 1e-3) / 1e9,
                               "peak": pk["hbm_gbs"], "unit": "GB/s",
                               "frac": d8["bytes"] / (f8_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                               "traffic": recorded_traffic("decode_kernel<128, e4m3>"),
                               "kernel": "decode_kernel<128, e4m3>"}}
    del d8
    torch.cuda.empty_cache()
    # ---- the same bf16 decode batch through the tensor-core (tcgen05) kernel
    dt = decode_setup(device, on_tensor_cores=True)
    tc_ms = statistics.median(time_steps(lambda: decode_step(dt), 200, 5, stream))
    tc_decode = {"workload": "batch_decode rows on the tcgen05 kernel (decode_on_tensor_cores: "
                             "one query token per item, the 4 qo heads of a kv head in the "
                             "128-row tile)",
                 "ms_per_step": tc_ms, "GB/s": dt["bytes"] / (tc_ms * 1e-3) / 1e9,
                 "vs_decode_kernel": step_ms / tc_ms}
    del dt
    torch.cuda.empty_cache()

    # ---- append + prefill (tensor cores)
    pf = prefill_setup(device)
    app_ms = statistics.median(time_steps(lambda: prefill_append(pf), 50, 5, stream))
    attn_ms = statistics.median(time_steps(lambda: prefill_attn(pf), 50, 5, stream))
    step_ms = statistics.median(time_steps(lambda: (prefill_append(pf), prefill_attn(pf)), 50, 5,
                                           stream))
    attn_tf = pf["flops"] / (attn_ms * 1e-3) / 1e12
    prefill = {"workload": "append_prefill: 16 req, qo_len U[128,1024], prefix U[0,4096] (seed "
                           "1002), causal, page 16, 32/8 heads, D 128, bf16 NHD; "
                           "append_paged_kv_cache then attention",
               "value": pf["flops"] / (step_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "ms_per_step": step_ms, "flops_per_step": pf["flops"],
               "attn_ms": attn_ms, "append_ms": app_ms,
               "append_gbs": pf["append_bytes"] / (app_ms * 1e-3) / 1e9,
               "roofline": {"bound": "tensor", "achieved": attn_tf, "peak": pk["bf16_tflops"],
                            "unit": "TFLOP/s", "frac": attn_tf / pk["bf16_tflops"],
                            "frac_of_sustained": attn_tf / pk.get("bf16_tflops_sustained",
                                                                  pk["bf16_tflops"]),
                            "traffic": recorded_traffic("prefill_kernel<128>"),
                            "kernel": "prefill_kernel<128>",
                            "peak_source": pk["source"]},
               "plan": pf["info"].as_dict()}
    app_gbs = pf["append_bytes"] / (app_ms * 1e-3) / 1e9
    append_roof = {"bound": "hbm", "achieved": app_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                   "frac": app_gbs / pk["hbm_gbs"], "bytes_per_launch": pf["append_bytes"],
                   "bytes_counted": "K and V rows of the appended tokens, read once and "
                                    "written once (2 * 2 * nnz * Hk * D * 2 B)",
                   "traffic": recorded_traffic("append_kernel append_prefill"),
                   "kernel": "append_kernel (append_paged_kv_cache)",
                   "peak_source": pk["source"]}
    del pf
    torch.cuda.empty_cache()
    # ---- the same append-prefill batch over e4m3 pools
    pf8 = prefill_fp8_setup(device)
    f8_attn_ms = statistics.median(time_steps(lambda: prefill_attn(pf8), 50, 5, stream))
    f8_step_ms = statistics.median(time_steps(lambda: (prefill_append(pf8), prefill_attn(pf8)),
                                              50, 5, stream))
    prefill_fp8 = {"workload": "append_prefill over e4m3 K/V (HND, page 16, k_scale 0.5, "
                               "v_scale 2): append_paged_kv_cache quantizes the new rows, then "
                               "attention (keys of the tensor-core rows decoded to a bf16 "
                               "scratch, then the tcgen05 kernel)",
                   "attn_ms": f8_attn_ms, "ms_per_step": f8_step_ms,
                   "tflops_attn": pf8["flops"] / (f8_attn_ms * 1e-3) / 1e12,
                   "value": pf8["flops"] / (f8_step_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                   "kv_scratch_rows": pf8["info"].kv_scratch_rows}
    del pf8
    torch.cuda.empty_cache()
    rg = ragged_setup(device)
    rg_ms = statistics.median(time_steps(lambda: ragged_step(rg), 50, 5, stream))
    import paged_kv_attention_plan_gb300 as pka
    pka.pka_packbits(rg["bools"], rg["packed"])
    rg_attn_ms = statistics.median(time_steps(
        lambda: rg["attn"].run(rg["q"], rg["k"], rg["v"], None, rg["packed"], out=rg["o"],
                               lse=rg["lse"]), 50, 5, stream))
    rg_tf = rg["flops_all"] / (rg_attn_ms * 1e-3) / 1e12
    ragged = {"workload": "ragged_custom_mask: 8 req, qo=kv U[256,2048] (seed 1004), 32/32 "
                          "heads, D 128, ragged K/V, Bernoulli(0.5) OR causal mask; packbits "
                          "then attention",
              "ms_per_step": rg_ms, "attn_ms": rg_attn_ms,
              "tflops_all_pairs": rg["flops_all"] / (rg_ms * 1e-3) / 1e12,
              "tflops_visible_pairs": rg["flops_visible"] / (rg_ms * 1e-3) / 1e12,
              "unit": "TFLOP/s",
              "roofline": {"bound": "tensor", "achieved": rg_tf, "peak": pk["bf16_tflops"],
                           "unit": "TFLOP/s", "frac": rg_tf / pk["bf16_tflops"],
                           "flops_per_launch": rg["flops_all"],
                           "flops_counted": "4*D*Hq per (query, key) pair over all pairs "
                                            "(every 128x128 tile has visible keys)",
                           "traffic": recorded_traffic("prefill_kernel<128> ragged_custom_mask"),
                           "kernel": "prefill_kernel<128> (custom mask, ragged K/V)",
                           "peak_source": pk["source"]}}
    del rg
    torch.cuda.empty_cache()

    mixed = {}
    for P, layout in ((1, "NHD"), (16, "HND")):
        mx = mixed_setup(device, P, layout)
        ms = statistics.median(time_steps(lambda: mixed_step(mx), 20, 3, stream))
        t_roof = mx["decode_bytes"] / (pk["hbm_gbs"] * 1e9) + \
            mx["prefill_flops"] / (pk["bf16_tflops"] * 1e12)
        mixed[f"page{P}_{layout}"] = {
            "ms_per_step": ms, "decode_kv_bytes": mx["decode_bytes"],
            "prefill_flops": mx["prefill_flops"],
            "decode_equiv_gbs": mx["decode_bytes"] / (ms * 1e-3) / 1e9,
            "roofline_ms": t_roof * 1e3, "frac_of_summed_roofline": t_roof / (ms * 1e-3),
            "plan": {k: v for k, v in mx["info"].as_dict().items()
                     if k in ("num_decode_ctas", "num_prefill_ctas", "num_merge_tasks")}}
        del mx
        torch.cuda.empty_cache()
    cs = cascade_setup(device)
    c_ms = statistics.median(time_steps(lambda: cascade_step(cs), 50, 5, stream))
    f_ms = statistics.median(time_steps(lambda: cascade_flat_step(cs), 20, 3, stream))
    t_roof = (cs["own_bytes"] + cs["prompt_bytes"]) / (pk["hbm_gbs"] * 1e9) + \
        cs["shared_flops"] / (pk["bf16_tflops"] * 1e12)
    cascade = {"workload": "shared_prompt_decode: 64 decode rows share a 32768-token prompt, own "
                           "suffix U[512,2048] (seed 1005), page 16 NHD, 32/8 heads, D 128; "
                           "two-level cascade plan vs flat plan listing the prompt pages per "
                           "request",
               "cascade_ms": c_ms, "flat_ms": f_ms, "speedup": f_ms / c_ms,
               "flat_equiv_gbs": cs["flat_bytes"] / (c_ms * 1e-3) / 1e9,
               "flat_gbs": cs["flat_bytes"] / (f_ms * 1e-3) / 1e9,
               "unique_kv_bytes": cs["unique_bytes"], "shared_flops": cs["shared_flops"],
               "roofline_ms": t_roof * 1e3, "frac_of_summed_roofline": t_roof / (c_ms * 1e-3),
               "plan_host_us": cs["plan_us"],
               "plan": {k: v for k, v in cs["info"].as_dict().items()
                        if k in ("num_decode_ctas", "num_prefill_ctas", "num_prefill_items",
                                 "num_merge_tasks", "num_partial_records")}}
    del cs
    torch.cuda.empty_cache()
    mixed["workload"] = ("mixed_step: 8 decodes kv U[32768,131072] + 120 decodes kv U[64,2048] + "
                         "4 chunks of 512 (prefix U[0,8192]) (seed 1003), 32/8 heads, D 128; "
                         "page 1 NHD and page 16 HND; one run() = decode + tensor-core + merge "
                         "kernels; roofline = decode bytes / HBM peak + chunk FLOPs / bf16 peak")

    e2e = e2e_decode(d, min(args.steps, 500), 5, stream, device)
    if world > 1:
        e2e["value"] = job_throughput(d["bytes"], max_over_ranks(e2e["ms_per_step"], world, device),
                                      world) / 1e9
    e2e.pop("ms_per_step")

    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": decode_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": "batch_decode: 64 req, kv_len U[512,4096] (seed 1001), page 16, "
                                   "32/8 heads, D 128, bf16 NHD, split-KV auto + LSE merge",
                       "kv_bytes_per_step": d["kv_bytes"], "bytes_per_step": d["bytes"],
                       "l2": "inputs (604 MB of K/V) larger than L2; no flush",
                       "parallelism": f"replicas x{world}"},
            "roofline": roof,
            "roofline_prefill": prefill["roofline"], "roofline_append": append_roof,
            "roofline_ragged_custom_mask": ragged["roofline"],
            "fp8_kv_decode": fp8_decode, "fp8_kv_append_prefill": prefill_fp8,
            "tensor_core_decode": tc_decode,
            "prefill": prefill,
            "ragged_custom_mask": ragged,
            "mixed_step": mixed, "cascade": cascade, "e2e": e2e,
            "gpu_launches": d["launches"] * args.steps,
            "clocks": clocks.summary(), "plan": d["info"].as_dict(),
            "plan_host_us": d["plan_us"]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, nreq, secs = oracle_sample(seconds_budget=15.0)
        line["cpu_baseline"] = {"value": v, "unit": "GB/s", "cores": cpu_threads(),
                                "kind": "oracle",
                                "sample": f"{nreq} requests of the batch-decode workload, in "
                                          f"order, wrapping after the 64th ({secs:.1f} s of "
                                          f"CPU work)"}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
