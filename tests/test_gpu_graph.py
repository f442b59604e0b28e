"""run() under CUDA-graph capture ("Deep Dive - FlashInfer", "Plan then run":
plan does host work and copies, compatible run calls can be captured).

The plan is made outside the capture; one run() (decode kernel, tensor-core
kernel and merge kernel of a mixed batch) is captured and replayed with new
query contents and a remapped page table in the same buffers.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_plan_gb300 as pka
from paged_kv_attention_plan_gb300 import workloads as W
from tests.gpu_util import assert_parity, bf16, f64, i32, run_oracle

pytestmark = pytest.mark.gpu


def test_captured_run_replays_with_new_contents():
    qo = np.array([1, 40, 1, 300, 1], np.int32)
    kv = np.array([900, 40, 2000, 700, 17], np.int32)
    b = W.make_paged_batch(96, qo, kv, page_size=16, hq=32, hk=8, d=128)
    attn = pka.BatchAttention()
    info = attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, num_qo_heads=32, num_kv_heads=8,
                     head_dim=128, page_size=16)
    assert info.num_decode_items and info.num_prefill_items and info.num_merge_tasks
    q, k, v, idx = bf16(b.q), bf16(b.k_pool), bf16(b.v_pool), i32(b.kv_indices)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[0], 32, dtype=torch.float32, device="cuda")
    attn.run(q, k, v, idx, out=o, lse=lse)  # first call outside capture (one-time set-up)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            attn.run(q, k, v, idx, out=o, lse=lse, stream=stream)
    torch.cuda.synchronize()
    for seed in (1, 2):
        rng = np.random.default_rng(seed)
        # new query rows and a permuted page pool, written into the same buffers
        b.q = W.normal_bf16_bits(rng, b.q.shape)
        perm = rng.permutation(b.k_pool.shape[0])
        k2, v2 = np.empty_like(b.k_pool), np.empty_like(b.v_pool)
        k2[perm], v2[perm] = b.k_pool, b.v_pool
        b.k_pool, b.v_pool, b.kv_indices = k2, v2, perm[b.kv_indices].astype(np.int32)
        q.copy_(bf16(b.q))
        k.copy_(bf16(b.k_pool))
        v.copy_(bf16(b.v_pool))
        idx.copy_(i32(b.kv_indices))
        graph.replay()
        torch.cuda.synchronize()
        assert pka.pka_get_device_error() == 0
        assert_parity(f64(o), f64(lse), *run_oracle(b))
