"""pka_run_static_scratch: the run entry point that allocates nothing.

It serves callers that cannot call cudaMalloc when they run attention (for
example while a stream is being captured into a CUDA graph, or inside an
engine that owns every byte of device memory and gives the library no
allocator).  The split-KV partial states then live in the library's own
16 MiB static device array instead of a caller workspace.

Checked through the C ABI: on the split batch-decode workload its output
equals pka_run's (caller workspace) within the parity tolerance, on two
calls in a row (the array keeps the previous call's contents); it matches
the CPU oracle on split decode rows (merged inside the decode kernel), on
split prefill rows and on a three-level cascade (both merged by the merge
kernel from states in the static array); a plan that needs more scratch
than the array holds is refused before any launch.
This file is collected last so that a failure here never hides the others.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_plan_gb300 as pka
from inputs import workloads as W
from oracle import ref
from tests.gpu_util import O_MAX, O_MEAN, LSE_MAX, assert_parity, bf16, f64, i32, run_oracle

pytestmark = pytest.mark.gpu

WORKSPACE = 4


def _setup(b, **plan_kw):
    attn = pka.BatchAttention()
    info = attn.plan(None, b.kv_indptr, b.last_page_len, num_qo_heads=b.num_qo_heads,
                     num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, page_size=b.page_size,
                     **plan_kw)
    return attn, info


def _close(o_a, l_a, o_b, l_b):
    err = np.abs(f64(o_a) - f64(o_b))
    assert err.max() <= O_MAX and err.mean() <= O_MEAN
    assert np.abs(f64(l_a) - f64(l_b)).max() <= LSE_MAX


def test_static_scratch_matches_caller_workspace_twice():
    b = W.batch_decode()
    attn, info = _setup(b, split_mode="auto")
    assert info.num_merge_tasks > 0 and info.float_ws_bytes > 0  # the run needs scratch
    q, k, v, idx = bf16(b.q), bf16(b.k_pool), bf16(b.v_pool), i32(b.kv_indices)
    o_ref, lse_ref = attn.run(q, k, v, idx)
    for _ in range(2):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((b.nnz_q, b.num_qo_heads), float("nan"), device="cuda")
        pka.pka_run_static_scratch(attn.handle, attn.params, q, k, v, k.stride(0), idx, None, o,
                                   lse)
        torch.cuda.synchronize()
        _close(o, lse, o_ref, lse_ref)
    assert pka.pka_get_device_error() == 0


def test_static_scratch_refuses_oversized_plan():
    b = W.batch_decode()
    attn, info = _setup(b, split_mode="fixed", fixed_split_pages=1)
    assert info.float_ws_bytes > 16 << 20
    q = bf16(b.q)
    o = torch.empty_like(q)
    s = pka.pka_run_static_scratch(attn.handle, attn.params, q, bf16(b.k_pool[:1]),
                                   bf16(b.v_pool[:1]), 1, i32(b.kv_indices), None, o, None,
                                   check=False)
    assert s == WORKSPACE
    assert "16 MiB" in pka.pka_last_error()


def _run_static(attn, q, k, v, idx, nnz, heads):
    o = torch.full_like(q, float("nan"))
    lse = torch.full((nnz, heads), float("nan"), device="cuda")
    pka.pka_run_static_scratch(attn.handle, attn.params, q, k, v, k.stride(0), idx, None, o, lse)
    torch.cuda.synchronize()
    assert pka.pka_get_device_error() == 0
    return f64(o), f64(lse)


def test_static_scratch_split_decode_matches_oracle():
    b = W.batch_decode(n=16)
    attn, info = _setup(b, split_mode="fixed", fixed_split_pages=16)
    assert info.num_decode_joins > 0
    o_ref, lse_ref = run_oracle(b)
    q, k, v, idx = bf16(b.q), bf16(b.k_pool), bf16(b.v_pool), i32(b.kv_indices)
    for _ in range(2):
        assert_parity(*_run_static(attn, q, k, v, idx, b.nnz_q, b.num_qo_heads), o_ref, lse_ref)


def test_static_scratch_split_prefill_matches_oracle():
    b = W.make_paged_batch(31, [70, 2, 300, 1], [200, 40, 700, 900], page_size=16, hq=16, hk=4,
                           d=128)
    attn = pka.BatchAttention()
    info = attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, num_qo_heads=16, num_kv_heads=4,
                     head_dim=128, page_size=16, split_mode="fixed", fixed_split_pages=12)
    assert info.num_prefill_items > 0 and info.num_merge_tasks > 0
    assert 0 < info.float_ws_bytes <= 16 << 20  # fits the static array
    o_ref, lse_ref = run_oracle(b)
    q, k, v, idx = bf16(b.q), bf16(b.k_pool), bf16(b.v_pool), i32(b.kv_indices)
    for _ in range(2):
        assert_parity(*_run_static(attn, q, k, v, idx, b.nnz_q, 16), o_ref, lse_ref)


def test_static_scratch_cascade_matches_oracle():
    c = W.make_cascade_batch(22, [17, 1, 40, 3, 1, 9], [30, 5, 41, 3, 200, 9],
                             [[(6, 700)], [(2, 64), (1, 0), (3, 129)]], page_size=4, hq=16, hk=2,
                             d=64)
    attn = pka.BatchAttention()
    info = attn.plan_cascade(
        [(lv["qo_indptr"], lv["kv_indptr"], lv["last_page_len"]) for lv in c.levels],
        num_qo_heads=16, num_kv_heads=2, head_dim=64, page_size=4)
    assert info.num_merge_tasks > 0 and info.float_ws_bytes > 0
    o_ref, lse_ref = ref.cascade_attention(c.q, c.k_pool, c.v_pool, levels=c.levels, page_size=4,
                                           num_qo_heads=16, num_kv_heads=2)
    q, k, v, idx = bf16(c.q), bf16(c.k_pool), bf16(c.v_pool), i32(c.kv_indices)
    for _ in range(2):
        assert_parity(*_run_static(attn, q, k, v, idx, c.nnz_q, 16), o_ref, lse_ref)
