"""pka_run_static_scratch: the run entry point that allocates nothing.

It serves callers that cannot call cudaMalloc when they run attention (for
example while a stream is being captured into a CUDA graph, or inside an
engine that owns every byte of device memory and gives the library no
allocator).  The split-KV partial states then live in the library's own
16 MiB static device array instead of a caller workspace.

Checked through the C ABI: on the split batch-decode workload its output
equals pka_run's (caller workspace) within the parity tolerance, on two
calls in a row (the array keeps the previous call's contents); a plan that
needs more scratch than the array holds is refused before any launch.
This file is collected last so that a failure here never hides the others.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_plan_gb300 as pka
from paged_kv_attention_plan_gb300 import workloads as W
from tests.gpu_util import O_MAX, O_MEAN, LSE_MAX, bf16, f64, i32

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
