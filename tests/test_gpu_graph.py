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
from inputs import workloads as W
from tests.gpu_util import assert_parity, bf16, f64, i32, kv_tensor, run_oracle

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


# ---------------------------------------------------------------------------
# Graph mode: one capture serves later plans of other batches
# ---------------------------------------------------------------------------
PAGED_SPECS = [
    ([1, 40, 1, 300, 1], [900, 40, 2000, 700, 17]),          # mixed
    ([1] * 8, [5000, 1, 33, 800, 64, 2, 4096, 100]),          # decode only, at the batch cap
    ([600], [3000]),                                          # one long prefill
    ([2, 1], [2, 9000]),                                      # tiny prefill, long decode
    ([100, 200, 1, 1, 300, 1, 7, 1], [100, 1200, 1, 5, 310, 9000, 7, 64]),
]


@pytest.mark.parametrize("layout,page_size,tc", [("HND", 16, False), ("NHD", 1, False),
                                                ("HND", 16, True)])
def test_graph_mode_capture_serves_new_plans(layout, page_size, tc):
    """tc: decode rows on the tensor-core kernel too (one launch for every row)."""
    hq, hk, d = 32, 8, 128
    max_batch, max_rows = 8, 640
    pool_pages = (20000 + page_size - 1) // page_size + 8 * 2
    batches = [W.make_paged_batch(50 + i, qo, kv, page_size=page_size, layout=layout, hq=hq,
                                  hk=hk, d=d, pool_pages=pool_pages)
               for i, (qo, kv) in enumerate(PAGED_SPECS)]
    shape = batches[0].k_pool.shape
    q_buf = torch.zeros(max_rows, hq, d, dtype=torch.bfloat16, device="cuda")
    o_buf = torch.zeros_like(q_buf)
    lse_buf = torch.zeros(max_rows, hq, dtype=torch.float32, device="cuda")
    k_buf = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
    v_buf = torch.zeros_like(k_buf)
    idx_buf = torch.zeros(pool_pages, dtype=torch.int32, device="cuda")
    attn = pka.BatchAttention()
    stream = torch.cuda.Stream()
    kw = dict(num_qo_heads=hq, num_kv_heads=hk, head_dim=d, page_size=page_size, layout=layout,
              graph_max_batch=max_batch, graph_max_qo_rows=max_rows, decode_on_tensor_cores=tc,
              stream=stream)

    def load(b):
        q_buf[:b.nnz_q].copy_(bf16(b.q))
        k_buf.copy_(bf16(b.k_pool))
        v_buf.copy_(bf16(b.v_pool))
        idx_buf[:len(b.kv_indices)].copy_(i32(b.kv_indices))
        torch.cuda.synchronize()
        attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, **kw)

    def call():
        attn.run(q_buf, k_buf, v_buf, idx_buf, out=o_buf, lse=lse_buf, stream=stream)

    load(batches[0])
    with torch.cuda.stream(stream):
        call()  # first call outside capture (one-time set-up)
    torch.cuda.synchronize()
    ws = (attn.int_ws.data_ptr(), attn.float_ws.data_ptr())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            call()
    torch.cuda.synchronize()
    for b in batches[1:] + batches[:1]:
        load(b)
        assert (attn.int_ws.data_ptr(), attn.float_ws.data_ptr()) == ws
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        assert pka.pka_get_device_error() == 0
        n = b.nnz_q
        assert_parity(f64(o_buf[:n]), f64(lse_buf[:n]), *run_oracle(b))


def test_graph_mode_ragged_custom_mask():
    from oracle import ref
    hq, hk, d = 16, 4, 64
    max_batch, max_rows = 6, 700
    specs = [[300, 1, 200, 100], [1, 1, 1], [700], [64, 65, 1, 190, 2, 3]]
    batches = [W.make_ragged_batch(60 + i, lens, hq=hq, hk=hk, d=d) for i, lens in
               enumerate(specs)]
    max_bits = max(int(np.sum(np.asarray(s) ** 2)) for s in specs)
    q_buf = torch.zeros(max_rows, hq, d, dtype=torch.bfloat16, device="cuda")
    o_buf, lse_buf = torch.zeros_like(q_buf), torch.zeros(max_rows, hq, device="cuda")
    k_buf = torch.zeros(max_rows, hk, d, dtype=torch.bfloat16, device="cuda")
    v_buf = torch.zeros_like(k_buf)
    m_buf = torch.zeros((max_bits + 7) // 8 + 16, dtype=torch.uint8, device="cuda")
    attn = pka.BatchAttention()
    stream = torch.cuda.Stream()
    kw = dict(num_qo_heads=hq, num_kv_heads=hk, head_dim=d, mask_mode="custom", kv_ragged=True,
              graph_max_batch=max_batch, graph_max_qo_rows=max_rows,
              graph_max_kv_tokens=max_rows, stream=stream)

    def load(b):
        n = b.nnz_q
        packed = ref.packbits_little(b.mask_bool.astype(bool))
        q_buf[:n].copy_(bf16(b.q))
        k_buf[:n].copy_(bf16(b.k_pool))
        v_buf[:n].copy_(bf16(b.v_pool))
        m_buf[:len(packed)].copy_(torch.from_numpy(packed))
        torch.cuda.synchronize()
        attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, **kw)
        return packed

    def call():
        attn.run(q_buf, k_buf, v_buf, None, m_buf, out=o_buf, lse=lse_buf, stream=stream)

    load(batches[0])
    with torch.cuda.stream(stream):
        call()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            call()
    torch.cuda.synchronize()
    for b in batches[1:] + batches[:1]:
        packed = load(b)
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        assert pka.pka_get_device_error() == 0
        n = b.nnz_q
        assert_parity(f64(o_buf[:n]), f64(lse_buf[:n]), *run_oracle(b, packed_mask=packed))


def test_graph_mode_e4m3_capture_serves_new_plans():
    """Graph mode over e4m3 pools with rows of qo_len >= 2: the bf16 scratch
    is laid out for graph_max_kv_tokens rows, the dequant kernel reads each
    plan's unit and row counts from the device image, and one captured run()
    serves plans with and without tensor-core rows."""
    hq, hk, d, page_size = 32, 8, 128, 16
    max_batch, max_rows, max_tc_keys = 8, 640, 12000
    specs = PAGED_SPECS
    pool_pages = (20000 + page_size - 1) // page_size + 8 * 2
    # V's scale stays 1: rows that see one or two keys (kv_len 2, 17) output a V
    # row itself, and with V's scale at 2 such values reach 7.5, where one bf16
    # step of the output is 2^-5 and rounding alone nears the 2e-2 bound
    batches = [W.make_paged_batch(70 + i, qo, kv, page_size=page_size, layout="HND", hq=hq,
                                  hk=hk, d=d, pool_pages=pool_pages, kv_dtype="e4m3",
                                  k_scale=0.5, v_scale=1.0)
               for i, (qo, kv) in enumerate(specs)]
    shape = batches[0].k_pool.shape
    q_buf = torch.zeros(max_rows, hq, d, dtype=torch.bfloat16, device="cuda")
    o_buf = torch.zeros_like(q_buf)
    lse_buf = torch.zeros(max_rows, hq, dtype=torch.float32, device="cuda")
    k_buf = torch.zeros(shape, dtype=torch.uint8, device="cuda")
    v_buf = torch.zeros_like(k_buf)
    idx_buf = torch.zeros(pool_pages, dtype=torch.int32, device="cuda")
    attn = pka.BatchAttention()
    stream = torch.cuda.Stream()
    kw = dict(num_qo_heads=hq, num_kv_heads=hk, head_dim=d, page_size=page_size, layout="HND",
              graph_max_batch=max_batch, graph_max_qo_rows=max_rows,
              graph_max_kv_tokens=max_tc_keys, kv_dtype="e4m3", k_scale=0.5, v_scale=1.0,
              stream=stream)

    def load(b):
        q_buf[:b.nnz_q].copy_(bf16(b.q))
        k_buf.copy_(kv_tensor(b.k_pool))
        v_buf.copy_(kv_tensor(b.v_pool))
        idx_buf[:len(b.kv_indices)].copy_(i32(b.kv_indices))
        torch.cuda.synchronize()
        return attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, **kw)

    def call():
        attn.run(q_buf, k_buf, v_buf, idx_buf, out=o_buf, lse=lse_buf, stream=stream)

    info = load(batches[0])
    assert info.kv_scratch_rows > 0
    with torch.cuda.stream(stream):
        call()  # first call outside capture (one-time set-up)
    torch.cuda.synchronize()
    ws = (attn.int_ws.data_ptr(), attn.float_ws.data_ptr())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            call()
    torch.cuda.synchronize()
    for b in batches[1:] + batches[:1]:
        load(b)
        assert (attn.int_ws.data_ptr(), attn.float_ws.data_ptr()) == ws
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        assert pka.pka_get_device_error() == 0
        n = b.nnz_q
        assert_parity(f64(o_buf[:n]), f64(lse_buf[:n]), *run_oracle(b))
