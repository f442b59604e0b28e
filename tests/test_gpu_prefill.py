"""GPU parity of the tensor-core append / prefill path (qo_len >= 2 rows).

Covers the worked three-request batch (printed and seeded page ids), the GPU
smoke-check shape of "Deep Dive - FlashInfer" (32/8 heads, D 128, page size
4) in bf16, NHD and HND pages of sizes 1..32, head ratios 1/2/4/8, head_dim
64/128, causal / none / custom masks, ragged K/V, mixed decode + prefill
batches, every split mode, and the append-prefill, mixed-step and ragged-mask
workloads at full size (against the oracle on the first and last token of
every query tile of every work item of the real plan).
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_plan_gb300 as pka
from oracle import ref
from inputs import workloads as W
from tests.gpu_util import assert_parity, bf16, f64, i32, plan_item_rows, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

SPLITS = [("off", 1), ("auto", 1), ("fixed", 1), ("fixed", 2), ("fixed", 7)]


@pytest.mark.parametrize("split", SPLITS)
@pytest.mark.parametrize("literal", [False, True])
def test_worked_example(split, literal):
    b = W.worked_example(literal_pages=literal)
    o, lse, _ = run_gpu(b, split)
    assert_parity(o, lse, *run_oracle(b))


@pytest.mark.parametrize("split", [("auto", 1), ("fixed", 1)])
def test_smoke_check_shape(split):
    b = W.worked_example(literal_pages=True, hq=32, hk=8, d=128)
    o, lse, _ = run_gpu(b, split)
    assert_parity(o, lse, *run_oracle(b))


def _rand_batch(seed, page_size, layout, hq, hk, d, mask="causal", n=5):
    rng = np.random.default_rng(seed)
    qo = rng.integers(2, 300, size=n)
    kv = qo + rng.integers(0, 500, size=n)
    qo[1] = 2
    return W.make_paged_batch(seed, qo, kv, page_size=page_size, layout=layout, hq=hq, hk=hk,
                              d=d, mask_mode=mask)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("page_size", [1, 4, 16, 32])
@pytest.mark.parametrize("hq,hk,d", [(32, 8, 128), (8, 8, 64), (16, 8, 128), (16, 2, 64)])
def test_prefill_shapes(layout, page_size, hq, hk, d):
    b = _rand_batch(page_size * 7 + hq + d, page_size, layout, hq, hk, d)
    for split in (("auto", 1), ("fixed", 8)):
        o, lse, _ = run_gpu(b, split)
        assert_parity(o, lse, *run_oracle(b))


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_prefill_mask_modes(mask):
    b = _rand_batch(91, 16, "NHD", 32, 8, 128, mask=mask)
    o, lse, _ = run_gpu(b, ("off", 1))
    assert_parity(o, lse, *run_oracle(b))


def test_prefill_custom_mask_paged():
    b = _rand_batch(92, 16, "NHD", 16, 4, 128, mask="custom")
    rng = np.random.default_rng(3)
    bits = []
    for q, k in zip(b.qo_lens, b.kv_lens):
        keep = rng.random((q, k)) < 0.5
        keep[:, -1] = True
        bits.append(keep.reshape(-1))
    packed = ref.packbits_little(np.concatenate(bits))
    for split in (("off", 1), ("fixed", 3)):
        o, lse, _ = run_gpu(b, split, packed_mask=packed)
        assert_parity(o, lse, *run_oracle(b, packed_mask=packed))


def test_ragged_custom_mask_small():
    b = W.make_ragged_batch(93, [130, 2, 257, 64], hq=8, hk=8, d=128, mask_mode="custom")
    packed = ref.packbits_little(b.mask_bool)
    o, lse, _ = run_gpu(b, ("auto", 1), packed_mask=packed)
    assert_parity(o, lse, *run_oracle(b, packed_mask=packed))


def test_mixed_decode_and_prefill_small():
    qo = np.array([1, 40, 1, 1, 130, 2, 1], np.int32)
    kv = np.array([900, 40, 33, 2000, 600, 9, 1], np.int32)
    for P, layout in ((1, "NHD"), (16, "HND")):
        b = W.make_paged_batch(94 + P, qo, kv, page_size=P, layout=layout, hq=32, hk=8, d=128)
        o, lse, info = run_gpu(b, ("auto", 1))
        assert info.num_decode_items > 0 and info.num_prefill_items > 0
        assert_parity(o, lse, *run_oracle(b))


def _sample_rows(b, per_req=3, seed=0):
    rng = np.random.default_rng(seed)
    rows = set()
    for r in range(b.batch_size):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        if q1 > q0:
            rows.update({q0, q1 - 1})
            rows.update(int(x) for x in rng.integers(q0, q1, size=per_req))
    return rows


def test_append_prefill_full_size():
    """16 requests: append_paged_kv_cache writes the new K/V, then attention."""
    b = W.append_prefill()
    params = pka.make_params(32, 8, 128, 16)
    k, v = bf16(b.k_pool), bf16(b.v_pool)
    pka.pka_append_paged_kv_cache(params, bf16(b.k_new), bf16(b.v_new), i32(b.qo_indptr),
                                  i32(b.kv_indptr), i32(b.kv_indices), i32(b.last_page_len), k,
                                  v, k.stride(0))
    attn = pka.BatchAttention()
    attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, num_qo_heads=32, num_kv_heads=8,
              head_dim=128, page_size=16)
    o, lse = attn.run(bf16(b.q), k, v, i32(b.kv_indices))
    torch.cuda.synchronize()
    assert pka.pka_get_device_error() == 0
    # the oracle sees the pool with the appended rows written by its own append
    kr, vr = ref.append_paged_kv_cache(b.k_new, b.v_new, b.qo_indptr, b.k_pool, b.v_pool,
                                       kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                       last_page_len=b.last_page_len, page_size=16)
    b.k_pool, b.v_pool = kr, vr
    # both ends of every query tile of every work item, plus random rows
    rows = _sample_rows(b) | plan_item_rows(attn)
    print(f"append_prefill: {len(rows)} of {b.nnz_q} rows compared with the oracle "
          f"({attn.info.num_prefill_items} items, {attn.info.num_prefill_ctas} CTAs)")
    o_ref, lse_ref = run_oracle(b, rows=rows)
    assert_parity(f64(o), f64(lse), o_ref, lse_ref, rows=rows)


def test_ragged_custom_mask_full_size():
    b = W.ragged_custom_mask()
    bools = torch.from_numpy(b.mask_bool).cuda()
    packed = torch.empty((bools.numel() + 7) // 8, dtype=torch.uint8, device="cuda")
    pka.pka_packbits(bools, packed)
    torch.cuda.synchronize()
    packed_ref = ref.packbits_little(b.mask_bool)
    assert np.array_equal(packed.cpu().numpy(), packed_ref)
    attn = pka.BatchAttention()
    o, lse, _ = run_gpu(b, ("auto", 1), packed_mask=packed_ref, attn=attn)
    rows = _sample_rows(b, per_req=2) | plan_item_rows(attn)
    print(f"ragged_custom_mask: {len(rows)} of {b.nnz_q} rows compared with the oracle "
          f"({attn.info.num_prefill_items} items, {attn.info.num_prefill_ctas} CTAs)")
    o_ref, lse_ref = run_oracle(b, packed_mask=packed_ref, rows=rows)
    assert_parity(o, lse, o_ref, lse_ref, rows=rows)


@pytest.mark.parametrize("page_size,layout", [(1, "NHD"), (16, "HND")])
def test_mixed_step_full_size(page_size, layout):
    """8 long decodes (32K-131K keys), 120 short decodes and 4 prefill chunks of
    512 tokens in one plan; every decode row and both ends of every query tile
    of the tensor-core items against the oracle."""
    from inputs import workloads as Wk
    b = Wk.mixed_step(page_size=page_size, layout=layout, with_payload=False)
    # payload drawn on the device (seeded), then copied to the host for the oracle
    hk, d = 8, 128
    pool = int(b.extra["pool_pages"])
    shape = (pool, page_size, hk, d) if layout == "NHD" else (pool, hk, page_size, d)
    g = torch.Generator(device="cuda").manual_seed(1003)
    k = torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn((b.nnz_q, 32, d), generator=g, device="cuda").to(torch.bfloat16)
    attn = pka.BatchAttention()
    info = attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, num_qo_heads=32, num_kv_heads=8,
                     head_dim=128, page_size=page_size, layout=layout)
    assert info.num_decode_items > 0 and info.num_prefill_items > 0 and info.num_merge_tasks > 0
    o, lse = attn.run(q, k, v, i32(b.kv_indices))
    torch.cuda.synchronize()
    assert pka.pka_get_device_error() == 0
    # every decode row (each split piece's row among them), both ends of every
    # query tile of every tensor-core item, and the last row of every chunk
    rows = plan_item_rows(attn)
    for r in range(b.batch_size):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        rows.update({q0, q1 - 1})
    print(f"mixed_step page {page_size}: {len(rows)} of {b.nnz_q} rows compared with the "
          f"oracle ({info.num_decode_items} decode items, {info.num_prefill_items} tensor-core "
          f"items, {info.num_merge_tasks} merge tasks)")
    b.q = q.view(torch.int16).cpu().numpy().view(np.uint16)
    b.k_pool = k.view(torch.int16).cpu().numpy().view(np.uint16)
    b.v_pool = v.view(torch.int16).cpu().numpy().view(np.uint16)
    o_ref, lse_ref = run_oracle(b, rows=rows)
    assert_parity(f64(o), f64(lse), o_ref, lse_ref, rows=rows)


def test_custom_mask_unaligned_buffer():
    """A packed mask that starts at an odd address (byte loads only)."""
    b = W.make_ragged_batch(95, [200, 67], hq=8, hk=8, d=64, mask_mode="custom")
    packed = ref.packbits_little(b.mask_bool)
    store = torch.zeros(packed.size + 1, dtype=torch.uint8, device="cuda")
    store[1:] = torch.from_numpy(packed).cuda()
    attn = pka.BatchAttention()
    attn.plan(b.qo_indptr, b.kv_indptr, None, num_qo_heads=8, num_kv_heads=8, head_dim=64,
              mask_mode="custom", kv_ragged=True)
    o, lse = attn.run(bf16(b.q), bf16(b.k_pool), bf16(b.v_pool), None, store[1:])
    torch.cuda.synchronize()
    assert_parity(f64(o), f64(lse), *run_oracle(b, packed_mask=packed))


@pytest.mark.parametrize("d", [64, 128])
def test_output_only_16_byte_aligned(d):
    """O at an address that is 16- but not 32-byte aligned (the epilogue's
    16-byte store path)."""
    b = W.make_paged_batch(96, [70, 3, 130], [90, 40, 130], page_size=8, hq=8, hk=2, d=d)
    attn = pka.BatchAttention()
    attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, num_qo_heads=8, num_kv_heads=2,
              head_dim=d, page_size=8, split_mode="off")
    n = b.nnz_q * 8 * d
    store = torch.zeros(n + 8, dtype=torch.bfloat16, device="cuda")
    out = store[8:].view(b.nnz_q, 8, d)
    assert out.data_ptr() % 32 == 16
    o, lse = attn.run(bf16(b.q), bf16(b.k_pool), bf16(b.v_pool), i32(b.kv_indices), out=out)
    torch.cuda.synchronize()
    assert_parity(f64(o), f64(lse), *run_oracle(b))


@pytest.mark.parametrize("qo,kv,last", [([0], [0], []), ([0, 0, 0], [0, 2, 3], [3, 1])])
def test_run_without_query_rows(qo, kv, last):
    """Empty batches run without launching anything, with empty (null) buffers."""
    attn = pka.BatchAttention()
    info = attn.plan(np.asarray(qo, np.int32), np.asarray(kv, np.int32),
                     np.asarray(last, np.int32), num_qo_heads=8, num_kv_heads=2, head_dim=64,
                     page_size=4)
    assert info.nnz_qo == 0
    q = torch.empty((0, 8, 64), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((4, 4, 2, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = attn.run(q, pool, pool, torch.zeros(3, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert o.shape == (0, 8, 64) and lse.shape == (0, 8)
    assert pka.pka_get_device_error() == 0
