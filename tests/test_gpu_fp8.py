"""GPU parity of attention over e4m3 K/V pools (one scale per pool) against
the oracle, which decodes each code by the format's definition.

Decode rows: NHD and HND pages, page sizes 1, 3 and 16, head ratios 1/4/8,
head dims 64/128, split auto and fixed, scales of 1 and of 0.37 (K) / 1.9
(V), ragged K/V, and the 64-request batch-decode workload at full size.
Rows with qo_len >= 2 (their keys decoded to a bf16 scratch, then the
tensor-core kernel): mixed decode + prefill batches over the same shapes,
causal, no mask and custom masks, ragged K/V, split modes, and the
append-prefill workload at full size with the new rows quantized into the
pools by append_paged_kv_cache.
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_plan_gb300 as pka
from inputs import workloads as W
from oracle import ref
from tests.gpu_util import (assert_parity, bf16, f64, i32, kv_tensor, plan_item_rows, run_gpu,
                            run_oracle)

pytestmark = pytest.mark.gpu


def _fp8_batch(seed, kv, page_size=4, layout="NHD", hq=8, hk=2, d=64, ks=1.0, vs=1.0):
    return W.make_paged_batch(seed, np.ones(len(kv), np.int32), kv, page_size=page_size,
                              layout=layout, hq=hq, hk=hk, d=d, name="decode_fp8",
                              is_decode=True, kv_dtype="e4m3", k_scale=ks, v_scale=vs)


def test_fp8_worked_lengths():
    b = _fp8_batch(1, [6, 2, 9])
    for split in (("off", 1), ("auto", 1), ("fixed", 1)):
        o, lse, _ = run_gpu(b, split)
        assert_parity(o, lse, *run_oracle(b))


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("page_size", [1, 3, 16])
@pytest.mark.parametrize("hq,hk,d", [(32, 8, 128), (8, 8, 64), (16, 2, 64), (64, 8, 128)])
@pytest.mark.parametrize("scales", [(1.0, 1.0), (0.37, 1.9)])
def test_fp8_decode_shapes(layout, page_size, hq, hk, d, scales):
    rng = np.random.default_rng(page_size * 17 + hq + d)
    kv = rng.integers(1, 600, size=6)
    kv[0] = 1
    b = _fp8_batch(int(rng.integers(1 << 30)), kv, page_size, layout, hq, hk, d, *scales)
    for split in (("auto", 1), ("fixed", 2)):
        o, lse, _ = run_gpu(b, split)
        assert_parity(o, lse, *run_oracle(b))


def test_fp8_ragged_kv():
    lens = np.array([1, 33, 250, 7], np.int32)
    b = W.make_ragged_batch(8, lens, hq=16, hk=4, d=128, mask_mode="none", with_payload=False)
    rng = np.random.default_rng(8)
    b.q = W.normal_bf16_bits(rng, (4, 16, 128))
    b.k_pool = W.e4m3_codes(rng, (int(lens.sum()), 4, 128))
    b.v_pool = W.e4m3_codes(rng, (int(lens.sum()), 4, 128))
    b.qo_lens = np.ones(4, np.int32)
    b.qo_indptr = np.arange(5, dtype=np.int32)
    b.is_decode = True
    b.kv_dtype, b.k_scale, b.v_scale = "e4m3", 0.5, 2.0
    o, lse, _ = run_gpu(b, ("auto", 1))
    assert_parity(o, lse, *run_oracle(b))


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_fp8_batch_decode_full_size(layout):
    b = W.batch_decode(layout=layout, kv_dtype="e4m3", k_scale=0.6, v_scale=1.5)
    o, lse, info = run_gpu(b, ("auto", 1))
    assert info.num_decode_joins > 0
    assert_parity(o, lse, *run_oracle(b))



# ---------------------------------------------------------------------------
# Rows with qo_len >= 2 over e4m3 pools
# ---------------------------------------------------------------------------

def _fp8_mixed(seed, page_size, layout, hq, hk, d, ks, vs, mask="causal"):
    rng = np.random.default_rng(seed)
    qo = rng.integers(2, 200, size=5)
    qo[2] = 1  # a decode row in the same batch
    kv = qo + rng.integers(0, 400, size=5)
    return W.make_paged_batch(seed, qo, kv, page_size=page_size, layout=layout, hq=hq, hk=hk,
                              d=d, mask_mode=mask, kv_dtype="e4m3", k_scale=ks, v_scale=vs)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("page_size", [1, 4, 16])
@pytest.mark.parametrize("hq,hk,d", [(32, 8, 128), (8, 8, 64), (16, 2, 64)])
@pytest.mark.parametrize("scales", [(1.0, 1.0), (0.37, 1.9)])
def test_fp8_prefill_shapes(layout, page_size, hq, hk, d, scales):
    b = _fp8_mixed(page_size * 31 + hq + d, page_size, layout, hq, hk, d, *scales)
    for split in (("auto", 1), ("fixed", 3)):
        o, lse, info = run_gpu(b, split)
        assert info.num_prefill_items > 0 and info.kv_scratch_rows == int(
            np.sum(b.kv_lens[b.qo_lens >= 2]))
        assert_parity(o, lse, *run_oracle(b))


@pytest.mark.parametrize("mask", ["none", "custom"])
def test_fp8_prefill_mask_modes(mask):
    b = _fp8_mixed(77, 16, "HND", 16, 4, 128, 0.5, 2.0, mask=mask)
    packed = None
    if mask == "custom":
        rng = np.random.default_rng(4)
        bits = []
        for q, k in zip(b.qo_lens, b.kv_lens):
            keep = rng.random((q, k)) < 0.5
            keep[:, -1] = True
            bits.append(keep.reshape(-1))
        packed = ref.packbits_little(np.concatenate(bits))
    o, lse, _ = run_gpu(b, ("auto", 1), packed_mask=packed)
    assert_parity(o, lse, *run_oracle(b, packed_mask=packed))


def test_fp8_ragged_prefill_custom_mask():
    b = W.make_ragged_batch(12, [130, 2, 257, 64], hq=8, hk=8, d=128, mask_mode="custom",
                            with_payload=False)
    rng = np.random.default_rng(12)
    n = int(b.kv_indptr[-1])
    b.q = W.normal_bf16_bits(rng, (n, 8, 128))
    b.k_pool = W.e4m3_codes(rng, (n, 8, 128))
    b.v_pool = W.e4m3_codes(rng, (n, 8, 128))
    b.kv_dtype, b.k_scale, b.v_scale = "e4m3", 0.75, 1.5
    packed = ref.packbits_little(b.mask_bool)
    o, lse, info = run_gpu(b, ("auto", 1), packed_mask=packed)
    assert info.kv_scratch_rows == n
    assert_parity(o, lse, *run_oracle(b, packed_mask=packed))


def test_fp8_append_prefill_full_size():
    """The append-prefill workload over e4m3 pools (HND, page 16): the new rows
    are quantized into the pools by append_paged_kv_cache, then attention."""
    b = W.append_prefill(layout="HND", kv_dtype="e4m3", k_scale=0.5, v_scale=2.0)
    params = pka.make_params(32, 8, 128, 16, layout="HND", kv_dtype="e4m3", k_scale=0.5,
                             v_scale=2.0)
    k, v = kv_tensor(b.k_pool), kv_tensor(b.v_pool)
    pka.pka_append_paged_kv_cache(params, bf16(b.k_new), bf16(b.v_new), i32(b.qo_indptr),
                                  i32(b.kv_indptr), i32(b.kv_indices), i32(b.last_page_len), k,
                                  v, k.stride(0))
    attn = pka.BatchAttention()
    info = attn.plan(b.qo_indptr, b.kv_indptr, b.last_page_len, num_qo_heads=32, num_kv_heads=8,
                     head_dim=128, page_size=16, layout="HND", kv_dtype="e4m3", k_scale=0.5,
                     v_scale=2.0)
    assert info.kv_scratch_rows == int(np.sum(b.kv_lens))
    o, lse = attn.run(bf16(b.q), k, v, i32(b.kv_indices))
    torch.cuda.synchronize()
    assert pka.pka_get_device_error() == 0
    kr, vr = ref.append_paged_kv_cache(b.k_new, b.v_new, b.qo_indptr, b.k_pool, b.v_pool,
                                       kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                       last_page_len=b.last_page_len, page_size=16,
                                       layout="HND", kv_dtype="e4m3", k_scale=0.5, v_scale=2.0)
    assert np.array_equal(k.cpu().numpy(), kr) and np.array_equal(v.cpu().numpy(), vr)
    b.k_pool, b.v_pool = kr, vr
    rows = plan_item_rows(attn)
    for r in range(b.batch_size):
        rows.update({int(b.qo_indptr[r]), int(b.qo_indptr[r + 1]) - 1})
    print(f"e4m3 append_prefill: {len(rows)} of {b.nnz_q} rows compared with the oracle")
    o_ref, lse_ref = run_oracle(b, rows=rows)
    assert_parity(f64(o), f64(lse), o_ref, lse_ref, rows=rows)

