"""Pins of the oracle's 8-bit (e4m3) K/V path.

* The decoder against the format's fixed points (1.0, the largest finite
  value 448, the smallest normal 2^-6 and subnormal 2^-9, negative zero, the
  NaN) and, for all 256 codes, against PyTorch's float8_e4m3fn conversion (a
  library routine for the same format).
* Attention over e4m3 pools with power-of-two scales equals attention over
  bf16 pools holding the decoded values times the scales (exact: those values
  are bf16 numbers), so the decoding and the place of each scale are tied to
  the bf16 path, which has its own pins.
* A planted decoder with the wrong exponent bias fails the table pin.
"""
import math

import numpy as np
import pytest

from oracle import ref
from inputs import workloads as W


def test_e4m3_fixed_points():
    v = ref.e4m3_to_f64(np.array([0x38, 0x7E, 0x08, 0x01, 0x80, 0xB8, 0x00, 0x07, 0x77], np.uint8))
    assert v[0] == 1.0
    assert v[1] == 448.0            # S.1111.110: the largest finite value
    assert v[2] == 2.0 ** -6        # smallest normal
    assert v[3] == 2.0 ** -9        # smallest subnormal
    assert v[4] == 0.0 and math.copysign(1.0, v[4]) == -1.0
    assert v[5] == -1.0
    assert v[6] == 0.0
    assert v[7] == 7 / 8 * 2.0 ** -6  # largest subnormal
    assert v[8] == 1.875 * 2.0 ** 7   # S.1110.111
    assert np.isnan(ref.e4m3_to_f64(np.array([0x7F, 0xFF], np.uint8))).all()


def test_e4m3_table_matches_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this PyTorch")
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = ref.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    fin = ~np.isnan(want)
    assert np.array_equal(got[fin], want[fin])


def test_planted_wrong_bias_fails_table():
    codes = np.arange(256, dtype=np.uint8)
    good = ref.e4m3_to_f64(codes)
    c = codes.astype(np.int64)
    e, m = (c >> 3) & 15, (c & 7) / 8.0
    wrong = np.where(c >> 7, -1.0, 1.0) * np.where(e == 0, m * 2.0 ** -7, (1 + m) * np.exp2(e - 8.0))
    fin = ~np.isnan(good)
    assert not np.array_equal(good[fin], wrong[fin])


def _bf16_copy(pool_codes, scale):
    vals = ref.e4m3_to_f64(pool_codes) * scale
    f32 = vals.astype(np.float32)
    bits = (f32.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(ref.bf16_bits_to_f64(bits)[~np.isnan(vals)], vals[~np.isnan(vals)])
    return bits


@pytest.mark.parametrize("layout,page_size", [("NHD", 4), ("HND", 3), ("NHD", 1)])
@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.25, 4.0), (8.0, 0.5)])
def test_fp8_attention_equals_bf16_of_decoded_values(layout, page_size, k_scale, v_scale):
    b = W.make_paged_batch(5, np.ones(4, np.int32), [1, 9, 30, 17], page_size=page_size,
                           layout=layout, hq=8, hk=2, d=64, is_decode=True, kv_dtype="e4m3",
                           k_scale=k_scale, v_scale=v_scale)
    kw = dict(qo_indptr=b.qo_indptr, kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
              last_page_len=b.last_page_len, page_size=page_size, num_qo_heads=8,
              num_kv_heads=2, layout=layout)
    o8, l8 = ref.batch_attention(b.q, b.k_pool, b.v_pool, kv_dtype="e4m3", k_scale=k_scale,
                                 v_scale=v_scale, **kw)
    o16, l16 = ref.batch_attention(b.q, _bf16_copy(b.k_pool, k_scale),
                                   _bf16_copy(b.v_pool, v_scale), **kw)
    assert np.allclose(o8, o16, rtol=0, atol=1e-12)
    assert np.allclose(l8, l16, rtol=0, atol=1e-12)


def test_fp8_scales_act_on_scores_and_values():
    """K's scale multiplies every score (the same as a larger softmax scale),
    V's scale multiplies the output and leaves the LSE alone."""
    b = W.make_paged_batch(6, np.ones(3, np.int32), [12, 40, 5], page_size=4, hq=4, hk=2, d=64,
                           is_decode=True, kv_dtype="e4m3")
    kw = dict(qo_indptr=b.qo_indptr, kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
              last_page_len=b.last_page_len, page_size=4, num_qo_heads=4, num_kv_heads=2,
              kv_dtype="e4m3")
    o1, l1 = ref.batch_attention(b.q, b.k_pool, b.v_pool, **kw)
    o2, l2 = ref.batch_attention(b.q, b.k_pool, b.v_pool, v_scale=3.0, **kw)
    assert np.allclose(o2, 3.0 * o1, rtol=1e-12, atol=1e-12) and np.array_equal(l1, l2)
    o3, l3 = ref.batch_attention(b.q, b.k_pool, b.v_pool, k_scale=2.5, **kw)
    o4, l4 = ref.batch_attention(b.q, b.k_pool, b.v_pool, sm_scale=2.5 / 8.0, **kw)
    assert np.allclose(o3, o4, rtol=0, atol=1e-12) and np.allclose(l3, l4, rtol=0, atol=1e-12)


def test_unused_slots_are_nan_codes():
    b = W.make_paged_batch(7, np.ones(2, np.int32), [5, 3], page_size=4, hq=4, hk=2, d=64,
                           is_decode=True, kv_dtype="e4m3")
    assert b.k_pool.dtype == np.uint8
    assert np.isnan(ref.e4m3_to_f64(b.k_pool)).any()  # any over-read would poison a result


# ---------------------------------------------------------------------------
# Quantization to e4m3 (appends into e4m3 pools)
# ---------------------------------------------------------------------------

def _midpoints():
    v = ref.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    return ((v[:-1] + v[1:]) / 2).astype(np.float32)


def test_quantize_round_trips_every_finite_code():
    codes = np.arange(256, dtype=np.uint8)
    vals = ref.e4m3_to_f64(codes)
    fin = ~np.isnan(vals)
    assert np.array_equal(ref.f32_to_e4m3(vals[fin].astype(np.float32)), codes[fin])


def test_quantize_matches_torch_within_range():
    """PyTorch's float8_e4m3fn cast rounds to nearest even; the two agree
    wherever PyTorch does not overflow (|x| <= 464, the midpoint above 448)."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this PyTorch")
    rng = np.random.default_rng(11)
    x = np.concatenate([
        (rng.standard_normal(20000) * np.exp2(rng.integers(-12, 9, 20000))).astype(np.float32),
        _midpoints(), -_midpoints(),                       # exact ties
        np.float32([0.0, -0.0, 2.0 ** -10, 448.0, 464.0, -464.0])])
    x = x[np.abs(x) <= 464.0]
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref.f32_to_e4m3(x), want)


def test_quantize_saturates_and_keeps_nan():
    x = np.float32([465.0, 1e6, np.inf, -500.0, -np.inf, np.nan])
    assert list(ref.f32_to_e4m3(x)) == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F]


def test_planted_ties_away_from_zero_fails():
    mids = _midpoints()
    good = ref.f32_to_e4m3(mids)
    v = ref.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    away = np.searchsorted(v, mids.astype(np.float64), side="left").astype(np.uint8)
    assert not np.array_equal(good, away)


def test_quantizing_append_round_trip():
    """Appending bf16 rows into e4m3 pools stores round(value / scale); reading
    the pools back (the attention gather) yields the decoded codes times the
    scale, and untouched (NaN-coded) slots stay as they were."""
    b = W.make_paged_batch(12, [3, 1, 5], [7, 2, 9], page_size=4, hq=4, hk=2, d=64,
                           append_new=True)
    k8 = np.full(b.k_pool.shape, W.E4M3_NAN_CODE, np.uint8)
    v8 = np.full(b.v_pool.shape, W.E4M3_NAN_CODE, np.uint8)
    ko, vo = ref.append_paged_kv_cache(b.k_new, b.v_new, b.qo_indptr, k8, v8,
                                       kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                       last_page_len=b.last_page_len, page_size=4,
                                       kv_dtype="e4m3", k_scale=0.25, v_scale=3.0)
    want_k = ref.quantize_kv_e4m3(b.k_new, 0.25)
    for r in range(3):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        rows = ref.gather_request_kv(ko, layout="NHD", page_size=4, kv_indptr=b.kv_indptr,
                                     kv_indices=b.kv_indices, req=r, kv_len=int(b.kv_lens[r]))
        assert np.array_equal(rows[-(q1 - q0):], want_k[q0:q1])
    touched = ko != W.E4M3_NAN_CODE
    assert touched.sum() <= b.k_new.size and (vo != W.E4M3_NAN_CODE).sum() <= b.v_new.size


# ---------------------------------------------------------------------------
# Rows with qo_len >= 2 over e4m3 pools (append / prefill): the same reading,
# one scale per pool, for every row length and mask mode
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("layout,page_size", [("HND", 16), ("NHD", 4), ("HND", 1)])
@pytest.mark.parametrize("mask_mode", ["causal", "none"])
def test_fp8_prefill_rows_equal_bf16_of_decoded_values(layout, page_size, mask_mode):
    b = W.make_paged_batch(8, [5, 1, 33, 2], [9, 30, 40, 2], page_size=page_size, layout=layout,
                           hq=8, hk=2, d=64, mask_mode=mask_mode, kv_dtype="e4m3",
                           k_scale=0.5, v_scale=4.0)
    kw = dict(qo_indptr=b.qo_indptr, kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
              last_page_len=b.last_page_len, page_size=page_size, num_qo_heads=8,
              num_kv_heads=2, layout=layout, mask_mode=mask_mode)
    o8, l8 = ref.batch_attention(b.q, b.k_pool, b.v_pool, kv_dtype="e4m3", k_scale=0.5,
                                 v_scale=4.0, **kw)
    o16, l16 = ref.batch_attention(b.q, _bf16_copy(b.k_pool, 0.5), _bf16_copy(b.v_pool, 4.0), **kw)
    assert np.all(np.isfinite(o8))
    assert np.allclose(o8, o16, rtol=0, atol=1e-12)
    assert np.allclose(l8, l16, rtol=0, atol=1e-12)


def test_fp8_prefill_custom_mask_equals_bf16_of_decoded_values():
    b = W.make_paged_batch(9, [6, 3], [10, 7], page_size=4, layout="HND", hq=4, hk=4, d=64,
                           mask_mode="custom", kv_dtype="e4m3", k_scale=2.0, v_scale=0.25)
    rng = np.random.default_rng(9)
    bits = np.concatenate([(rng.random((q, k)) < 0.6).reshape(-1)
                           for q, k in zip(b.qo_lens, b.kv_lens)])
    packed = ref.packbits_little(bits)
    kw = dict(qo_indptr=b.qo_indptr, kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
              last_page_len=b.last_page_len, page_size=4, num_qo_heads=4, num_kv_heads=4,
              layout="HND", mask_mode="custom", packed_mask=packed)
    o8, l8 = ref.batch_attention(b.q, b.k_pool, b.v_pool, kv_dtype="e4m3", k_scale=2.0,
                                 v_scale=0.25, **kw)
    o16, l16 = ref.batch_attention(b.q, _bf16_copy(b.k_pool, 2.0), _bf16_copy(b.v_pool, 0.25),
                                   **kw)
    assert np.allclose(o8, o16, rtol=0, atol=1e-12, equal_nan=False)
    fin = np.isfinite(l16)
    assert np.array_equal(fin, np.isfinite(l8)) and np.allclose(l8[fin], l16[fin], atol=1e-12)


def test_fp8_appended_prefill_attends_to_quantized_rows():
    """Append into e4m3 pools, then attend: the new rows the attention sees
    are the quantized rows (value / scale rounded to e4m3, times scale)."""
    b = W.make_paged_batch(10, [4, 3], [9, 3], page_size=4, layout="HND", hq=4, hk=2, d=64,
                           append_new=True)
    shape = b.k_pool.shape
    k8 = np.full(shape, W.E4M3_NAN_CODE, np.uint8)
    v8 = np.full(shape, W.E4M3_NAN_CODE, np.uint8)
    fin = ~np.isnan(ref.bf16_bits_to_f64(b.k_pool))
    k8[fin] = ref.quantize_kv_e4m3(b.k_pool[fin], 0.5)
    v8[fin] = ref.quantize_kv_e4m3(b.v_pool[fin], 2.0)
    ko, vo = ref.append_paged_kv_cache(b.k_new, b.v_new, b.qo_indptr, k8, v8,
                                       kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                       last_page_len=b.last_page_len, page_size=4, layout="HND",
                                       kv_dtype="e4m3", k_scale=0.5, v_scale=2.0)
    kw = dict(qo_indptr=b.qo_indptr, kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
              last_page_len=b.last_page_len, page_size=4, num_qo_heads=4, num_kv_heads=2,
              layout="HND")
    o8, l8 = ref.batch_attention(b.q, ko, vo, kv_dtype="e4m3", k_scale=0.5, v_scale=2.0, **kw)
    o16, l16 = ref.batch_attention(b.q, _bf16_copy(ko, 0.5), _bf16_copy(vo, 2.0), **kw)
    assert np.all(np.isfinite(o8))
    assert np.allclose(o8, o16, rtol=0, atol=1e-12) and np.allclose(l8, l16, rtol=0, atol=1e-12)
