"""GPU parity of append_paged_kv_cache, merge_states and packbits.

append and packbits are bit-exact against the oracle; merge_states is within
the bf16 output tolerance and 1e-4 on the base-2 LSE.
"""
import math

import numpy as np
import pytest
import torch

import paged_kv_attention_plan_gb300 as pka
from oracle import ref
from inputs import workloads as W
from tests.gpu_util import LSE_MAX, O_MAX, O_MEAN, bf16, bits_of, f64, i32

pytestmark = pytest.mark.gpu


def _append(b):
    params = pka.make_params(b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.layout)
    k, v = bf16(b.k_pool), bf16(b.v_pool)
    pka.pka_append_paged_kv_cache(params, bf16(b.k_new), bf16(b.v_new), i32(b.qo_indptr),
                                  i32(b.kv_indptr), i32(b.kv_indices), i32(b.last_page_len), k,
                                  v, k.stride(0))
    torch.cuda.synchronize()
    return bits_of(k), bits_of(v)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_append_bit_exact_small(layout, page_size):
    b = W.make_paged_batch(50 + page_size, [3, 1, 0, 17, 40], [6, 2, 5, 40, 41],
                           page_size=page_size, layout=layout, hq=8, hk=2, d=64, append_new=True)
    k, v = _append(b)
    k_ref, v_ref = ref.append_paged_kv_cache(b.k_new, b.v_new, b.qo_indptr, b.k_pool, b.v_pool,
                                             kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                             last_page_len=b.last_page_len,
                                             page_size=page_size, layout=layout)
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def test_append_bit_exact_full_size():
    """The append-prefill workload: 16 requests, 128..1024 new tokens each."""
    b = W.append_prefill()
    k, v = _append(b)
    k_ref, v_ref = ref.append_paged_kv_cache(b.k_new, b.v_new, b.qo_indptr, b.k_pool, b.v_pool,
                                             kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                             last_page_len=b.last_page_len, page_size=16)
    assert np.array_equal(k, k_ref) and np.array_equal(v, v_ref)


def _fp8_pools(b, seed):
    """e4m3 pools of the batch's shape holding random codes everywhere; the
    append overwrites its own slots."""
    rng = np.random.default_rng(seed)
    k8 = W.e4m3_codes(rng, b.k_pool.shape)
    v8 = W.e4m3_codes(rng, b.v_pool.shape)
    return k8, v8


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("page_size,d,scales", [(1, 64, (1.0, 1.0)), (4, 128, (0.3, 2.5)),
                                                (16, 128, (0.004, 0.75))])
def test_append_into_e4m3_pools_bit_exact(layout, page_size, d, scales):
    """bf16 rows appended into e4m3 pools: value / scale rounded to nearest
    even e4m3, saturating (k_scale 0.004 drives most values past 448)."""
    b = W.make_paged_batch(60 + page_size, [3, 1, 0, 17, 40], [6, 2, 5, 40, 41],
                           page_size=page_size, layout=layout, hq=8, hk=2, d=d, append_new=True)
    k8, v8 = _fp8_pools(b, page_size)
    params = pka.make_params(8, 2, d, page_size, layout, kv_dtype="e4m3", k_scale=scales[0],
                             v_scale=scales[1])
    k, v = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    pka.pka_append_paged_kv_cache(params, bf16(b.k_new), bf16(b.v_new), i32(b.qo_indptr),
                                  i32(b.kv_indptr), i32(b.kv_indices), i32(b.last_page_len), k,
                                  v, k.stride(0))
    torch.cuda.synchronize()
    k_ref, v_ref = ref.append_paged_kv_cache(b.k_new, b.v_new, b.qo_indptr, k8, v8,
                                             kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                             last_page_len=b.last_page_len, page_size=page_size,
                                             layout=layout, kv_dtype="e4m3", k_scale=scales[0],
                                             v_scale=scales[1])
    assert np.array_equal(k.cpu().numpy(), k_ref) and np.array_equal(v.cpu().numpy(), v_ref)
    if scales[0] < 0.01:
        assert (k_ref == 0x7E).any() or (k_ref == 0xFE).any()  # saturation was exercised


def test_append_then_decode_e4m3():
    """A decode step over e4m3 pools whose newest token was just appended from
    bf16: the oracle quantizes the same way and decodes the codes."""
    b = W.make_paged_batch(70, [1, 1, 1], [33, 70, 16], page_size=16, hq=32, hk=8, d=128,
                           append_new=True, is_decode=True)
    k8, v8 = _fp8_pools(b, 7)
    params = pka.make_params(32, 8, 128, 16, kv_dtype="e4m3", k_scale=0.5, v_scale=1.5)
    k, v = torch.from_numpy(k8).cuda(), torch.from_numpy(v8).cuda()
    pka.pka_append_paged_kv_cache(params, bf16(b.k_new), bf16(b.v_new), i32(b.qo_indptr),
                                  i32(b.kv_indptr), i32(b.kv_indices), i32(b.last_page_len), k,
                                  v, k.stride(0))
    attn = pka.BatchAttention()
    attn.plan(None, b.kv_indptr, b.last_page_len, num_qo_heads=32, num_kv_heads=8, head_dim=128,
              page_size=16, kv_dtype="e4m3", k_scale=0.5, v_scale=1.5)
    o, lse = attn.run(bf16(b.q), k, v, i32(b.kv_indices))
    torch.cuda.synchronize()
    k_ref, v_ref = ref.append_paged_kv_cache(b.k_new, b.v_new, b.qo_indptr, k8, v8,
                                             kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                             last_page_len=b.last_page_len, page_size=16,
                                             kv_dtype="e4m3", k_scale=0.5, v_scale=1.5)
    o_ref, lse_ref = ref.batch_attention(b.q, k_ref, v_ref, qo_indptr=b.qo_indptr,
                                         kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                         last_page_len=b.last_page_len, page_size=16,
                                         num_qo_heads=32, num_kv_heads=8, kv_dtype="e4m3",
                                         k_scale=0.5, v_scale=1.5)
    from tests.gpu_util import assert_parity
    assert_parity(f64(o), f64(lse), o_ref, lse_ref)


@pytest.mark.parametrize("dim", [64, 128])
def test_merge_states_matches_oracle(dim):
    rng = np.random.default_rng(dim)
    counts = [1, 2, 5, 0, 3, 7, 33, 70]  # rows past 32 states take further rounds of slots
    heads = 3
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    S = int(indptr[-1])
    v = rng.normal(size=(S, heads, dim)).astype(np.float32)
    s = (rng.normal(size=(S, heads)) * 4).astype(np.float32)
    s[1, 0] = -np.inf  # an empty state inside a row
    v[1, 0] = 0
    s[7:10, 1] = -np.inf  # a row whose states are all empty for head 1
    v[7:10, 1] = 0
    r7 = int(indptr[7])
    s[r7 + 40:r7 + 45, 2] = -np.inf  # empty states in the second round of slots
    v[r7 + 40:r7 + 45, 2] = 0
    s[r7 + 65, 0] = 30.0  # the largest statistic of a row in its third round

    v_out = torch.empty(len(counts), heads, dim, dtype=torch.bfloat16, device="cuda")
    s_out = torch.empty(len(counts), heads, dtype=torch.float32, device="cuda")
    pka.pka_merge_states(torch.from_numpy(v).cuda(), torch.from_numpy(s).cuda(), i32(indptr),
                         v_out, s_out)
    torch.cuda.synchronize()
    got_v, got_s = f64(v_out), f64(s_out)
    for r in range(len(counts)):
        for h in range(heads):
            states = [(v[k, h].astype(np.float64), float(s[k, h]))
                      for k in range(indptr[r], indptr[r + 1])]
            if not states:
                want_v, want_s = np.zeros(dim), -math.inf
            else:
                want_v, want_s = ref.merge_states(states)
            err = np.abs(got_v[r, h] - want_v)
            assert err.max() <= O_MAX and err.mean() <= O_MEAN
            if want_s == -math.inf:
                assert got_s[r, h] == -math.inf
            else:
                assert abs(got_s[r, h] - want_s) <= LSE_MAX


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, 12_345_679])
def test_packbits_bit_exact(n):
    rng = np.random.default_rng(n)
    bools = (rng.random(n) < 0.5).astype(np.uint8) * rng.integers(1, 255, size=n).astype(np.uint8)
    out = torch.empty((n + 7) // 8, dtype=torch.uint8, device="cuda")
    pka.pka_packbits(torch.from_numpy(bools).cuda(), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref.packbits_little(bools))


def test_packbits_unaligned_input():
    rng = np.random.default_rng(3)
    bools = (rng.random(1001) < 0.5).astype(np.uint8)
    dev = torch.from_numpy(bools).cuda()
    out = torch.empty(125, dtype=torch.uint8, device="cuda")
    pka.pka_packbits(dev[1:], out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), ref.packbits_little(bools[1:]))
