"""Pins of the oracle's batched attention against things other than itself.

* Textbook causal attention (torch's scaled_dot_product_attention, float64,
  is_causal=True) on a request whose query rows are its whole history.
* "Deep Dive - FlashInfer", release checklist: incremental decode equals the
  matching rows of full-prefix attention; this pins the bottom-right alignment
  (section "Causality uses logical positions, not page numbers").
* GQA head map of the GPU smoke check in "Deep Dive - FlashInfer" (kv heads
  repeated with repeat_interleave), checked through the library routine.
* Closed forms: constant scores give lse2 = s/ln2 + log2(n) and the mean value.
* Split-then-merge over any cut equals the unsplit state (section "A worked
  split-KV example").
* Page-size-1 view equals the page-size-P view of the same tokens
  ("GPU attention backends: FlashInfer and FlashAttention").
* All-ones custom mask equals no mask; a custom mask holding the causal pattern
  equals causal mode ("KV-Cache layouts", "Mask layout (2D Ragged Tensor)").
* Planted mistakes in the oracle (top-left mask, wrong head map, natural-log
  LSE, missing scale) each fail one of these pins.
"""
import math

import numpy as np
import pytest
import torch

from oracle import ref
from inputs import workloads as W


def _run(b, **kw):
    args = dict(qo_indptr=b.qo_indptr, kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                last_page_len=b.last_page_len, page_size=b.page_size,
                num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads, layout=b.layout,
                mask_mode=b.mask_mode, kv_ragged=b.kv_ragged)
    args.update(kw)
    return ref.batch_attention(b.q, b.k_pool, b.v_pool, **args)


def _dense_request(b, r):
    """Logical K/V rows of request r as float64 torch tensors [K, Hk, D]."""
    k = ref.gather_request_kv(b.k_pool, layout=b.layout, page_size=b.page_size,
                              kv_indptr=b.kv_indptr, kv_indices=b.kv_indices, req=r,
                              kv_len=int(b.kv_lens[r]), kv_ragged=b.kv_ragged)
    v = ref.gather_request_kv(b.v_pool, layout=b.layout, page_size=b.page_size,
                              kv_indptr=b.kv_indptr, kv_indices=b.kv_indices, req=r,
                              kv_len=int(b.kv_lens[r]), kv_ragged=b.kv_ragged)
    return (torch.from_numpy(ref.bf16_bits_to_f64(k)), torch.from_numpy(ref.bf16_bits_to_f64(v)))


def _sdpa(q, k, v, group, causal):
    """torch SDPA, float64, heads first; kv heads repeated for GQA."""
    k = k.repeat_interleave(group, dim=1)
    v = v.repeat_interleave(group, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(
        q.transpose(0, 1), k.transpose(0, 1), v.transpose(0, 1), is_causal=causal)
    return out.transpose(0, 1)


def pin_full_causal_matches_sdpa(oracle=ref):
    """Query rows == full history: oracle equals textbook causal attention."""
    b = W.make_paged_batch(11, [37, 20], [37, 20], page_size=8, hq=4, hk=2, d=16)
    o, _ = oracle.batch_attention(b.q, b.k_pool, b.v_pool, qo_indptr=b.qo_indptr,
                                  kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                  last_page_len=b.last_page_len, page_size=8, num_qo_heads=4,
                                  num_kv_heads=2, mask_mode="causal")
    for r in range(2):
        k, v = _dense_request(b, r)
        q = torch.from_numpy(ref.bf16_bits_to_f64(b.q[b.qo_indptr[r]:b.qo_indptr[r + 1]]))
        want = _sdpa(q, k, v, 2, True).numpy()
        got = o[b.qo_indptr[r]:b.qo_indptr[r + 1]]
        if not np.allclose(got, want, atol=1e-12, rtol=0):
            return False
    return True


def pin_incremental_equals_full_prefix(oracle=ref):
    """Q new rows after a prefix equal the last Q rows of full causal attention."""
    b = W.make_paged_batch(12, [5, 1, 3], [13, 9, 3], page_size=4, hq=4, hk=1, d=16)
    o, _ = oracle.batch_attention(b.q, b.k_pool, b.v_pool, qo_indptr=b.qo_indptr,
                                  kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                  last_page_len=b.last_page_len, page_size=4, num_qo_heads=4,
                                  num_kv_heads=1, mask_mode="causal")
    rng = np.random.default_rng(5)
    for r in range(3):
        K, Q = int(b.kv_lens[r]), int(b.qo_lens[r])
        k, v = _dense_request(b, r)
        qfull = torch.from_numpy(rng.normal(size=(K, 4, 16)))
        qfull[K - Q:] = torch.from_numpy(ref.bf16_bits_to_f64(b.q[b.qo_indptr[r]:b.qo_indptr[r + 1]]))
        want = _sdpa(qfull, k, v, 4, True).numpy()[K - Q:]
        if not np.allclose(o[b.qo_indptr[r]:b.qo_indptr[r + 1]], want, atol=1e-12, rtol=0):
            return False
    return True


def pin_gqa_head_map(oracle=ref):
    """No mask, 8 qo heads on 2 kv heads: equals SDPA with repeat_interleave."""
    b = W.make_paged_batch(13, [6], [11], page_size=4, hq=8, hk=2, d=8, mask_mode="none")
    o, _ = oracle.batch_attention(b.q, b.k_pool, b.v_pool, qo_indptr=b.qo_indptr,
                                  kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                  last_page_len=b.last_page_len, page_size=4, num_qo_heads=8,
                                  num_kv_heads=2, mask_mode="none")
    k, v = _dense_request(b, 0)
    q = torch.from_numpy(ref.bf16_bits_to_f64(b.q))
    want = _sdpa(q, k, v, 4, False).numpy()
    return bool(np.allclose(o, want, atol=1e-12, rtol=0))


def pin_lse_closed_form(oracle=ref):
    """All keys equal: every score is s = scale*q.k, lse2 = s/ln2 + log2(n_visible)."""
    b = W.make_paged_batch(14, [3], [10], page_size=4, hq=2, hk=1, d=16, mask_mode="causal")
    row = b.k_pool[b.kv_indices[0], 0].copy()
    b.k_pool[:] = row  # every slot of every page holds the same key
    o, lse = oracle.batch_attention(b.q, b.k_pool, b.v_pool, qo_indptr=b.qo_indptr,
                                    kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                    last_page_len=b.last_page_len, page_size=4, num_qo_heads=2,
                                    num_kv_heads=1, mask_mode="causal")
    kv = ref.bf16_bits_to_f64(row[0])
    _, v = _dense_request(b, 0)
    for i in range(3):
        nvis = 10 - 3 + i + 1
        for h in range(2):
            s = (ref.bf16_bits_to_f64(b.q[i, h]) @ kv) / 4.0
            if abs(lse[i, h] - (s / math.log(2) + math.log2(nvis))) > 1e-12:
                return False
            if not np.allclose(o[i, h], v[:nvis, 0].numpy().mean(axis=0), atol=1e-12):
                return False
    return True


PINS = [pin_full_causal_matches_sdpa, pin_incremental_equals_full_prefix, pin_gqa_head_map,
        pin_lse_closed_form]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin_holds(pin):
    assert pin()


def test_split_then_merge_equals_unsplit():
    b = W.make_paged_batch(15, [4, 1], [23, 17], page_size=4, hq=4, hk=2, d=16)
    full_o, full_l = _run(b)
    for cuts in ([0, 23], [0, 4, 23], [0, 1, 2, 9, 15, 23], [0, 8, 8, 16, 23]):
        states_o, states_l = [], []
        for t0, t1 in zip(cuts[:-1], cuts[1:]):
            o, l = _run(b, kv_range=(t0, t1))
            states_o.append(o)
            states_l.append(l)
        for row in range(b.nnz_q):
            for h in range(4):
                o, l = ref.merge_states([(so[row, h], sl[row, h]) for so, sl in zip(states_o, states_l)])
                assert np.max(np.abs(o - full_o[row, h])) < 1e-12
                assert abs(l - full_l[row, h]) < 1e-12


def test_page_size_1_view_equals_page_size_p():
    bp = W.make_paged_batch(16, [2, 1], [5, 6], page_size=4, hq=4, hk=2, d=16)
    # the same logical tokens laid out one token per page
    toks_k = [_dense_request(bp, r)[0] for r in range(2)]
    kv_lens = [5, 6]
    total = sum(kv_lens)
    perm = np.random.default_rng(0).permutation(total)
    k1 = np.zeros((total, 1, 2, 16), np.uint16)
    v1 = np.zeros((total, 1, 2, 16), np.uint16)
    indices, c = [], 0
    for r in range(2):
        kr = ref.gather_request_kv(bp.k_pool, layout="NHD", page_size=4, kv_indptr=bp.kv_indptr,
                                   kv_indices=bp.kv_indices, req=r, kv_len=kv_lens[r])
        vr = ref.gather_request_kv(bp.v_pool, layout="NHD", page_size=4, kv_indptr=bp.kv_indptr,
                                   kv_indices=bp.kv_indices, req=r, kv_len=kv_lens[r])
        for j in range(kv_lens[r]):
            k1[perm[c], 0] = kr[j]
            v1[perm[c], 0] = vr[j]
            indices.append(int(perm[c]))
            c += 1
    assert len(toks_k) == 2
    o4, l4 = _run(bp)
    o1, l1 = ref.batch_attention(bp.q, k1, v1, qo_indptr=bp.qo_indptr, kv_indptr=[0, 5, 11],
                                 kv_indices=indices, last_page_len=[1, 1], page_size=1,
                                 num_qo_heads=4, num_kv_heads=2, mask_mode="causal")
    assert np.array_equal(o1, o4) and np.array_equal(l1, l4)


def test_nhd_equals_hnd():
    bn = W.make_paged_batch(17, [3, 2], [9, 14], page_size=4, hq=4, hk=2, d=8, layout="NHD")
    bh = W.make_paged_batch(17, [3, 2], [9, 14], page_size=4, hq=4, hk=2, d=8, layout="HND")
    on, ln = _run(bn)
    oh, lh = _run(bh)
    assert np.array_equal(on, oh) and np.array_equal(ln, lh)


def test_custom_mask_special_cases():
    b = W.make_paged_batch(18, [3, 1, 4], [6, 2, 9], page_size=4, hq=4, hk=2, d=16)
    ones = ref.packbits_little(np.ones(sum(q * k for q, k in zip([3, 1, 4], [6, 2, 9])), np.uint8))
    o_none, l_none = _run(b, mask_mode="none")
    o_all, l_all = _run(b, mask_mode="custom", packed_mask=ones)
    assert np.array_equal(o_none, o_all) and np.array_equal(l_none, l_all)
    causal_bits = []
    for qlen, klen in zip([3, 1, 4], [6, 2, 9]):
        for i in range(qlen):
            causal_bits += [int(ref.causal_visible(i, j, qlen, klen)) for j in range(klen)]
    o_c, l_c = _run(b, mask_mode="causal")
    o_m, l_m = _run(b, mask_mode="custom", packed_mask=ref.packbits_little(causal_bits))
    assert np.array_equal(o_c, o_m) and np.array_equal(l_c, l_m)


def test_decode_row_is_plain_softmax():
    b = W.make_paged_batch(19, [1], [7], page_size=4, hq=2, hk=1, d=8)
    o_c, l_c = _run(b, mask_mode="causal")
    o_n, l_n = _run(b, mask_mode="none")
    assert np.array_equal(o_c, o_n) and np.array_equal(l_c, l_n)


def test_uniform_value_invariant():
    b = W.make_paged_batch(20, [4], [10], page_size=4, hq=2, hk=1, d=8)
    c = W.f32_to_bf16_bits(np.linspace(-1, 1, 8, dtype=np.float32))
    b.v_pool[:] = c
    o, _ = _run(b)
    assert np.allclose(o, ref.bf16_bits_to_f64(c)[None, None, :], atol=1e-12)


def test_empty_and_fully_masked_rows():
    b = W.make_paged_batch(21, [0, 2], [3, 4], page_size=4, hq=2, hk=1, d=8)
    bits = ref.packbits_little([0] * 8)  # request 1: both rows see nothing
    o, l = _run(b, mask_mode="custom", packed_mask=bits)
    assert np.all(o == 0) and np.all(l == -math.inf)
    o, l = _run(b)
    assert o.shape[0] == 2 and np.all(np.isfinite(o))


def test_causal_rejects_short_history():
    b = W.make_paged_batch(22, [3], [3], page_size=4, hq=2, hk=1, d=8)
    with pytest.raises(ValueError):
        _run(b, kv_indptr=b.kv_indptr, last_page_len=np.array([2], np.int32))


# ---------------------------------------------------------------------------
# Planted mistakes: each variant of the oracle must fail at least one pin.
# ---------------------------------------------------------------------------

def test_planted_top_left_mask_is_caught(monkeypatch):
    monkeypatch.setattr(ref, "causal_visible", lambda i, j, q, k: j <= i)
    assert not pin_incremental_equals_full_prefix()


def test_planted_head_map_is_caught(monkeypatch):
    orig = ref.batch_attention

    def wrong(*a, **kw):
        # read kv head h % Hk instead of h // g by permuting qo heads
        hq = kw["num_qo_heads"]
        hk = kw["num_kv_heads"]
        perm = [(h % hk) * (hq // hk) + h // hk for h in range(hq)]
        q = np.asarray(a[0])[:, perm]
        o, l = orig(q, *a[1:], **kw)
        inv = np.argsort(perm)
        return o[:, inv], l[:, inv]

    class M:
        batch_attention = staticmethod(wrong)
    assert not pin_gqa_head_map(oracle=M)


def test_planted_natural_log_lse_is_caught(monkeypatch):
    orig = ref.direct_state

    def wrong(s, v):
        o, b = orig(s, v)
        return o, b * math.log(2)
    monkeypatch.setattr(ref, "direct_state", wrong)
    assert not pin_lse_closed_form()


def test_planted_missing_scale_is_caught(monkeypatch):
    orig = ref.batch_attention
    monkeypatch.setattr(ref, "batch_attention", lambda *a, **kw: orig(*a, sm_scale=1.0, **kw))
    assert not pin_full_causal_matches_sdpa()
