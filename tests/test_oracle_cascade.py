"""Pins of the oracle's multi-level cascade ("KV-Cache layouts", "Multi-level
cascade inference data layout"; "Deep Dive - FlashInfer", "Core mechanism").

The cascade is tied to the already-pinned flat batch attention in two ways
that do not go through cascade_attention's own loop: a shared prefix held
once at an upper level gives the same result as every request listing those
pages in its own page table (the pages' point of prefix sharing), and the
cascade equals the merge of per-level states, each computed by the flat
batch attention of that level alone.
"""
import math

import numpy as np
import pytest

from oracle import ref
from inputs import workloads as W


def _cascade(c, **kw):
    return ref.cascade_attention(c.q, c.k_pool, c.v_pool, levels=c.levels,
                                 page_size=c.page_size, num_qo_heads=c.num_qo_heads,
                                 num_kv_heads=c.num_kv_heads, layout=c.layout,
                                 mask_mode=c.mask_mode, **kw)


def _flat_tables(c):
    """Per-request page tables listing the pages of every level's node."""
    last = c.levels[-1]
    n = len(last["kv_lens"])
    kv_indptr, kv_indices = [0], []
    for r in range(n):
        row = int(last["qo_indptr"][r])
        for lv in c.levels:
            node = ref._node_of(lv["qo_indptr"], row)
            kv_indices.extend(lv["kv_indices"][lv["kv_indptr"][node]:lv["kv_indptr"][node + 1]])
        kv_indptr.append(len(kv_indices))
    return (np.asarray(kv_indptr, np.int32), np.asarray(kv_indices, np.int32),
            last["last_page_len"])


CASES = {
    # qo_lens, own kv lens, shared levels (root first): (requests, kv_len) nodes
    "two_level_decode": ([1, 1, 1, 1, 1], [3, 9, 1, 14, 6], [[(5, 16)]]),
    "two_level_append": ([3, 1, 4, 2], [5, 2, 9, 2], [[(2, 8), (2, 12)]]),
    "three_level": ([2, 1, 3, 1, 1, 2], [4, 7, 3, 1, 9, 2], [[(6, 8)], [(3, 4), (1, 0), (2, 16)]]),
}


@pytest.mark.parametrize("page_size", [1, 4])
@pytest.mark.parametrize("mask_mode", ["causal", "none"])
@pytest.mark.parametrize("case", list(CASES))
def test_shared_prefix_equals_flat_page_tables(case, mask_mode, page_size):
    qo, kv, shared = CASES[case]
    c = W.make_cascade_batch(11, qo, kv, shared, page_size=page_size, hq=4, hk=2, d=16,
                             mask_mode=mask_mode)
    o, lse = _cascade(c)
    kv_indptr, kv_indices, last = _flat_tables(c)
    o_ref, lse_ref = ref.batch_attention(
        c.q, c.k_pool, c.v_pool, qo_indptr=c.levels[-1]["qo_indptr"], kv_indptr=kv_indptr,
        kv_indices=kv_indices, last_page_len=last, page_size=page_size, num_qo_heads=4,
        num_kv_heads=2, mask_mode=mask_mode)
    assert np.allclose(o, o_ref, rtol=0, atol=1e-12)
    assert np.allclose(lse, lse_ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_cascade_is_the_merge_of_level_states(layout):
    # shared node lengths not multiples of the page size: partial shared pages
    c = W.make_cascade_batch(12, [2, 1, 3, 1], [3, 5, 4, 2], [[(4, 13)], [(1, 6), (3, 3)]],
                             page_size=4, layout=layout, hq=8, hk=2, d=16)
    o, lse = _cascade(c)
    states = []
    for li, lv in enumerate(c.levels):
        states.append(ref.batch_attention(
            c.q, c.k_pool, c.v_pool, qo_indptr=lv["qo_indptr"], kv_indptr=lv["kv_indptr"],
            kv_indices=lv["kv_indices"], last_page_len=lv["last_page_len"], page_size=4,
            num_qo_heads=8, num_kv_heads=2, layout=layout,
            mask_mode="none" if li < len(c.levels) - 1 else "causal"))
    for row in range(c.nnz_q):
        for h in range(8):
            om, bm = ref.merge_states([(s[0][row, h], s[1][row, h]) for s in states])
            assert np.allclose(om, o[row, h], rtol=0, atol=1e-12)
            assert math.isclose(bm, lse[row, h], rel_tol=0, abs_tol=1e-12)


def test_node_without_pages_adds_nothing():
    c = W.make_cascade_batch(13, [2, 3], [4, 5], [[(1, 0), (1, 7)]], page_size=4, hq=4, hk=2,
                             d=16)
    assert c.levels[0]["kv_indptr"][1] == 0  # request 0 has no shared pages
    o, lse = _cascade(c)
    last = c.levels[-1]
    o1, lse1 = ref.batch_attention(
        c.q, c.k_pool, c.v_pool, qo_indptr=last["qo_indptr"], kv_indptr=last["kv_indptr"],
        kv_indices=last["kv_indices"], last_page_len=last["last_page_len"], page_size=4,
        num_qo_heads=4, num_kv_heads=2, requests=[0])
    assert np.allclose(o[:2], o1[:2], rtol=0, atol=1e-12)
    assert np.allclose(lse[:2], lse1[:2], rtol=0, atol=1e-12)
    assert not np.allclose(o[2:], ref.batch_attention(
        c.q, c.k_pool, c.v_pool, qo_indptr=last["qo_indptr"], kv_indptr=last["kv_indptr"],
        kv_indices=last["kv_indices"], last_page_len=last["last_page_len"], page_size=4,
        num_qo_heads=4, num_kv_heads=2, requests=[1])[0][2:])


def test_single_level_is_flat_attention():
    c = W.make_cascade_batch(14, [3, 1, 4], [6, 2, 9], [], page_size=4, hq=4, hk=2, d=16)
    o, lse = _cascade(c)
    lv = c.levels[0]
    o_ref, lse_ref = ref.batch_attention(
        c.q, c.k_pool, c.v_pool, qo_indptr=lv["qo_indptr"], kv_indptr=lv["kv_indptr"],
        kv_indices=lv["kv_indices"], last_page_len=lv["last_page_len"], page_size=4,
        num_qo_heads=4, num_kv_heads=2)
    assert np.array_equal(o, o_ref) and np.array_equal(lse, lse_ref)


def test_causal_at_a_shared_level_would_be_caught():
    """A planted mistake (the last level's causal rule applied to a shared
    node whose query rows outnumber its keys) changes the result."""
    c = W.make_cascade_batch(15, [3, 4], [3, 4], [[(2, 4)]], page_size=4, hq=4, hk=2, d=16)
    o, _ = _cascade(c)
    shared = c.levels[0]
    wrong = ref.batch_attention(
        c.q, c.k_pool, c.v_pool, qo_indptr=shared["qo_indptr"], kv_indptr=shared["kv_indptr"],
        kv_indices=shared["kv_indices"], last_page_len=shared["last_page_len"], page_size=4,
        num_qo_heads=4, num_kv_heads=2, mask_mode="none")
    last = c.levels[1]
    own = ref.batch_attention(
        c.q, c.k_pool, c.v_pool, qo_indptr=last["qo_indptr"], kv_indptr=last["kv_indptr"],
        kv_indices=last["kv_indices"], last_page_len=last["last_page_len"], page_size=4,
        num_qo_heads=4, num_kv_heads=2)
    # rows 0..2 of the shared node see all 4 keys; a causal rule with Q=7 > K=4
    # would leave them nothing from that level
    for row in range(3):
        om, _ = ref.merge_states([(wrong[0][row, 0], wrong[1][row, 0]),
                                  (own[0][row, 0], own[1][row, 0])])
        assert np.allclose(om, o[row, 0], atol=1e-12)
        assert not np.allclose(own[0][row, 0], o[row, 0], atol=1e-6)


# ---------------------------------------------------------------------------
# e4m3 pools: the same reading as flat attention (code times the pool scale)
# ---------------------------------------------------------------------------

def _bf16_copy(codes, scale):
    vals = ref.e4m3_to_f64(codes) * scale
    bits = (vals.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    fin = ~np.isnan(vals)
    assert np.array_equal(ref.bf16_bits_to_f64(bits)[fin], vals[fin])  # exact in bf16
    return bits


@pytest.mark.parametrize("layout,page_size", [("NHD", 4), ("HND", 16)])
def test_fp8_cascade_equals_bf16_of_decoded_values(layout, page_size):
    c = W.make_cascade_batch(41, [17, 1, 40, 3], [30, 5, 41, 3], [[(4, 300)], [(2, 64), (2, 20)]],
                             page_size=page_size, layout=layout, hq=8, hk=2, d=64,
                             kv_dtype="e4m3")
    o8, l8 = _cascade(c, kv_dtype="e4m3", k_scale=0.5, v_scale=2.0)
    c16 = W.make_cascade_batch(41, [17, 1, 40, 3], [30, 5, 41, 3],
                               [[(4, 300)], [(2, 64), (2, 20)]], page_size=page_size,
                               layout=layout, hq=8, hk=2, d=64, with_payload=False)
    c16.q, c16.k_pool, c16.v_pool = c.q, _bf16_copy(c.k_pool, 0.5), _bf16_copy(c.v_pool, 2.0)
    o16, l16 = _cascade(c16)
    assert np.all(np.isfinite(o8))
    assert np.allclose(o8, o16, rtol=0, atol=1e-12) and np.allclose(l8, l16, rtol=0, atol=1e-12)


def test_fp8_cascade_equals_flat_page_tables():
    # the shared node fills whole pages, so that the flat tables list every key once
    c = W.make_cascade_batch(42, [9, 1, 1, 22], [12, 40, 7, 30], [[(4, 128)]], page_size=4,
                             hq=8, hk=2, d=64, kv_dtype="e4m3")
    o, lse = _cascade(c, kv_dtype="e4m3", k_scale=0.75, v_scale=1.5)
    kv_indptr, kv_indices, last = _flat_tables(c)
    qo = c.levels[-1]["qo_indptr"]
    of, lf = ref.batch_attention(c.q, c.k_pool, c.v_pool, qo_indptr=qo, kv_indptr=kv_indptr,
                                 kv_indices=kv_indices, last_page_len=last, page_size=4,
                                 num_qo_heads=8, num_kv_heads=2, kv_dtype="e4m3", k_scale=0.75,
                                 v_scale=1.5)
    assert np.allclose(o, of, rtol=0, atol=1e-12) and np.allclose(lse, lf, rtol=0, atol=1e-12)
