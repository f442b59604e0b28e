"""GPU parity of multi-level cascade attention against the oracle ("KV-Cache
layouts", "Multi-level cascade inference data layout").

One plan holds the work of every level; each piece writes an fp32 partial
state and the merge kernel combines each row's states from all levels in the
same run().  Covers shared system prompts under decode rows, three-level
trees with append rows and nodes without pages, page size 1 HND, no mask,
and every split mode; the same trees over e4m3 pools (decode nodes read the
codes, tensor-core nodes a bf16 scratch of each node's keys).
"""
import numpy as np
import pytest
import torch

import paged_kv_attention_plan_gb300 as pka
from oracle import ref
from inputs import workloads as W
from tests.gpu_util import assert_parity, bf16, f64, i32, kv_tensor

pytestmark = pytest.mark.gpu


def run_cascade(c, split=("auto", 1)):
    attn = pka.BatchAttention()
    info = attn.plan_cascade(
        [(lv["qo_indptr"], lv["kv_indptr"], lv["last_page_len"]) for lv in c.levels],
        num_qo_heads=c.num_qo_heads, num_kv_heads=c.num_kv_heads, head_dim=c.head_dim,
        page_size=c.page_size, layout=c.layout, mask_mode=c.mask_mode, split_mode=split[0],
        fixed_split_pages=split[1])
    o, lse = attn.run(bf16(c.q), bf16(c.k_pool), bf16(c.v_pool), i32(c.kv_indices))
    torch.cuda.synchronize()
    assert pka.pka_get_device_error() == 0
    return f64(o), f64(lse), info


def oracle(c):
    return ref.cascade_attention(c.q, c.k_pool, c.v_pool, levels=c.levels,
                                 page_size=c.page_size, num_qo_heads=c.num_qo_heads,
                                 num_kv_heads=c.num_kv_heads, layout=c.layout,
                                 mask_mode=c.mask_mode)


CASES = {
    "shared_prompt_decode": lambda: W.make_cascade_batch(
        21, [1] * 64, np.random.default_rng(0).integers(1, 512, 64), [[(64, 4096)]],
        page_size=16, hq=32, hk=8, d=128),
    "three_levels_append": lambda: W.make_cascade_batch(
        22, [17, 1, 40, 3, 1, 9], [30, 5, 41, 3, 200, 9], [[(6, 700)], [(2, 64), (1, 0), (3, 129)]],
        page_size=4, hq=16, hk=2, d=64),
    "page1_hnd": lambda: W.make_cascade_batch(
        23, [5, 1, 1, 300], [5, 80, 2, 400], [[(4, 333)]], page_size=1, layout="HND", hq=8, hk=8,
        d=64),
    "no_mask_hnd16": lambda: W.make_cascade_batch(
        24, [4, 1, 6, 1], [2, 7, 3, 40], [[(2, 100), (2, 5)]], page_size=16, layout="HND", hq=32,
        hk=8, d=128, mask_mode="none"),
    "shared_prefix_prefill": lambda: W.make_cascade_batch(
        25, [128] * 8, [128] * 8, [[(8, 2000)]], page_size=16, hq=32, hk=8, d=128),
}


@pytest.mark.parametrize("split", [("auto", 1), ("off", 1), ("fixed", 3)])
@pytest.mark.parametrize("case", list(CASES))
def test_cascade_parity(case, split):
    c = CASES[case]()
    o, lse, info = run_cascade(c, split)
    assert info.num_merge_tasks == c.nnz_q * c.num_qo_heads
    assert_parity(o, lse, *oracle(c))


def test_cascade_equals_flat_plan_of_the_same_tokens():
    """Prefix held once at the root vs. listed in every request's own page
    table: the GPU's two paths agree within the parity tolerance."""
    c = CASES["shared_prompt_decode"]()
    o, lse, _ = run_cascade(c)
    root, own = c.levels
    kv_indptr, kv_indices = [0], []
    for r in range(len(own["kv_lens"])):
        kv_indices += list(root["kv_indices"]) + list(
            own["kv_indices"][own["kv_indptr"][r]:own["kv_indptr"][r + 1]])
        kv_indptr.append(len(kv_indices))
    attn = pka.BatchAttention()
    attn.plan(None, np.asarray(kv_indptr, np.int32), own["last_page_len"], num_qo_heads=32,
              num_kv_heads=8, head_dim=128, page_size=16)
    o2, lse2 = attn.run(bf16(c.q), bf16(c.k_pool), bf16(c.v_pool),
                        i32(np.asarray(kv_indices, np.int32)))
    torch.cuda.synchronize()
    assert_parity(o, lse, f64(o2), f64(lse2))


FP8_CASES = {
    "shared_prompt_decode": lambda: W.make_cascade_batch(
        31, [1] * 32, np.random.default_rng(1).integers(1, 512, 32), [[(32, 2048)]],
        page_size=16, layout="HND", hq=32, hk=8, d=128, kv_dtype="e4m3"),
    "three_levels_append": lambda: W.make_cascade_batch(
        32, [17, 1, 40, 3, 1, 9], [30, 5, 41, 3, 200, 9],
        [[(6, 700)], [(2, 64), (1, 0), (3, 129)]], page_size=4, hq=16, hk=2, d=64,
        kv_dtype="e4m3"),
    "shared_prefix_prefill": lambda: W.make_cascade_batch(
        33, [128] * 4, [128] * 4, [[(4, 1500)]], page_size=16, layout="HND", hq=32, hk=8,
        d=128, kv_dtype="e4m3"),
}


@pytest.mark.parametrize("split", [("auto", 1), ("fixed", 3)])
@pytest.mark.parametrize("case", list(FP8_CASES))
def test_fp8_cascade_parity(case, split):
    c = FP8_CASES[case]()
    attn = pka.BatchAttention()
    info = attn.plan_cascade(
        [(lv["qo_indptr"], lv["kv_indptr"], lv["last_page_len"]) for lv in c.levels],
        num_qo_heads=c.num_qo_heads, num_kv_heads=c.num_kv_heads, head_dim=c.head_dim,
        page_size=c.page_size, layout=c.layout, mask_mode=c.mask_mode, split_mode=split[0],
        fixed_split_pages=split[1], kv_dtype="e4m3", k_scale=0.5, v_scale=2.0)
    o, lse = attn.run(bf16(c.q), kv_tensor(c.k_pool), kv_tensor(c.v_pool), i32(c.kv_indices))
    torch.cuda.synchronize()
    assert pka.pka_get_device_error() == 0
    if info.num_prefill_items > 0:
        assert info.kv_scratch_rows > 0
    o_ref, lse_ref = ref.cascade_attention(c.q, c.k_pool, c.v_pool, levels=c.levels,
                                           page_size=c.page_size, num_qo_heads=c.num_qo_heads,
                                           num_kv_heads=c.num_kv_heads, layout=c.layout,
                                           mask_mode=c.mask_mode, kv_dtype="e4m3", k_scale=0.5,
                                           v_scale=2.0)
    assert_parity(f64(o), f64(lse), o_ref, lse_ref)


def test_cascade_full_size_sampled_rows():
    """The benchmark's cascade at full size (64 decode rows under a 32,768-token
    shared prompt, own suffixes U[512, 2048], page 16, 32/8 heads, D 128) in
    the plan the benchmark times: every root-level piece (the tensor-core
    items, split over the CTAs) feeds every row, so the sampled rows check all
    of them through the merge, together with the own-level decode items of
    those rows."""
    c = W.shared_prompt_decode()
    attn = pka.BatchAttention()
    info = attn.plan_cascade(
        [(lv["qo_indptr"], lv["kv_indptr"], lv["last_page_len"]) for lv in c.levels],
        num_qo_heads=32, num_kv_heads=8, head_dim=128, page_size=16)
    assert info.num_prefill_items > 1 and info.num_decode_items > 0
    o, lse = attn.run(bf16(c.q), bf16(c.k_pool), bf16(c.v_pool), i32(c.kv_indices))
    torch.cuda.synchronize()
    assert pka.pka_get_device_error() == 0
    rng = np.random.default_rng(5)
    rows = {0, c.nnz_q - 1} | {int(r) for r in rng.choice(c.nnz_q, 14, replace=False)}
    o_ref, lse_ref = ref.cascade_attention(c.q, c.k_pool, c.v_pool, levels=c.levels,
                                           page_size=16, num_qo_heads=32, num_kv_heads=8,
                                           rows=rows)
    assert_parity(f64(o), f64(lse), o_ref, lse_ref, rows=rows)
