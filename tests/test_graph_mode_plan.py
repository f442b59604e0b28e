"""Graph mode of the planner, on the host: no GPU needed.

"Deep Dive - FlashInfer", "Plan then run": the plan step does the host work
and the copies, so that compatible run calls can be captured in a CUDA graph.
In graph mode the image has one fixed layout for given parameters (sizes,
section offsets, CTA counts), so that a run() captured once reads every later
plan; these tests check that layout is invariant across batches, that the work
list in it still covers every (request, head, query tile, key) exactly once,
and that batches beyond the declared capacities are refused.
"""
import numpy as np
import pytest

import paged_kv_attention_plan_gb300 as pka
from inputs import workloads as W
from tests.plan_image import parse
from tests.test_host_abi import SMALL, check_coverage

OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 3, 4
SMS = 152


def _params(b, split="auto", max_batch=64, max_rows=4096, max_kv=0, num_sms=SMS):
    return pka.make_params(b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.layout,
                           b.mask_mode, kv_ragged=b.kv_ragged, split_mode=split, num_sms=num_sms,
                           graph_max_batch=max_batch, graph_max_qo_rows=max_rows,
                           graph_max_kv_tokens=max_kv if b.kv_ragged else 0)


def _plan(params, b, size=1 << 22):
    h = pka.pka_plan_create()
    try:
        buf = np.zeros(size, np.uint8)
        qo = None if b.is_decode else b.qo_indptr
        s = pka.pka_plan(h, params, qo, b.kv_indptr, b.last_page_len, None, buf, check=False)
        info = pka.pka_plan_get_info(h)
        return s, info, buf
    finally:
        pka.pka_plan_destroy(h)


def _layout(buf):
    hdr = parse(buf)["header"]
    keys = ["total_words", "num_decode_ctas", "num_prefill_ctas", "off_decode_cta_ptr",
            "off_decode_items", "off_prefill_cta_ptr", "off_prefill_items", "off_merge_tasks",
            "decode_heads_per_cta", "graph_mode"]
    return {k: hdr[k] for k in keys}


@pytest.mark.parametrize("split", ["auto", "off"])
@pytest.mark.parametrize("cfg", list(SMALL))
def test_graph_plan_covers_every_key_once(cfg, split):
    b = SMALL[cfg]()
    s, info, buf = _plan(_params(b, split, max_batch=16, max_rows=4096, max_kv=8192), b)
    assert s == OK
    plan = parse(buf)
    assert plan["header"]["graph_mode"] == 1
    assert plan["header"]["num_decode_ctas"] == SMS and plan["header"]["num_prefill_ctas"] == SMS
    check_coverage(plan, b, b.num_qo_heads, b.num_kv_heads, b.mask_mode == "causal", info,
                   allow_empty_ctas=True)


@pytest.mark.parametrize("cfg", ["decode", "mixed_p16_hnd", "ragged"])
def test_graph_plan_full_size(cfg):
    b = {"decode": lambda: W.batch_decode(with_payload=False),
         "mixed_p16_hnd": lambda: W.mixed_step(page_size=16, layout="HND", with_payload=False),
         "ragged": lambda: W.ragged_custom_mask(with_payload=False)}[cfg]()
    kv = int(np.sum(b.kv_lens))
    s, info, buf = _plan(_params(b, max_batch=len(b.kv_lens), max_rows=b.nnz_q, max_kv=kv), b,
                         size=1 << 24)
    assert s == OK, pka.pka_last_error()
    check_coverage(parse(buf), b, b.num_qo_heads, b.num_kv_heads, b.mask_mode == "causal", info,
                   allow_empty_ctas=True)


def test_layout_and_sizes_do_not_depend_on_the_batch():
    rng = np.random.default_rng(0)
    layouts, sizes = [], []
    for trial in range(12):
        n = int(rng.integers(1, 17))
        qo = rng.integers(1, 90, size=n)
        qo[rng.random(n) < 0.5] = 1
        while qo.sum() > 512:
            qo[np.argmax(qo)] //= 2
        kv = qo + rng.integers(0, 2000, size=n)
        b = W.make_paged_batch(trial, qo, kv, page_size=16, hq=32, hk=8, d=128,
                               with_payload=False)
        s, info, buf = _plan(_params(b, max_batch=16, max_rows=512), b)
        assert s == OK, pka.pka_last_error()
        check_coverage(parse(buf), b, 32, 8, True, info, allow_empty_ctas=True)
        layouts.append(_layout(buf))
        sizes.append((info.int_ws_bytes, info.float_ws_bytes))
    assert all(x == layouts[0] for x in layouts)
    assert len(set(sizes)) == 1


@pytest.mark.parametrize("hq,hk", [(32, 8), (8, 8), (64, 8), (16, 2)])
def test_capacities_hold_for_extreme_length_mixes(hq, hk):
    """Decode splits at their most fragmented: one huge request among many
    one-key requests, every request at the cap, all rows in one request."""
    rng = np.random.default_rng(hq * 100 + hk)
    B, R = 40, 700
    cases = [np.ones(B, np.int64), np.full(B, 1, np.int64)]
    kvs = [np.concatenate([[200000], np.ones(B - 1, np.int64)]),
           rng.integers(1, 40, size=B)]
    cases.append(np.concatenate([[R - (B - 1)], np.ones(B - 1, np.int64)]))
    kvs.append(np.concatenate([[5000], rng.integers(1, 300, size=B - 1)]))
    cases.append(np.full(B, R // B))
    kvs.append(np.full(B, 7000))
    for qo, kv in zip(cases, kvs):
        kv = np.maximum(kv, qo)
        b = W.make_paged_batch(1, qo, kv, page_size=8, hq=hq, hk=hk, d=64, with_payload=False)
        s, info, buf = _plan(_params(b, max_batch=B, max_rows=R), b, size=1 << 24)
        assert s == OK, pka.pka_last_error()
        check_coverage(parse(buf), b, hq, hk, True, info, allow_empty_ctas=True)


def test_over_capacity_batches_are_refused():
    b = _small = SMALL["small_p4"]()
    n, rows = len(b.kv_lens), b.nnz_q
    assert _plan(_params(b, max_batch=n - 1, max_rows=rows), b)[0] == WORKSPACE
    assert "capacit" in pka.pka_last_error()
    assert _plan(_params(b, max_batch=n, max_rows=rows - 1), b)[0] == WORKSPACE
    assert _plan(_params(b, max_batch=n, max_rows=rows), b)[0] == OK
    r = SMALL["small_ragged"]()
    kv = int(np.sum(r.kv_lens))
    assert _plan(_params(r, max_batch=16, max_rows=4096, max_kv=kv - 1), r)[0] == WORKSPACE
    assert _plan(_params(r, max_batch=16, max_rows=4096, max_kv=kv), r)[0] == OK


def test_graph_parameter_rules():
    b = SMALL["small_p4"]()
    assert _plan(_params(b, split="fixed"), b)[0] == UNSUPPORTED
    p = _params(b, max_batch=0, max_rows=64)
    assert pka.pka_validate(p, b.qo_indptr, b.kv_indptr, b.last_page_len) == INVALID
    p = _params(b, max_batch=4, max_rows=0)
    assert pka.pka_validate(p, b.qo_indptr, b.kv_indptr, b.last_page_len) == INVALID
    r = SMALL["small_ragged"]()
    p = _params(r, max_batch=16, max_rows=512, max_kv=0)
    assert pka.pka_validate(p, r.qo_indptr, r.kv_indptr, r.last_page_len) == INVALID


def test_graph_mode_e4m3_ragged_layout_is_fixed():
    """Ragged e4m3 K/V in graph mode: graph_max_kv_tokens bounds both the
    ragged rows and the bf16 scratch of the rows with qo_len >= 2, so the image
    layout and the float workspace stay the same across batches, and each
    plan's dequant units cover exactly its tensor-core requests."""
    params = pka.make_params(16, 4, 64, 1, mask_mode="causal", kv_ragged=True, num_sms=SMS,
                             graph_max_batch=6, graph_max_qo_rows=700, graph_max_kv_tokens=700,
                             kv_dtype="e4m3")
    layouts = []
    for i, lens in enumerate([[300, 1, 200, 100], [1, 1, 1], [700], [64, 65, 1, 190, 2, 3]]):
        b = W.make_ragged_batch(80 + i, lens, hq=16, hk=4, d=64, mask_mode="causal",
                                with_payload=False)
        s, info, buf = _plan(params, b)
        assert s == OK, lens
        img = parse(buf[: info.int_ws_bytes])
        h = img["header"]
        tc = [n for n in lens if n >= 2]
        assert h["num_dequant_units"] == len(tc) and h["dequant_rows"] == sum(tc)
        assert sorted(u["kv_len"] for u in img["dequant_units"]) == sorted(tc)  # in dealing order
        layouts.append((info.int_ws_bytes, info.float_ws_bytes, h["off_dequant_units"],
                        h["off_prefill_items"], h["num_prefill_ctas"]))
    assert len(set(layouts)) == 1
