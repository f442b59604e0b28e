"""Cascade planning on the host: no GPU needed ("KV-Cache layouts",
"Multi-level cascade inference data layout").

The plan of a multi-level cascade must give every (level, node, head, query
tile) its whole visible key range exactly once, mark the levels above the
last as fully visible, send every piece's state to a partial record, and give
every (row, head) one merge task listing exactly the records of its row and
head from all levels.
"""
import numpy as np
import pytest

import paged_kv_attention_plan_gb300 as pka
from inputs import workloads as W
from tests.plan_image import parse

OK, INVALID, METADATA, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3, 4


def _levels(c):
    return [(lv["qo_indptr"], lv["kv_indptr"], lv["last_page_len"]) for lv in c.levels]


def _params(c, split="auto", **kw):
    base = dict(num_qo_heads=c.num_qo_heads, num_kv_heads=c.num_kv_heads, head_dim=c.head_dim,
                page_size=c.page_size, layout=c.layout, mask_mode=c.mask_mode,
                split_mode=split, fixed_split_pages=3, num_sms=152)
    base.update(kw)
    return pka.make_params(**base)


def _dry(c, levels=None, **kw):
    h = pka.pka_plan_create()
    try:
        buf = np.zeros(1 << 24, np.uint8)
        s = pka.pka_plan_cascade(h, _params(c, **kw), levels or _levels(c), None, buf,
                                 check=False)
        return s, pka.pka_plan_get_info(h), buf
    finally:
        pka.pka_plan_destroy(h)


def _ranges_tile(ranges, n):
    pos = 0
    for a, b in sorted(ranges):
        if a != pos or b <= a:
            return False
        pos = b
    return pos == n


def check_cascade_plan(c, info, buf):
    plan = parse(buf)
    hq, hk = c.num_qo_heads, c.num_kv_heads
    g = hq // hk
    hpc = plan["header"]["decode_heads_per_cta"]
    last = len(c.levels) - 1
    offs = np.cumsum([0] + [int(lv["kv_indptr"][-1]) for lv in c.levels])
    node_of = {}
    for li, lv in enumerate(c.levels):
        for n in range(len(lv["kv_lens"])):
            if lv["kv_lens"][n] > 0:
                node_of[(int(lv["qo_indptr"][n]), int(offs[li] + lv["kv_indptr"][n]))] = (li, n)
    units, rec_owner = {}, {}
    for kind in ("decode", "prefill"):
        for it in plan[f"{kind}_items"]:
            li, n = node_of[(it["q_row0"] - it["q_local0"], it["kv_base"])]
            lv = c.levels[li]
            assert it["qo_len"] == lv["qo_indptr"][n + 1] - lv["qo_indptr"][n]
            assert it["kv_len"] == lv["kv_lens"][n]
            shared_flag = 1 if (li < last and c.mask_mode != "none") else 0
            assert it["flags"] == shared_flag
            assert it["out_rec"] >= 0  # every cascade piece writes a partial state
            units.setdefault((li, n, kind, it["kv_head0"], it["q_local0"]), []).append(it)
            heads = range(it["kv_head0"] * g, (it["kv_head0"] + it["n_kv_heads"]) * g)
            for i in range(it["q_count"]):
                for k, h in enumerate(heads):
                    rec = it["out_rec"] + i * len(heads) + k
                    assert rec not in rec_owner
                    rec_owner[rec] = (it["q_row0"] + i, h)
    seen = set()
    for li, lv in enumerate(c.levels):
        for n in range(len(lv["kv_lens"])):
            Q = int(lv["qo_indptr"][n + 1] - lv["qo_indptr"][n])
            K = int(lv["kv_lens"][n])
            if K == 0 or Q == 0:
                continue
            if Q == 1:
                keys = [(li, n, "decode", h0, 0) for h0 in range(0, hk, hpc)]
                ends = [K] * len(keys)
            else:
                tq = 256 // g
                keys, ends = [], []
                for h in range(hk):
                    for q0 in range(0, Q, tq):
                        qc = min(tq, Q - q0)
                        keys.append((li, n, "prefill", h, q0))
                        causal = li == last and c.mask_mode == "causal"
                        ends.append(K - Q + q0 + qc if causal else K)
            for key, end in zip(keys, ends):
                assert _ranges_tile([(i["t0"], i["t1"]) for i in units[key]], end), key
                seen.add(key)
    assert seen == set(units)
    assert set(rec_owner) == set(range(info.num_partial_records))
    # one merge task per (row, head), listing exactly that row's records
    want = {}
    for rec, rh in rec_owner.items():
        want.setdefault(rh, set()).add(rec)
    got = {}
    for m in plan["merges"]:
        assert m["rec_stride"] == 0
        key = (m["out_row"], m["head"])
        assert key not in got
        got[key] = set(plan["merge_slots"][m["rec_first"]:m["rec_first"] + m["nslots"]])
        assert len(got[key]) == m["nslots"]
    assert got == want
    assert set(got) == {(r, h) for r in range(c.nnz_q) for h in range(hq)}
    assert info.float_ws_bytes >= info.num_partial_records * (c.head_dim + 1) * 4


CASCADES = {
    "decode_shared_prompt": lambda: W.make_cascade_batch(
        1, [1] * 12, np.arange(1, 13) * 37, [[(12, 5000)]], page_size=16, hq=32, hk=8, d=128,
        with_payload=False),
    "append_three_levels": lambda: W.make_cascade_batch(
        2, [17, 1, 40, 3, 1, 9], [30, 5, 41, 3, 200, 9], [[(6, 700)], [(2, 64), (1, 0), (3, 129)]],
        page_size=4, hq=16, hk=2, d=64, with_payload=False),
    "page1_hnd": lambda: W.make_cascade_batch(
        3, [5, 1, 1, 300], [5, 80, 2, 400], [[(4, 333)]], page_size=1, layout="HND", hq=8, hk=8,
        d=64, with_payload=False),
    "no_mask": lambda: W.make_cascade_batch(
        4, [4, 1, 6], [2, 7, 3], [[(1, 10), (2, 5)]], page_size=8, hq=8, hk=2, d=64,
        mask_mode="none", with_payload=False),
    "single_level": lambda: W.make_cascade_batch(
        5, [3, 1, 4], [6, 2, 9], [], page_size=4, hq=4, hk=2, d=64, with_payload=False),
}


@pytest.mark.parametrize("split", ["off", "auto", "fixed"])
@pytest.mark.parametrize("cfg", list(CASCADES))
def test_cascade_plan_covers_each_level_once(cfg, split):
    c = CASCADES[cfg]()
    s, info, buf = _dry(c, split=split)
    assert s == OK
    check_cascade_plan(c, info, buf)
    assert info.nnz_qo == c.nnz_q
    assert info.total_kv == sum(int(np.sum(lv["kv_lens"])) for lv in c.levels)


def test_cascade_rejections():
    c = CASCADES["append_three_levels"]()
    assert _dry(c, mask_mode="custom")[0] == UNSUPPORTED
    assert _dry(c, graph_max_batch=8, graph_max_qo_rows=100)[0] == UNSUPPORTED
    levels = _levels(c)
    # a level that splits a different number of rows
    bad = [(np.asarray(levels[0][0]) + np.array([0, 1], np.int32), levels[0][1], levels[0][2])]
    assert _dry(c, levels=bad + levels[1:])[0] == METADATA
    # a node without pages is allowed above the last level, not at it
    q, kv, last = levels[-1]
    kv2 = kv.copy()
    kv2[1:] -= kv2[1] - kv2[0]  # node 0 loses its pages
    assert _dry(c, levels=levels[:-1] + [(q, kv2, last)])[0] == METADATA
    assert _dry(c, levels=levels)[0] == OK
    h = pka.pka_plan_create()
    try:
        s = pka.pka_plan_cascade(h, _params(c), [], None, np.zeros(64, np.uint8), check=False)
        assert s == INVALID
    finally:
        pka.pka_plan_destroy(h)


def test_fp8_cascade_dequantizes_each_tensor_core_node_once():
    """e4m3 pools: every node that tensor-core items read gets one dequant unit
    (its page-list start and kv_len), and those items read its scratch rows."""
    c = W.make_cascade_batch(5, [9, 1, 30, 3], [12, 40, 31, 3], [[(4, 257)], [(2, 64), (2, 20)]],
                             page_size=4, hq=8, hk=2, d=64, with_payload=False)
    p = pka.make_params(8, 2, 64, 4, kv_dtype="e4m3", num_sms=152)
    h = pka.pka_plan_create()
    buf = np.zeros(1 << 20, np.uint8)
    levels = [(lv["qo_indptr"], lv["kv_indptr"], lv["last_page_len"]) for lv in c.levels]
    assert pka.pka_plan_cascade(h, p, levels, None, buf, check=False) == 0
    info = pka.pka_plan_get_info(h)
    img = parse(buf[: info.int_ws_bytes])
    units = img["dequant_units"]
    assert len({u["kv_base"] for u in units}) == len(units)  # one unit per node
    assert info.kv_scratch_rows == sum(u["kv_len"] for u in units) > 0
    starts = {u["dst_row0"]: u for u in units}
    for it in img["prefill_items"]:
        assert it["kv_base"] in starts and starts[it["kv_base"]]["kv_len"] == it["kv_len"]
    pka.pka_plan_destroy(h)
