"""Host-side tests of the C ABI: no GPU needed.

The library loads and exports every entry point include/pka.h declares; the
validator returns the documented status for each contract violation ("Deep
Dive - FlashInfer", "Why inference attention becomes irregular": empty page
list, tail outside 1..P; "KV-Cache layouts": int32 metadata); the planner's
work list covers every (request, head block, query tile, key) exactly once,
is deterministic, and reports workspace sizes.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import paged_kv_attention_plan_gb300 as pka
from paged_kv_attention_plan_gb300 import _pka
from inputs import workloads as W
from tests.plan_image import parse

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, METADATA, UNSUPPORTED, WORKSPACE, STALE = 0, 1, 2, 3, 4, 5


def _i32(x):
    return np.asarray(x, dtype=np.int32)


def test_library_exports_every_declared_symbol():
    header = open(os.path.join(ROOT, "include", "pka.h")).read()
    declared = sorted(set(re.findall(r"\b(pka_[a-z_]+)\s*\(", header)))
    assert declared, "no declarations found"
    lib = _pka.lib()
    missing = [name for name in declared if not hasattr(lib, name)]
    assert not missing, missing
    assert set(declared) == set(_pka.EXPORTED)


def test_version_and_status_strings():
    assert pka.pka_version() == (1, 0)
    for code in range(8):
        assert pka.pka_status_str(code)


def _p(**kw):
    base = dict(num_qo_heads=4, num_kv_heads=2, head_dim=64, page_size=4, num_sms=152)
    base.update(kw)
    return pka.make_params(**base)


WORKED = (_i32([0, 3, 4, 8]), _i32([0, 2, 3, 6]), _i32([2, 2, 1]))


def test_validate_worked_example():
    assert pka.pka_validate(_p(), *WORKED) == OK


@pytest.mark.parametrize("qo,kv,last,params,want", [
    ([0, 3, 4, 8], [1, 2, 3, 6], [2, 2, 1], {}, METADATA),       # kv_indptr[0] != 0
    ([1, 3, 4, 8], [0, 2, 3, 6], [2, 2, 1], {}, METADATA),       # qo_indptr[0] != 0
    ([0, 3, 4, 8], [0, 2, 1, 6], [2, 2, 1], {}, METADATA),       # decreasing kv_indptr
    ([0, 3, 2, 8], [0, 2, 3, 6], [2, 2, 1], {}, METADATA),       # decreasing qo_indptr
    ([0, 3, 4, 8], [0, 2, 2, 6], [2, 2, 1], {}, METADATA),       # request without a page
    ([0, 3, 4, 8], [0, 2, 3, 6], [2, 0, 1], {}, METADATA),       # tail 0
    ([0, 3, 4, 8], [0, 2, 3, 6], [2, 5, 1], {}, METADATA),       # tail P + 1
    ([0, 3, 6, 8], [0, 2, 3, 6], [2, 2, 1], {}, METADATA),       # causal with K=2 < Q=3
    ([0, 3, 6, 8], [0, 2, 3, 6], [2, 2, 1], {"mask_mode": "none"}, OK),
    ([0, 3, 4, 8], [0, 2, 3, 6], [2, 2, 1], {"num_qo_heads": 5}, UNSUPPORTED),
    ([0, 3, 4, 8], [0, 2, 3, 6], [2, 2, 1], {"num_qo_heads": 6}, UNSUPPORTED),  # g = 3
    ([0, 3, 4, 8], [0, 2, 3, 6], [2, 2, 1], {"head_dim": 96}, UNSUPPORTED),
    ([0, 3, 4, 8], [0, 2, 3, 6], [2, 2, 1], {"layout": 7}, INVALID),
    ([0, 3, 4, 8], [0, 2, 3, 6], [2, 2, 1], {"split_mode": "fixed", "fixed_split_pages": 0},
     INVALID),
])
def test_validate_rejections(qo, kv, last, params, want):
    assert pka.pka_validate(_p(**params), _i32(qo), _i32(kv), _i32(last)) == want


def test_reserved_fields_must_be_zero():
    p = _p()
    p.reserved[0] = 1
    assert pka.pka_validate(p, *WORKED) == INVALID
    p = _p()
    p.decode_on_tensor_cores = 2
    assert pka.pka_validate(p, *WORKED) == INVALID


def test_int64_metadata_rejected_by_binding():
    with pytest.raises(TypeError):
        pka.pka_validate(_p(), np.array([0, 3, 4, 8]), WORKED[1], WORKED[2])


def _dry_plan(params, qo, kv, last):
    h = pka.pka_plan_create()
    try:
        buf = np.zeros(64, np.uint8)
        s = pka.pka_plan(h, params, qo, kv, last, None, buf, check=False)
        info = pka.pka_plan_get_info(h)
        if s == WORKSPACE:
            buf = np.zeros(int(info.int_ws_bytes), np.uint8)
            s = pka.pka_plan(h, params, qo, kv, last, None, buf, check=False)
            info = pka.pka_plan_get_info(h)
        assert s == OK, s
        return parse(buf), info, buf
    finally:
        pka.pka_plan_destroy(h)


def _ranges_tile(ranges, n):
    ranges = sorted(ranges)
    if n == 0:
        return all(a == b == 0 for a, b in ranges)
    pos = 0
    for a, b in ranges:
        if a != pos or b <= a:
            return False
        pos = b
    return pos == n


def check_coverage(plan, b, hq, hk, causal, info, allow_empty_ctas=False):
    g = hq // hk
    qo_len = np.diff(b.qo_indptr)
    kv_len = np.asarray(b.kv_lens)
    hpc = plan["header"]["decode_heads_per_cta"]
    # every CTA has at least one item (graph mode: at most zero) and the item
    # lists tile the item array
    for key in ("decode", "prefill"):
        ptr = plan[f"{key}_cta_ptr"]
        assert ptr[0] == 0 and ptr[-1] == len(plan[f"{key}_items"])
        if allow_empty_ctas:
            assert all(x <= y for x, y in zip(ptr[:-1], ptr[1:]))
        else:
            assert all(x < y for x, y in zip(ptr[:-1], ptr[1:]))
    units = {}
    for it in plan["decode_items"]:
        assert qo_len[it["req"]] == 1 and it["q_count"] == 1 and it["n_kv_heads"] == hpc
        units.setdefault((it["req"], it["kv_head0"]), []).append(it)
    for r in np.nonzero(qo_len == 1)[0]:
        for h0 in range(0, hk, hpc):
            its = units.pop((int(r), h0))
            assert _ranges_tile([(i["t0"], i["t1"]) for i in its], int(kv_len[r]))
            assert all(i["q_row0"] == b.qo_indptr[r] for i in its)
    assert not units
    tq = 256 // g  # two 128-row tiles of packed (token, head) rows per item
    for it in plan["prefill_items"]:
        assert qo_len[it["req"]] >= 2 and it["n_kv_heads"] == 1
        units.setdefault((it["req"], it["kv_head0"], it["q_local0"]), []).append(it)
    for r in np.nonzero(qo_len >= 2)[0]:
        Q, K = int(qo_len[r]), int(kv_len[r])
        for h in range(hk):
            for q0 in range(0, Q, tq):
                its = units.pop((int(r), h, q0))
                qc = min(tq, Q - q0)
                kend = K - Q + q0 + qc if causal else K
                assert all(i["q_count"] == qc for i in its)
                assert _ranges_tile([(i["t0"], i["t1"]) for i in its], kend)
    assert not units
    # partial records: disjoint, inside the float workspace, merged exactly once
    recs = set()
    for key, heads in (("decode_items", hpc * g), ("prefill_items", g)):
        for it in plan[key]:
            if it["out_rec"] >= 0:
                span = range(it["out_rec"], it["out_rec"] + it["q_count"] * heads)
                assert not recs.intersection(span)
                recs.update(span)
    assert recs == set(range(info.num_partial_records))
    merged = set()
    for m in plan["merges"]:
        for k in range(m["nslots"]):
            rec = m["rec_first"] + k * m["rec_stride"]
            assert rec not in merged
            merged.add(rec)
        assert m["nslots"] >= 2
    # split decode units: merged in the decode kernel through their joins
    joins = plan["joins"]
    for j in joins:
        assert j["arrived"] == 0 and j["nslots"] >= 2
        for k in range(j["nslots"]):
            for h in range(g):
                rec = j["rec_first"] + k * j["rec_stride"] + h
                assert rec not in merged
                merged.add(rec)
    for it in plan["decode_items"]:
        assert (it["join"] >= 0) == (it["out_rec"] >= 0)
        if it["join"] >= 0:
            for hl in range(hpc):
                j = joins[it["join"] + hl]
                k, r = divmod(it["out_rec"] + hl * g - j["rec_first"], j["rec_stride"])
                assert r == 0 and 0 <= k < j["nslots"]
    for it in plan["prefill_items"]:
        assert it["join"] == -1
    assert merged == recs
    assert info.num_decode_joins == len(joins)
    assert info.float_ws_bytes >= info.num_partial_records * (b.head_dim + 1) * 4


CONFIGS = {
    "worked": lambda: W.worked_example(),
    "decode": lambda: W.batch_decode(with_payload=False),
    "prefill": lambda: W.append_prefill(with_payload=False),
    "mixed_p1": lambda: W.mixed_step(page_size=1, with_payload=False),
    "mixed_p16_hnd": lambda: W.mixed_step(page_size=16, layout="HND", with_payload=False),
    "ragged": lambda: W.ragged_custom_mask(with_payload=False),
}


def _small_mixed(seed, layout="NHD", page_size=4, ragged=False):
    rng = np.random.default_rng(seed)
    n = 9
    qo = rng.integers(0, 40, size=n)
    qo[::3] = 1
    kv = qo + rng.integers(0, 300, size=n)
    if ragged:
        b = W.make_ragged_batch(seed, kv, hq=8, hk=2, d=64, mask_mode="custom", with_payload=False)
        return b
    return W.make_paged_batch(seed, qo, kv, page_size=page_size, layout=layout, hq=8, hk=2, d=64,
                              with_payload=False)


SMALL = {
    "worked": lambda: W.worked_example(),
    "small_p4": lambda: _small_mixed(1),
    "small_p1_hnd": lambda: _small_mixed(2, "HND", 1),
    "small_p16": lambda: _small_mixed(3, "NHD", 16),
    "small_ragged": lambda: _small_mixed(4, ragged=True),
}


def _check_cfg(b, split):
    params = pka.make_params(b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.layout,
                             b.mask_mode, kv_ragged=b.kv_ragged, split_mode=split[0],
                             fixed_split_pages=split[1], num_sms=152)
    qo = None if b.is_decode else b.qo_indptr
    plan, info, _ = _dry_plan(params, qo, b.kv_indptr, b.last_page_len)
    check_coverage(plan, b, b.num_qo_heads, b.num_kv_heads, b.mask_mode == "causal", info)
    assert info.nnz_qo == b.nnz_q and info.total_kv == int(np.sum(b.kv_lens))


@pytest.mark.parametrize("split", [("off", 1), ("auto", 1), ("fixed", 1), ("fixed", 2),
                                   ("fixed", 7)])
@pytest.mark.parametrize("cfg", list(SMALL))
def test_plan_covers_every_key_once_small(cfg, split):
    _check_cfg(SMALL[cfg](), split)


@pytest.mark.parametrize("split", [("off", 1), ("auto", 1), ("fixed", 64)])
@pytest.mark.parametrize("cfg", list(CONFIGS))
def test_plan_covers_every_key_once_full_size(cfg, split):
    if cfg == "ragged" and split[0] == "fixed":
        split = ("fixed", 2048)  # ragged chunks count tokens
    _check_cfg(CONFIGS[cfg](), split)


def test_auto_split_balances_decode_keys():
    b = W.batch_decode(with_payload=False)
    params = pka.make_params(32, 8, 128, 16, num_sms=152)
    plan, info, _ = _dry_plan(params, None, b.kv_indptr, b.last_page_len)
    loads = []
    ptr = plan["decode_cta_ptr"]
    for c in range(len(ptr) - 1):
        loads.append(sum(i["t1"] - i["t0"] for i in plan["decode_items"][ptr[c]:ptr[c + 1]]))
    assert len(loads) <= 153
    assert max(loads) <= info.decode_chunk_tokens
    assert sum(loads) == int(np.sum(b.kv_lens))


@pytest.mark.parametrize("cfg", ["prefill", "ragged"])
def test_prefill_deal_is_list_scheduling(cfg):
    """Tensor-core items are dealt longest first, each to the least loaded CTA
    (cost = keys + 64): every CTA's load then stays within the mean load plus
    the largest item, and the per-CTA loads are as even as that greedy rule
    makes them (no CTA is idle while another holds two or more items)."""
    b = CONFIGS[cfg]()
    params = pka.make_params(b.num_qo_heads, b.num_kv_heads, b.head_dim, b.page_size, b.layout,
                             b.mask_mode, kv_ragged=b.kv_ragged, num_sms=152)
    plan, _, _ = _dry_plan(params, b.qo_indptr, b.kv_indptr, b.last_page_len)
    ptr, items = plan["prefill_cta_ptr"], plan["prefill_items"]
    cost = [i["t1"] - i["t0"] + 64 for i in items]
    loads = [sum(cost[ptr[c]:ptr[c + 1]]) for c in range(len(ptr) - 1)]
    assert len(loads) == min(152, len(items))
    assert min(ptr[c + 1] - ptr[c] for c in range(len(ptr) - 1)) >= 1
    assert max(loads) <= sum(loads) / len(loads) + max(cost)
    # inside a CTA the items come in dealing order: longest first
    for c in range(len(ptr) - 1):
        cs = cost[ptr[c]:ptr[c + 1]]
        assert cs == sorted(cs, reverse=True)


def test_plan_is_deterministic():
    b = W.mixed_step(page_size=16, layout="HND", with_payload=False)
    params = pka.make_params(32, 8, 128, 16, "HND", num_sms=152)
    _, _, a = _dry_plan(params, b.qo_indptr, b.kv_indptr, b.last_page_len)
    _, _, c = _dry_plan(params, b.qo_indptr, b.kv_indptr, b.last_page_len)
    assert np.array_equal(a, c)


def test_replanning_one_handle_matches_fresh_handles():
    """A plan object reuses its planner lists from plan to plan: a sequence of
    different batches and cascades planned on one handle gives, byte for byte,
    the images that a fresh handle gives for each."""
    c = W.make_cascade_batch(31, [1, 1, 5, 1, 40], [300, 17, 900, 64, 1200],
                             [[(5, 2000)], [(2, 160), (3, 0)]], page_size=4, with_payload=False)
    levels = [(lv["qo_indptr"], lv["kv_indptr"], lv["last_page_len"]) for lv in c.levels]
    dec = W.batch_decode(with_payload=False)
    mix = W.mixed_step(page_size=16, layout="HND", with_payload=False)
    runs = [
        ("cascade", pka.make_params(32, 8, 128, 4, num_sms=152), levels),
        ("plan", pka.make_params(32, 8, 128, 16, num_sms=152),
         (None, dec.kv_indptr, dec.last_page_len)),
        ("plan", pka.make_params(32, 8, 128, 16, "HND", split_mode="fixed", fixed_split_pages=5,
                                 num_sms=152), (mix.qo_indptr, mix.kv_indptr, mix.last_page_len)),
        ("cascade", pka.make_params(32, 8, 128, 4, mask_mode="none", split_mode="off",
                                    num_sms=152), levels),
        ("plan", pka.make_params(32, 8, 128, 16, "HND", num_sms=152, graph_max_batch=200,
                                 graph_max_qo_rows=4096),
         (mix.qo_indptr, mix.kv_indptr, mix.last_page_len)),
    ]

    def image(h, kind, params, args):
        buf = np.zeros(1 << 24, np.uint8)
        if kind == "cascade":
            s = pka.pka_plan_cascade(h, params, args, None, buf, check=False)
        else:
            s = pka.pka_plan(h, params, *args, None, buf, check=False)
        assert s == 0
        return buf[:int(pka.pka_plan_get_info(h).int_ws_bytes)].copy()

    fresh = []
    for r in runs:
        h = pka.pka_plan_create()
        try:
            fresh.append(image(h, *r))
        finally:
            pka.pka_plan_destroy(h)
    h = pka.pka_plan_create()
    try:
        for r, want in zip(runs + runs[::-1], fresh + fresh[::-1]):
            assert np.array_equal(image(h, *r), want)
    finally:
        pka.pka_plan_destroy(h)


def test_workspace_too_small_reports_sizes():
    h = pka.pka_plan_create()
    try:
        s = pka.pka_plan(h, _p(), *WORKED, None, np.zeros(16, np.uint8), check=False)
        assert s == WORKSPACE
        info = pka.pka_plan_get_info(h)
        assert info.int_ws_bytes > 16
    finally:
        pka.pka_plan_destroy(h)


def test_stale_plan_detected_before_any_cuda_call():
    h = pka.pka_plan_create()
    try:
        buf = np.zeros(1 << 16, np.uint8)
        pka.pka_plan(h, _p(), *WORKED, None, buf)
        lib = _pka.lib()
        other = _p(page_size=8)
        import ctypes
        s = lib.pka_run(h, ctypes.byref(other), 16, 16, 16, 64, 16, None, 16, None, None, 0, None)
        assert s == STALE
        same = _p()
        s = lib.pka_run(h, ctypes.byref(same), 16, 16, 16, 64, 16, None, 16, None, None, 0, None)
        assert s == INVALID  # a dry-run plan has no device work list
    finally:
        pka.pka_plan_destroy(h)


def test_null_arguments_rejected():
    lib = _pka.lib()
    assert lib.pka_plan_create(None) == INVALID
    assert lib.pka_packbits(None, 5, None, None) == INVALID
    assert lib.pka_packbits(None, 0, None, None) == OK
    assert lib.pka_merge_states(None, None, None, 3, 2, 64, None, None, None) == INVALID
    assert lib.pka_merge_states(None, None, None, 3, 2, 96, None, None, None) == UNSUPPORTED
    p = _p()
    import ctypes
    assert lib.pka_append_paged_kv_cache(ctypes.byref(p), 3, None, None, None, 5, None, None,
                                         None, None, None, 64, None) == INVALID


def test_append_rejects_misaligned_buffers_and_strides():
    """pka_append_paged_kv_cache moves 16-byte row pieces: buffers that are not
    16-byte aligned, or a page stride that is not whole 16-byte units, are
    refused before any device work (the pointers below are never read)."""
    import ctypes
    lib = _pka.lib()
    A = 1 << 20  # a 16-byte-aligned stand-in address

    def call(params, k_new=A, v_new=A, k=A, v=A, stride=1024, nnz=5):
        return lib.pka_append_paged_kv_cache(ctypes.byref(params), 3, k_new, v_new, A, nnz, A, A,
                                             A, k, v, stride, None)

    bf = _p()
    for bad in (dict(k_new=A + 8), dict(v_new=A + 2), dict(k=A + 4), dict(v=A + 1),
                dict(stride=1024 + 4), dict(stride=0), dict(stride=-16)):
        assert call(bf, **bad) == INVALID, bad
    f8 = _p(kv_dtype="e4m3")
    assert call(f8, stride=1024 + 8) == INVALID  # e4m3 rows: 16 elements per 16 bytes
    assert call(_p(kv_ragged=True)) == UNSUPPORTED
    assert call(bf, nnz=0) == OK  # nothing to append: no device work


def test_fp8_kv_tensor_core_rows_plan_a_bf16_scratch():
    """e4m3 K/V: rows with qo_len >= 2 are planned over a bf16 scratch of their
    requests' keys (dequant units in the image, items reading scratch rows);
    graph mode needs graph_max_kv_tokens for them and then keeps one layout
    (scratch laid out for the capacity), decode-only batches need no scratch."""
    b = W.make_paged_batch(3, [1, 5, 1, 3], [10, 20, 30, 7], page_size=4, hq=8, hk=2, d=64,
                           with_payload=False)
    p = pka.make_params(8, 2, 64, 4, kv_dtype="e4m3", num_sms=152)
    assert pka.pka_validate(p, b.qo_indptr, b.kv_indptr, b.last_page_len) == OK
    h = pka.pka_plan_create()
    buf = np.zeros(1 << 20, np.uint8)
    assert pka.pka_plan(h, p, b.qo_indptr, b.kv_indptr, b.last_page_len, None, buf,
                        check=False) == OK
    info = pka.pka_plan_get_info(h)
    assert info.kv_scratch_rows == 20 + 7  # the two requests with qo_len >= 2
    scratch = 2 * ((27 * 2 * 64 * 2 + 255) // 256 * 256)
    assert info.float_ws_bytes >= scratch
    img = parse(buf[: info.int_ws_bytes])
    assert img["header"]["dequant_rows"] == 27
    units = img["dequant_units"]
    assert [u["kv_base"] for u in units] == [int(b.kv_indptr[1]), int(b.kv_indptr[3])]
    assert [u["kv_len"] for u in units] == [20, 7] and [u["dst_row0"] for u in units] == [0, 20]
    for it in img["prefill_items"]:
        assert it["kv_base"] == (0 if it["req"] == 1 else 20)
    for it in img["decode_items"]:
        assert it["kv_base"] == int(b.kv_indptr[it["req"]])
    assert pka.pka_plan(h, p, None, b.kv_indptr, b.last_page_len, None, buf, check=False) == 0
    assert pka.pka_plan_get_info(h).kv_scratch_rows == 0
    g = pka.make_params(8, 2, 64, 4, kv_dtype="e4m3", graph_max_batch=8, graph_max_qo_rows=64)
    assert pka.pka_plan(h, g, b.qo_indptr, b.kv_indptr, b.last_page_len, None, buf,
                        check=False) == UNSUPPORTED  # no scratch capacity declared
    # graph mode with a declared capacity: one fixed layout, scratch laid out for it
    g = pka.make_params(8, 2, 64, 4, kv_dtype="e4m3", graph_max_batch=8, graph_max_qo_rows=64,
                        graph_max_kv_tokens=100, num_sms=152)
    layouts = []
    for qo, kv in (([1, 5, 1, 3], [10, 20, 30, 7]), ([2, 1], [60, 9]), ([1, 1, 1], [4, 5, 6])):
        c = W.make_paged_batch(4, qo, kv, page_size=4, hq=8, hk=2, d=64, with_payload=False)
        buf[:] = 0
        assert pka.pka_plan(h, g, c.qo_indptr, c.kv_indptr, c.last_page_len, None, buf,
                            check=False) == OK
        gi = pka.pka_plan_get_info(h)
        hdr = parse(buf[: gi.int_ws_bytes])["header"]
        tc = [k for q, k in zip(qo, kv) if q >= 2]
        assert hdr["dequant_rows"] == sum(tc) and hdr["num_dequant_units"] == len(tc)
        layouts.append((gi.int_ws_bytes, gi.float_ws_bytes, hdr["off_dequant_units"]))
    assert len(set(layouts)) == 1 and layouts[0][2] > 0
    assert layouts[0][1] >= 2 * ((100 * 2 * 64 * 2 + 255) // 256 * 256)
    c = W.make_paged_batch(5, [3, 2], [70, 40], page_size=4, hq=8, hk=2, d=64,
                           with_payload=False)
    assert pka.pka_plan(h, g, c.qo_indptr, c.kv_indptr, c.last_page_len, None, buf,
                        check=False) == WORKSPACE  # 110 keys > the 100-row scratch
    pka.pka_plan_destroy(h)
    bad = pka.make_params(8, 2, 64, 4)
    bad.kv_dtype = 7
    assert pka.pka_plan(pka.pka_plan_create(), bad, None, b.kv_indptr, b.last_page_len, None,
                        buf, check=False) == INVALID


@pytest.mark.parametrize("cfg", ["worked", "decode", "mixed_p16_hnd"])
def test_decode_rows_on_tensor_cores_plan(cfg):
    """With decode_on_tensor_cores, rows with qo_len == 1 become tensor-core
    items (one query token, the g heads of each kv head packed into the tile)
    whose key ranges tile [0, kv_len) per (request, kv head); the decode list
    is empty.  Graph mode keeps one layout with the option; over e4m3 pools the
    rows read the bf16 scratch (in graph mode within graph_max_kv_tokens)."""
    b = CONFIGS[cfg]()
    hq, hk = b.num_qo_heads, b.num_kv_heads
    params = pka.make_params(hq, hk, b.head_dim, b.page_size, b.layout, b.mask_mode,
                             num_sms=152, decode_on_tensor_cores=True)
    h = pka.pka_plan_create()
    buf = np.zeros(1 << 24, np.uint8)
    qo = None if b.is_decode else b.qo_indptr
    assert pka.pka_plan(h, params, qo, b.kv_indptr, b.last_page_len, None, buf, check=False) == OK
    info = pka.pka_plan_get_info(h)
    pka.pka_plan_destroy(h)
    plan = parse(buf)
    assert info.num_decode_items == 0 and not plan["decode_items"]
    qo_len = np.diff(b.qo_indptr)
    units = {}
    for it in plan["prefill_items"]:
        units.setdefault((it["req"], it["kv_head0"], it["q_local0"]), []).append(it)
    for r in np.nonzero(qo_len == 1)[0]:
        for kh in range(hk):
            its = units[(int(r), kh, 0)]
            assert all(i["q_count"] == 1 for i in its)
            assert _ranges_tile([(i["t0"], i["t1"]) for i in its], int(b.kv_lens[r]))
    g = pka.make_params(hq, hk, b.head_dim, b.page_size, b.layout, b.mask_mode,
                        decode_on_tensor_cores=True, graph_max_batch=len(b.kv_lens),
                        graph_max_qo_rows=int(b.nnz_q), num_sms=152)
    assert pka.pka_validate(g, b.qo_indptr, b.kv_indptr, b.last_page_len) == OK
    h = pka.pka_plan_create()
    assert pka.pka_plan(h, g, qo, b.kv_indptr, b.last_page_len, None, buf, check=False) == OK
    assert pka.pka_plan_get_info(h).num_decode_items == 0
    # e4m3: every row (decode rows too) reads the bf16 scratch of its request
    f = pka.make_params(hq, hk, b.head_dim, b.page_size, b.layout, b.mask_mode,
                        decode_on_tensor_cores=True, kv_dtype="e4m3", num_sms=152)
    assert pka.pka_plan(h, f, qo, b.kv_indptr, b.last_page_len, None, buf, check=False) == OK
    assert pka.pka_plan_get_info(h).kv_scratch_rows == int(np.sum(b.kv_lens))
    fg = pka.make_params(hq, hk, b.head_dim, b.page_size, b.layout, b.mask_mode,
                         decode_on_tensor_cores=True, kv_dtype="e4m3",
                         graph_max_batch=len(b.kv_lens), graph_max_qo_rows=int(b.nnz_q))
    assert pka.pka_validate(fg, b.qo_indptr, b.kv_indptr, b.last_page_len) == UNSUPPORTED
    fg.graph_max_kv_tokens = int(np.sum(b.kv_lens))
    assert pka.pka_plan(h, fg, qo, b.kv_indptr, b.last_page_len, None, buf, check=False) == OK
    pka.pka_plan_destroy(h)


@pytest.mark.parametrize("qo,kv,last", [([0], [0], []), ([0, 0, 0], [0, 2, 3], [3, 1])])
def test_empty_batches_plan_to_nothing(qo, kv, last):
    """An empty batch, and a batch whose requests append no rows, plan to no
    work and no workspace."""
    h = pka.pka_plan_create()
    buf = np.zeros(1 << 16, np.uint8)
    assert pka.pka_plan(h, _p(), _i32(qo), _i32(kv), _i32(last), None, buf, check=False) == OK
    info = pka.pka_plan_get_info(h)
    pka.pka_plan_destroy(h)
    assert info.nnz_qo == 0 and info.num_decode_items == 0 and info.num_prefill_items == 0
    assert info.float_ws_bytes == 0 and info.num_merge_tasks == 0


@pytest.mark.parametrize("arrive,polls", [(2, 10), (-1, 10), (0, 0), (1, 1001), (0, -5)])
def test_wait_selftest_rejects_bad_arguments(arrive, polls):
    """Checked before any launch, so no GPU is needed."""
    assert _pka.lib().pka_selftest_bounded_wait(arrive, polls, None) == INVALID


# ---------------------------------------------------------------------------
# pka_check_indices: page ids against the pool, appended slots against other
# requests ("Deep Dive - FlashInfer", "Where FlashInfer sits in a serving
# stack": reused pages and page tables that disagree with last_page_len)
# ---------------------------------------------------------------------------

def _check(kv, idx, last, pool, app=None, P=4):
    return pka.pka_check_indices(_p(page_size=P), _i32(kv), _i32(idx), _i32(last), pool,
                                 None if app is None else _i32(app))


def test_check_indices_accepts_the_worked_batch():
    # printed page ids [7, 2], [11], [3, 14, 6] in a 15-page pool, appends 3/1/4
    assert _check([0, 2, 3, 6], [7, 2, 11, 3, 14, 6], [2, 2, 1], 15) == (OK, -1)
    assert _check([0, 2, 3, 6], [7, 2, 11, 3, 14, 6], [2, 2, 1], 15, app=[0, 3, 4, 8]) == (OK, -1)


@pytest.mark.parametrize("bad_at,value", [(0, -1), (4, 15), (5, 1 << 30)])
def test_check_indices_rejects_ids_outside_the_pool(bad_at, value):
    idx = [7, 2, 11, 3, 14, 6]
    idx[bad_at] = value
    assert _check([0, 2, 3, 6], idx, [2, 2, 1], 15) == (METADATA, bad_at)


def test_check_indices_rejects_two_requests_appending_one_slot():
    # both requests end in page 5; request 0 appends slots 1..2 of it (kv 7, last 3),
    # request 1 appends slot 2 of it (kv 3 in one page, appends 1: position 2)
    s, bad = _check([0, 2, 3], [4, 5, 5], [3, 3], 8, app=[0, 2, 3])
    assert s == METADATA and bad == 2


def test_check_indices_rejects_appending_into_another_requests_history():
    # request 1 reads page 5 slots 0..2 as history; request 0 appends slot 1 of page 5
    s, bad = _check([0, 2, 3], [4, 5, 5], [2, 4], 8, app=[0, 1, 2])
    assert s == METADATA and bad == 2


def test_check_indices_allows_a_shared_read_only_prefix():
    # pages 1, 2 hold a shared prefix read by both requests; each appends into its own page
    assert _check([0, 3, 6], [1, 2, 3, 1, 2, 4], [2, 3], 5, app=[0, 2, 5]) == (OK, -1)


def test_check_indices_argument_errors():
    assert _check([0, 2, 3, 6], [7, 2, 11, 3, 14], [2, 2, 1], 15)[0] == INVALID  # short indices
    assert _check([0, 2, 3, 6], [7, 2, 11, 3, 14, 6], [2, 5, 1], 15)[0] == METADATA  # last > P
    assert _check([0, 2, 3, 6], [7, 2, 11, 3, 14, 6], [2, 2, 1], 15,
                  app=[0, 9, 10, 11])[0] == METADATA  # appends beyond kv_len
    assert _check([0], [], [], 0) == (OK, -1)  # empty batch


def test_check_indices_seeded_workloads_are_clean():
    for b in (W.worked_example(), W.append_prefill(with_payload=False),
              W.mixed_step(page_size=16, layout="HND", with_payload=False)):
        s, bad = pka.pka_check_indices(_p(page_size=b.page_size), b.kv_indptr, b.kv_indices,
                                       b.last_page_len, int(b.extra["pool_pages"]),
                                       b.qo_indptr)
        assert (s, bad) == (OK, -1), b.name
