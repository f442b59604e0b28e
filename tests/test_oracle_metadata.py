"""Pins of the oracle's metadata helpers against values the pages print.

* "Deep Dive - FlashInfer", section "Why inference attention becomes
  irregular": the three-request batch (qo_indptr [0,3,4,8], kv_indptr
  [0,2,3,6], kv_len [6,2,9]) and the four rejected page lists/tails.
* "GPU attention backends: FlashInfer and FlashAttention", section "What it
  prints": the page-size-1 view and the page-number table of the same two
  requests.
* "KV-Cache layouts", section "Mask layout (2D Ragged Tensor)": mask_indptr.
"""
import json
import os

import numpy as np
import pytest

from oracle import ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_worked_example_pointer_arrays_and_lengths():
    g = _load("worked_example_metadata.json")
    pages, tails, P = g["pages"], g["last_page_len"], g["page_size"]
    assert ref.indptr_from_lengths(g["qo_lens"]) == g["printed"]["qo_indptr"]
    assert ref.indptr_from_lengths([len(p) for p in pages]) == g["printed"]["kv_indptr"]
    assert [ref.kv_len_from_pages(p, t, P) for p, t in zip(pages, tails)] == g["printed"]["kv_len"]
    lens = ref.kv_lens_from_csr(g["printed"]["kv_indptr"], g["kv_indices"], tails, P)
    assert lens == g["printed"]["kv_len"]


@pytest.mark.parametrize("case", range(4))
def test_worked_example_rejections(case):
    g = _load("worked_example_metadata.json")
    pages, tail = g["rejected_page_lists_and_tails"][case]
    with pytest.raises(ValueError):
        ref.kv_len_from_pages(pages, tail, g["page_size"])


def test_length_contract_bounds_of_tail():
    # last_page_len may be any of 1..P and nothing else
    for t in range(1, 5):
        assert ref.kv_len_from_pages([0, 1], t, 4) == 4 + t
    for t in (0, 5, -1):
        with pytest.raises(ValueError):
            ref.kv_len_from_pages([0, 1], t, 4)


def _minisgl_rows():
    g = _load("minisgl_metadata_example.json")
    rows = {}
    for r, (a, b) in g["setup"]["token_rows"].items():
        rows[int(r)] = list(range(a, b + 1))
    return g, rows


def test_page_size_1_view_of_token_pool():
    g, rows = _minisgl_rows()
    dev = g["setup"]["prompt_lens"]
    cached = g["setup"]["cached_lens"]
    want = g["printed_page_size_1"]
    assert ref.indptr_from_lengths([d - c for d, c in zip(dev, cached)]) == want["qo_indptr"]
    assert ref.indptr_from_lengths(dev) == want["kv_indptr"]
    indices = [x for r in (0, 1) for x in rows[r][:dev[r]]]
    assert indices == want["kv_indices"]
    # with one token per page every page is full
    assert ref.kv_lens_from_csr(want["kv_indptr"], indices, want["last_page_len"], 1) == dev


def test_page_number_table_and_csr_conversion():
    g, rows = _minisgl_rows()
    P = g["setup"]["fa_page_size"]
    dev = g["setup"]["prompt_lens"]
    want = g["printed_page_size_4"]
    max_len = max(dev)
    table = [ref.token_locations_to_page_numbers(rows[r], max_len, P) for r in (0, 1)]
    assert table == want["page_table"]
    assert dev == want["cache_seqlens"]
    indptr, indices, last = ref.page_table_to_csr(table, dev, P)
    assert indptr == [0, 2, 4]
    assert indices == [4, 5, 10, 11]
    assert last == [1, 2]
    assert ref.kv_lens_from_csr(indptr, indices, last, P) == dev


def test_mask_indptr_matches_prefix_of_products():
    qo, kv = [3, 1, 4], [6, 2, 9]
    assert ref.mask_indptr(qo, kv) == [0, 18, 20, 56]
    lens = np.array([5, 0, 7])
    assert ref.mask_indptr(lens, lens) == [0, 25, 25, 74]
