"""Pins of the oracle's append_paged_kv_cache.

"KV-Cache layouts", section "Page table layout" (the append API writes a
ragged batch of new rows into pages allocated beforehand) and "Deep Dive -
FlashInfer", section "Why inference attention becomes irregular" (reported KV
lengths already include the appended tokens).  Round trip: after the append,
gathering each request's last qo_len logical rows returns the appended rows
bit for bit, and every other slot (including NaN-poisoned ones) is unchanged.
"""
import numpy as np
import pytest

from oracle import ref
from inputs import workloads as W


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_append_round_trip(layout, page_size):
    b = W.make_paged_batch(30 + page_size, [3, 1, 0, 17], [6, 2, 5, 40], page_size=page_size,
                           layout=layout, hq=4, hk=2, d=8, append_new=True)
    before_k, before_v = b.k_pool.copy(), b.v_pool.copy()
    k, v = ref.append_paged_kv_cache(b.k_new, b.v_new, b.qo_indptr, b.k_pool, b.v_pool,
                                     kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                                     last_page_len=b.last_page_len, page_size=page_size,
                                     layout=layout)
    touched = np.zeros(k.shape[:-1], bool)  # per (page, slot, head) or (page, head, slot)
    for r in range(b.batch_size):
        K, Q = int(b.kv_lens[r]), int(b.qo_lens[r])
        rows = ref.gather_request_kv(k, layout=layout, page_size=page_size,
                                     kv_indptr=b.kv_indptr, kv_indices=b.kv_indices, req=r,
                                     kv_len=K)
        q0 = int(b.qo_indptr[r])
        assert np.array_equal(rows[K - Q:], b.k_new[q0:q0 + Q])
        pages = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]]
        for j in range(K - Q, K):
            pg, s = ref.token_address(pages, j, page_size)
            if layout == "NHD":
                touched[pg, s] = True
            else:
                touched[pg, :, s] = True
    assert np.array_equal(k[~touched], before_k[~touched])
    assert np.array_equal(v[~touched], before_v[~touched])
    # inputs are not modified in place
    assert np.array_equal(b.k_pool, before_k)


def test_append_more_rows_than_length_rejected():
    b = W.make_paged_batch(40, [2], [2], page_size=4, hq=2, hk=1, d=8, append_new=True)
    with pytest.raises(ValueError):
        ref.append_paged_kv_cache(np.zeros((3, 1, 8), np.uint16), np.zeros((3, 1, 8), np.uint16),
                                  [0, 3], b.k_pool, b.v_pool, kv_indptr=b.kv_indptr,
                                  kv_indices=b.kv_indices, last_page_len=b.last_page_len,
                                  page_size=4)
