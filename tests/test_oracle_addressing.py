"""Pins of addressing, causal alignment, layouts and mask packing.

* "Deep Dive - FlashInfer", section "Causality uses logical positions, not
  page numbers": R2's token 5 sits in page 14 slot 1, its last token in page 6
  slot 0, and the printed 4x9 visibility picture (row sums 6, 7, 8, 9).
* "KV-Cache layouts", sections "NHD/HND" and "Page table layout" (5-D vs tuple
  storage) and "Mask layout (2D Ragged Tensor)" (little-endian packbits, as
  numpy.packbits with bitorder='little').
"""
import os

import numpy as np
import pytest

from oracle import ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_picture():
    lines = [l.strip() for l in open(os.path.join(GOLDEN, "causal_mask_r2.txt"))
             if l.strip() and not l.startswith("#")]
    tok5 = tuple(int(x) for x in lines[0].split()[1:])
    last = tuple(int(x) for x in lines[1].split()[1:])
    return tok5, last, lines[2:]


def test_r2_addresses():
    tok5, last, _ = _golden_picture()
    pages, P, K = [3, 14, 6], 4, 9
    addrs = [ref.token_address(pages, j, P) for j in range(K)]
    assert addrs[5] == tok5
    assert addrs[-1] == last
    assert [p for p, _ in addrs] != sorted(p for p, _ in addrs)


def test_r2_causal_picture():
    _, _, picture = _golden_picture()
    Q, K = 4, 9
    drawn = ["".join("1" if ref.causal_visible(i, j, Q, K) else "." for j in range(K))
             for i in range(Q)]
    assert drawn == picture
    assert [row.count("1") for row in drawn] == [6, 7, 8, 9]


def test_gather_nhd_equals_hnd_and_5d_view():
    rng = np.random.default_rng(0)
    pool_nhd = rng.integers(0, 2**16, size=(7, 4, 3, 8), dtype=np.uint16)
    pool_hnd = np.ascontiguousarray(pool_nhd.transpose(0, 2, 1, 3))
    indptr, indices = [0, 3], [5, 0, 2]
    a = ref.gather_request_kv(pool_nhd, layout="NHD", page_size=4, kv_indptr=indptr,
                              kv_indices=indices, req=0, kv_len=10)
    b = ref.gather_request_kv(pool_hnd, layout="HND", page_size=4, kv_indptr=indptr,
                              kv_indices=indices, req=0, kv_len=10)
    assert np.array_equal(a, b)
    # rows 0..3 come from page 5, 4..7 from page 0, 8..9 from page 2 (slots 0, 1)
    assert np.array_equal(a[:4], pool_nhd[5])
    assert np.array_equal(a[4:8], pool_nhd[0])
    assert np.array_equal(a[8:], pool_nhd[2, :2])
    # the 5-D storage [pages, 2, P, H, D] holds K at index 0 of dim 1
    five_d = np.stack([pool_nhd, pool_nhd + 1], axis=1)
    c = ref.gather_request_kv(five_d[:, 0], layout="NHD", page_size=4, kv_indptr=indptr,
                              kv_indices=indices, req=0, kv_len=10)
    assert np.array_equal(a, c)


def test_gather_ragged_slices_rows():
    rng = np.random.default_rng(1)
    data = rng.integers(0, 2**16, size=(9, 2, 4), dtype=np.uint16)
    got = ref.gather_request_kv(data, layout="NHD", page_size=1, kv_indptr=[0, 4, 9],
                                kv_indices=None, req=1, kv_len=5, kv_ragged=True)
    assert np.array_equal(got, data[4:9])


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 64, 1001])
def test_packbits_matches_numpy_little(n):
    rng = np.random.default_rng(n)
    bools = (rng.random(n) < 0.5).astype(np.uint8)
    want = np.packbits(bools, bitorder="little")
    got = ref.packbits_little(bools)
    assert got.dtype == np.uint8 and np.array_equal(got, want)
    unpacked = np.unpackbits(want, bitorder="little")
    assert all(ref.mask_bit(got, k) == bool(unpacked[k]) for k in range(n))


def test_packbits_nonzero_is_true():
    assert np.array_equal(ref.packbits_little([0, 2, 0, 255, 1]), np.array([0b11010], np.uint8))


def test_bf16_widening_exact():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x7F80], dtype=np.uint16)
    got = ref.bf16_bits_to_f64(bits)
    assert got[0] == 1.0 and got[1] == -1.0 and got[3] == 0.0 and np.isinf(got[4])
    assert got[2] == 3.140625
