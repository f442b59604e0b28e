"""GPU parity of the decode path over e4m3 K/V pools (one scale per pool)
against the oracle, which decodes each code by the format's definition.

Covers NHD and HND pages, page sizes 1, 3 and 16, head ratios 1/4/8, head
dims 64/128, split auto and fixed, scales of 1 and of 0.37 (K) / 1.9 (V),
ragged K/V, and the 64-request batch-decode workload at full size.
"""
import numpy as np
import pytest

from inputs import workloads as W
from tests.gpu_util import assert_parity, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _fp8_batch(seed, kv, page_size=4, layout="NHD", hq=8, hk=2, d=64, ks=1.0, vs=1.0):
    return W.make_paged_batch(seed, np.ones(len(kv), np.int32), kv, page_size=page_size,
                              layout=layout, hq=hq, hk=hk, d=d, name="decode_fp8",
                              is_decode=True, kv_dtype="e4m3", k_scale=ks, v_scale=vs)


def test_fp8_worked_lengths():
    b = _fp8_batch(1, [6, 2, 9])
    for split in (("off", 1), ("auto", 1), ("fixed", 1)):
        o, lse, _ = run_gpu(b, split)
        assert_parity(o, lse, *run_oracle(b))


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("page_size", [1, 3, 16])
@pytest.mark.parametrize("hq,hk,d", [(32, 8, 128), (8, 8, 64), (16, 2, 64), (64, 8, 128)])
@pytest.mark.parametrize("scales", [(1.0, 1.0), (0.37, 1.9)])
def test_fp8_decode_shapes(layout, page_size, hq, hk, d, scales):
    rng = np.random.default_rng(page_size * 17 + hq + d)
    kv = rng.integers(1, 600, size=6)
    kv[0] = 1
    b = _fp8_batch(int(rng.integers(1 << 30)), kv, page_size, layout, hq, hk, d, *scales)
    for split in (("auto", 1), ("fixed", 2)):
        o, lse, _ = run_gpu(b, split)
        assert_parity(o, lse, *run_oracle(b))


def test_fp8_ragged_kv():
    lens = np.array([1, 33, 250, 7], np.int32)
    b = W.make_ragged_batch(8, lens, hq=16, hk=4, d=128, mask_mode="none", with_payload=False)
    rng = np.random.default_rng(8)
    b.q = W.normal_bf16_bits(rng, (4, 16, 128))
    b.k_pool = W.e4m3_codes(rng, (int(lens.sum()), 4, 128))
    b.v_pool = W.e4m3_codes(rng, (int(lens.sum()), 4, 128))
    b.qo_lens = np.ones(4, np.int32)
    b.qo_indptr = np.arange(5, dtype=np.int32)
    b.is_decode = True
    b.kv_dtype, b.k_scale, b.v_scale = "e4m3", 0.5, 2.0
    o, lse, _ = run_gpu(b, ("auto", 1))
    assert_parity(o, lse, *run_oracle(b))


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_fp8_batch_decode_full_size(layout):
    b = W.batch_decode(layout=layout, kv_dtype="e4m3", k_scale=0.6, v_scale=1.5)
    o, lse, info = run_gpu(b, ("auto", 1))
    assert info.num_decode_joins > 0
    assert_parity(o, lse, *run_oracle(b))
