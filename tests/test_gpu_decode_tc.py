"""GPU parity of decode rows run on the tensor-core (tcgen05) kernel
(decode_on_tensor_cores): each row is an item of one query token whose g qo
heads fill the first rows of the 128-row tile.

Covers NHD and HND pages, page sizes 1 and 16, head ratios 1/4/8, head dims
64/128, split auto and fixed, a custom mask on decode rows, a mixed batch
(decode and prefill rows in one tensor-core launch) and the 64-request
batch-decode workload at full size.
"""
import numpy as np
import pytest

from oracle import ref
from inputs import workloads as W
from tests.gpu_util import assert_parity, run_gpu, run_oracle

pytestmark = pytest.mark.gpu
TC = dict(decode_on_tensor_cores=True)


def _decode_batch(seed, kv, page_size=4, layout="NHD", hq=4, hk=2, d=64):
    return W.make_paged_batch(seed, np.ones(len(kv), np.int32), kv, page_size=page_size,
                              layout=layout, hq=hq, hk=hk, d=d, name="decode", is_decode=True)


@pytest.mark.parametrize("split", [("off", 1), ("auto", 1), ("fixed", 2)])
def test_tc_worked_lengths_as_decode(split):
    b = _decode_batch(1, [6, 2, 9])
    o, lse, info = run_gpu(b, split, **TC)
    assert info.num_decode_items == 0 and info.num_prefill_items > 0
    assert_parity(o, lse, *run_oracle(b))


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("page_size", [1, 16])
@pytest.mark.parametrize("hq,hk,d", [(32, 8, 128), (8, 8, 64), (64, 8, 128), (16, 2, 64)])
def test_tc_decode_shapes(layout, page_size, hq, hk, d):
    rng = np.random.default_rng(page_size * 7 + hq + d)
    kv = rng.integers(1, 700, size=6)
    kv[0] = 1
    b = _decode_batch(int(rng.integers(1 << 30)), kv, page_size, layout, hq, hk, d)
    for split in (("auto", 1), ("fixed", 3)):
        o, lse, _ = run_gpu(b, split, **TC)
        assert_parity(o, lse, *run_oracle(b))


def test_tc_decode_custom_mask():
    b = _decode_batch(5, [40, 1, 77, 300], page_size=16, hq=32, hk=8, d=128)
    b.mask_mode = "custom"
    rng = np.random.default_rng(0)
    bits = rng.random(int(np.sum(b.kv_lens))) < 0.3
    bits[np.cumsum(b.kv_lens) - 1] = True
    packed = ref.packbits_little(bits)
    o, lse, _ = run_gpu(b, ("fixed", 1), packed_mask=packed, **TC)
    assert_parity(o, lse, *run_oracle(b, packed_mask=packed))


def test_tc_mixed_decode_and_prefill():
    b = W.make_paged_batch(9, [1, 37, 1, 5, 1], [300, 400, 17, 90, 1], page_size=16, hq=32,
                           hk=8, d=128)
    o, lse, info = run_gpu(b, ("auto", 1), **TC)
    assert info.num_decode_items == 0
    assert_parity(o, lse, *run_oracle(b))


def test_tc_batch_decode_full_size():
    b = W.batch_decode()
    o, lse, info = run_gpu(b, ("auto", 1), **TC)
    assert info.num_decode_items == 0
    assert_parity(o, lse, *run_oracle(b))


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_tc_decode_e4m3(layout):
    """Decode rows on the tensor-core kernel over e4m3 pools: every request's
    keys are decoded to the bf16 scratch, which the tile reads as ragged K/V."""
    qo = np.array([1, 1, 37, 1, 1], np.int32)
    kv = np.array([300, 1, 60, 2000, 17], np.int32)
    b = W.make_paged_batch(41, qo, kv, page_size=16, layout=layout, hq=32, hk=8, d=128,
                           kv_dtype="e4m3", k_scale=0.5, v_scale=1.5)
    o, lse, info = run_gpu(b, **TC)
    assert info.num_decode_items == 0 and info.kv_scratch_rows == int(kv.sum())
    assert_parity(o, lse, *run_oracle(b))
