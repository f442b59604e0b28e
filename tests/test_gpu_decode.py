"""GPU parity of the decode path (qo_len == 1 rows) against the oracle.

Covers NHD and HND pages, page sizes 1..32, head ratios 1/2/4/8, head_dim
64/128, split off / auto / fixed {1, 2, 7} pages, custom masks on decode
rows, ragged K/V, and the 64-request batch-decode workload at full size.
"""
import numpy as np
import pytest
import torch

from oracle import ref
from inputs import workloads as W
from tests.gpu_util import assert_parity, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _decode_batch(seed, kv, page_size=4, layout="NHD", hq=4, hk=2, d=64):
    return W.make_paged_batch(seed, np.ones(len(kv), np.int32), kv, page_size=page_size,
                              layout=layout, hq=hq, hk=hk, d=d, name="decode", is_decode=True)


@pytest.mark.parametrize("split", [("off", 1), ("auto", 1), ("fixed", 1), ("fixed", 2),
                                   ("fixed", 7)])
def test_worked_lengths_as_decode(split):
    b = _decode_batch(1, [6, 2, 9])
    o, lse, _ = run_gpu(b, split)
    assert_parity(o, lse, *run_oracle(b))


@pytest.mark.parametrize("layout", ["NHD", "HND"])
@pytest.mark.parametrize("page_size", [1, 3, 8, 16, 32])
@pytest.mark.parametrize("hq,hk,d", [(32, 8, 128), (8, 8, 64), (16, 8, 128), (16, 2, 64),
                                     (64, 8, 128), (32, 16, 128)])
def test_decode_shapes(layout, page_size, hq, hk, d):
    rng = np.random.default_rng(page_size * 131 + hq + d)
    kv = rng.integers(1, 700, size=7)
    kv[0] = 1
    b = _decode_batch(int(rng.integers(1 << 30)), kv, page_size, layout, hq, hk, d)
    for split in (("auto", 1), ("fixed", 2)):
        o, lse, _ = run_gpu(b, split)
        assert_parity(o, lse, *run_oracle(b))


def test_decode_custom_mask():
    b = _decode_batch(5, [40, 1, 77, 300], page_size=16, hq=32, hk=8, d=128)
    b.mask_mode = "custom"
    rng = np.random.default_rng(0)
    bits = rng.random(int(np.sum(b.kv_lens))) < 0.3
    bits[np.cumsum(b.kv_lens) - 1] = True  # every row keeps its newest key
    packed = ref.packbits_little(bits)
    o, lse, _ = run_gpu(b, ("fixed", 1), packed_mask=packed)
    assert_parity(o, lse, *run_oracle(b, packed_mask=packed))


def test_decode_fully_masked_row_is_zero_and_minus_inf():
    b = _decode_batch(6, [20, 5], page_size=4, hq=8, hk=2, d=64)
    b.mask_mode = "custom"
    bits = np.ones(25, bool)
    bits[:20] = False  # request 0 sees nothing
    packed = ref.packbits_little(bits)
    o, lse, _ = run_gpu(b, ("fixed", 2), packed_mask=packed)
    o_ref, lse_ref = run_oracle(b, packed_mask=packed)
    assert np.all(o[0] == 0) and np.all(lse[0] == -np.inf)
    assert_parity(o, lse, o_ref, lse_ref)


def test_decode_ragged_kv():
    lens = np.array([1, 33, 0, 250], np.int32)
    b = W.make_ragged_batch(7, lens, hq=16, hk=4, d=128, mask_mode="none")
    b.qo_lens = np.ones(4, np.int32)
    b.qo_indptr = np.arange(5, dtype=np.int32)
    b.q = b.q[:4]
    b.is_decode = True
    o, lse, _ = run_gpu(b, ("auto", 1))
    o_ref, lse_ref = run_oracle(b)
    assert np.all(o[2] == 0) and np.all(lse[2] == -np.inf)
    assert_parity(o, lse, o_ref, lse_ref)


def test_decode_five_d_storage():
    """K and V interleaved in one [pages, 2, P, Hk, D] tensor (page stride 2*P*Hk*D)."""
    b = _decode_batch(8, [50, 17, 3], page_size=8, hq=8, hk=2, d=64)
    from tests.gpu_util import bf16, f64, i32
    import paged_kv_attention_plan_gb300 as pka
    cache = torch.stack([bf16(b.k_pool), bf16(b.v_pool)], dim=1).contiguous()
    attn = pka.BatchAttention()
    attn.plan(None, b.kv_indptr, b.last_page_len, num_qo_heads=8, num_kv_heads=2, head_dim=64,
              page_size=8)
    o, lse = attn.run(bf16(b.q), cache[:, 0], cache[:, 1], i32(b.kv_indices))
    torch.cuda.synchronize()
    assert_parity(f64(o), f64(lse), *run_oracle(b))


@pytest.mark.parametrize("split", [("auto", 1), ("off", 1)])
def test_batch_decode_full_size(split):
    b = W.batch_decode()
    o, lse, info = run_gpu(b, split)
    assert_parity(o, lse, *run_oracle(b))
    if split[0] == "auto":
        assert info.num_merge_tasks > 0  # the bench configuration splits


def test_plan_reuse_after_page_remap():
    """kv_indices is read at run time: moving pages needs no new plan."""
    b = _decode_batch(9, [30, 64, 5], page_size=4, hq=8, hk=2, d=64)
    import paged_kv_attention_plan_gb300 as pka
    from tests.gpu_util import bf16, f64, i32
    attn = pka.BatchAttention()
    attn.plan(None, b.kv_indptr, b.last_page_len, num_qo_heads=8, num_kv_heads=2, head_dim=64,
              page_size=4, split_mode="fixed", fixed_split_pages=3)
    perm = np.random.default_rng(1).permutation(b.k_pool.shape[0])
    k2, v2 = np.empty_like(b.k_pool), np.empty_like(b.v_pool)
    k2[perm], v2[perm] = b.k_pool, b.v_pool
    b2 = _decode_batch(9, [30, 64, 5], page_size=4, hq=8, hk=2, d=64)
    b2.k_pool, b2.v_pool, b2.kv_indices = k2, v2, perm[b.kv_indices].astype(np.int32)
    for bb in (b, b2):
        o, lse = attn.run(bf16(bb.q), bf16(bb.k_pool), bf16(bb.v_pool), i32(bb.kv_indices))
        torch.cuda.synchronize()
        assert_parity(f64(o), f64(lse), *run_oracle(bb))


def test_split_decode_joins_rearm_across_runs():
    """Split decode rows are merged inside the decode kernel by the last
    piece to finish; its counters return to zero, so repeated runs of one
    plan give the same (bit-identical) result."""
    import paged_kv_attention_plan_gb300 as pka
    from tests.gpu_util import bf16, bits_of, f64, i32
    b = _decode_batch(10, [900, 33, 2000, 517, 1], page_size=16, hq=32, hk=8, d=128)
    attn = pka.BatchAttention()
    info = attn.plan(None, b.kv_indptr, b.last_page_len, num_qo_heads=32, num_kv_heads=8,
                     head_dim=128, page_size=16, split_mode="fixed", fixed_split_pages=9)
    assert info.num_decode_joins > 0
    q, k, v, idx = bf16(b.q), bf16(b.k_pool), bf16(b.v_pool), i32(b.kv_indices)
    o_ref, lse_ref = run_oracle(b)
    first = None
    for _ in range(3):
        o, lse = attn.run(q, k, v, idx)
        torch.cuda.synchronize()
        assert pka.pka_get_device_error() == 0
        assert_parity(f64(o), f64(lse), o_ref, lse_ref)
        got = (bits_of(o), f64(lse))
        if first is None:
            first = got
        else:
            assert np.array_equal(got[0], first[0]) and np.array_equal(got[1], first[1])


@pytest.mark.parametrize("d", [64, 128])
def test_split_decode_more_than_32_pieces(d):
    """One-page pieces: a row merges up to 125 states (lanes take pieces
    k, k + 32, ...)."""
    b = _decode_batch(11, [700, 1000, 40], page_size=8, hq=16, hk=2, d=d)
    o, lse, info = run_gpu(b, ("fixed", 1))
    assert info.num_decode_joins == 3 * 2  # 3 split rows x 2 kv heads
    assert_parity(o, lse, *run_oracle(b))


def test_split_decode_with_empty_pieces():
    """Pieces whose keys are all masked carry lse = -inf and no weight."""
    b = _decode_batch(12, [160, 96, 64], page_size=8, hq=8, hk=2, d=64)
    b.mask_mode = "custom"
    bits = np.zeros(int(np.sum(b.kv_lens)), bool)
    rng = np.random.default_rng(3)
    bits[100:160] = rng.random(60) < 0.5   # request 0: first 100 keys dropped
    bits[159] = True
    bits[160:256] = True                   # request 1: all visible
    # request 2 (keys 256..319): nothing visible -> zero output, -inf
    packed = ref.packbits_little(bits)
    o, lse, info = run_gpu(b, ("fixed", 2), packed_mask=packed)
    assert info.num_decode_joins > 0
    o_ref, lse_ref = run_oracle(b, packed_mask=packed)
    assert np.all(o[2] == 0) and np.all(lse[2] == -np.inf)
    assert_parity(o, lse, o_ref, lse_ref)
