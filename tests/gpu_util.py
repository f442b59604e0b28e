"""Helpers for the GPU parity tests: move a seeded batch to the device, run
it through the C ABI, and compare with the oracle."""
import numpy as np
import torch

import paged_kv_attention_plan_gb300 as pka
from oracle import ref

# Parity bar: bf16 outputs within max-abs 2e-2 and mean-abs 2e-3 of the fp64
# oracle, LSE (fp32, base 2) within 1e-4 absolute.
O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-4


def bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def kv_tensor(pool: np.ndarray, device="cuda") -> torch.Tensor:
    """A K/V pool on the device: bf16 from bit patterns, or uint8 e4m3 codes."""
    if pool.dtype == np.uint8:
        return torch.from_numpy(np.ascontiguousarray(pool)).to(device)
    return bf16(pool, device)


def i32(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


def run_gpu(b, split=("auto", 1), packed_mask=None, attn=None, with_lse=True, **plan_kw):
    attn = attn or pka.BatchAttention()
    qo = None if b.is_decode else b.qo_indptr
    info = attn.plan(qo, b.kv_indptr, b.last_page_len, num_qo_heads=b.num_qo_heads,
                     num_kv_heads=b.num_kv_heads, head_dim=b.head_dim, page_size=b.page_size,
                     layout=b.layout, mask_mode=b.mask_mode, kv_ragged=b.kv_ragged,
                     split_mode=split[0], fixed_split_pages=split[1], kv_dtype=b.kv_dtype,
                     k_scale=b.k_scale, v_scale=b.v_scale, **plan_kw)
    q = bf16(b.q)
    k, v = kv_tensor(b.k_pool), kv_tensor(b.v_pool)
    idx = i32(b.kv_indices)
    mask = None if packed_mask is None else torch.from_numpy(packed_mask).cuda()
    o, lse = attn.run(q, k, v, idx, mask, return_lse=with_lse)
    torch.cuda.synchronize()
    assert pka.pka_get_device_error() == 0
    return f64(o), (f64(lse) if with_lse else None), info


def run_oracle(b, packed_mask=None, rows=None):
    return ref.batch_attention(b.q, b.k_pool, b.v_pool, qo_indptr=b.qo_indptr,
                               kv_indptr=b.kv_indptr, kv_indices=b.kv_indices,
                               last_page_len=b.last_page_len, page_size=b.page_size,
                               num_qo_heads=b.num_qo_heads, num_kv_heads=b.num_kv_heads,
                               layout=b.layout, mask_mode=b.mask_mode, packed_mask=packed_mask,
                               sm_scale=b.sm_scale or None, kv_ragged=b.kv_ragged, rows=rows,
                               kv_dtype=b.kv_dtype, k_scale=b.k_scale, v_scale=b.v_scale)


def assert_parity(o, lse, o_ref, lse_ref, rows=None):
    if rows is not None:
        rows = sorted(rows)
        o, o_ref = o[rows], o_ref[rows]
        if lse is not None:
            lse, lse_ref = lse[rows], lse_ref[rows]
    assert np.all(np.isfinite(o_ref))
    assert np.all(np.isfinite(o)), "non-finite output"
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX, f"max abs error {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"mean abs error {err.mean():.3e}"
    if lse is not None:
        fin = np.isfinite(lse_ref)
        assert np.array_equal(fin, np.isfinite(lse)), "LSE -inf pattern differs"
        if fin.any():
            e = np.abs(lse[fin] - lse_ref[fin]).max()
            assert e <= LSE_MAX, f"LSE max abs error {e:.3e}"
        assert np.all(lse[~fin] == lse_ref[~fin])


def plan_item_rows(attn):
    """Global query rows at both ends of every work item of the plan `attn`
    holds, read from its plan image: each decode item's row, and the first
    and last token of every 128-row query tile of every tensor-core item.
    Comparing these rows with the oracle touches every item of the real plan,
    every split piece and the first and last item of every CTA."""
    from tests.plan_image import parse
    pka.pka_plan_wait(attn.handle)
    img = parse(attn.pinned.numpy()[: int(attn.info.int_ws_bytes)])
    g = attn.params.num_qo_heads // attn.params.num_kv_heads
    tq = 128 // g
    rows = set()
    for w in img["decode_items"]:
        rows.add(w["q_row0"])
    for w in img["prefill_items"]:
        for t0 in range(0, w["q_count"], tq):
            rows.add(w["q_row0"] + t0)
            rows.add(w["q_row0"] + min(t0 + tq, w["q_count"]) - 1)
    return rows
