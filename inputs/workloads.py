"""Seeded synthetic batches for paged KV attention.

This module only *constructs inputs*: request lengths, page tables, payload
tensors and boolean masks drawn from ``numpy.random.default_rng(seed)``.  It
holds none of the attention arithmetic (no scores, no softmax, no merge, no
planning, no packing of masks), so both the CUDA path and the CPU oracle can
take their inputs from here without sharing any of the method.

Shapes and distributions follow the workloads of the pages:

* the three-request batch of "Deep Dive - FlashInfer", section "Why inference
  attention becomes irregular" (query lengths 3/1/4, KV lengths 6/2/9,
  page size 4);
* the KV-cache layouts of "KV-Cache layouts" (FlashInfer docs), sections
  "NHD/HND", "Ragged Tensor", "Mask layout (2D Ragged Tensor)" and
  "Page table layout";
* the page-size-1 view of a token pool of "GPU attention backends: FlashInfer
  and FlashAttention" (mini-sglang), section "FlashInfer: plan and run".

Payloads are standard normal values rounded once to bfloat16 (round to nearest
even) and carried as raw ``uint16`` bit patterns, because NumPy has no bf16.
Unused page slots and unused pool pages are filled with a NaN bit pattern so
that any read past ``last_page_len`` shows up as a parity failure.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BF16_NAN_BITS = np.uint16(0x7FC1)
E4M3_NAN_CODE = np.uint8(0x7F)  # the e4m3 NaN (exponent and mantissa all ones)

NHD = "NHD"
HND = "HND"


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    out = ((u + rounding) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = BF16_NAN_BITS
    return out


def normal_bf16_bits(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0, 1) float32 draws rounded to bf16, as uint16 bits."""
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


@dataclass
class Batch:
    """One batch of the paged (or ragged) attention problem.

    Index arrays are int32, as the layout documentation requires.  ``k_pool``
    and ``v_pool`` are bf16 bit patterns in the layout named by ``layout``:
    NHD ``[pages, page_size, Hk, D]``, HND ``[pages, Hk, page_size, D]``; for
    ragged K/V they are ``[kv_indptr[-1], Hk, D]``.
    """

    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    layout: str
    mask_mode: str  # "none" | "causal" | "custom"
    qo_lens: np.ndarray
    kv_lens: np.ndarray
    qo_indptr: np.ndarray
    kv_indptr: np.ndarray
    kv_indices: np.ndarray
    last_page_len: np.ndarray
    kv_ragged: bool = False
    is_decode: bool = False
    sm_scale: float = 0.0  # 0 -> 1/sqrt(head_dim)
    q: np.ndarray | None = None
    k_pool: np.ndarray | None = None
    v_pool: np.ndarray | None = None
    mask_bool: np.ndarray | None = None  # flattened uint8 0/1, custom mask only
    kv_dtype: str = "bf16"  # "bf16" bit patterns, or "e4m3" codes (uint8 pools)
    k_scale: float = 1.0  # e4m3 pools: a code c stands for e4m3(c) * scale
    v_scale: float = 1.0
    k_new: np.ndarray | None = None  # appended rows [nnz_q, Hk, D] (bits)
    v_new: np.ndarray | None = None
    extra: dict = field(default_factory=dict)

    @property
    def batch_size(self) -> int:
        return int(len(self.kv_lens))

    @property
    def nnz_q(self) -> int:
        return int(self.qo_indptr[-1])

    @property
    def num_pages_total(self) -> int:
        return int(self.k_pool.shape[0]) if self.k_pool is not None else 0


def _prefix(lengths) -> np.ndarray:
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return out.astype(np.int32)


def build_page_table(rng, kv_lens, page_size, pool_pages=None, page_ids=None):
    """Draw page ids for each request (seeded permutation of the pool).

    Returns (kv_indptr, kv_indices, last_page_len, pool_pages).
    """
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    pages_per_req = (kv_lens + page_size - 1) // page_size
    total = int(pages_per_req.sum())
    if page_ids is None:
        if pool_pages is None:
            pool_pages = total
        assert pool_pages >= total
        page_ids = rng.permutation(pool_pages)[:total]
    else:
        page_ids = np.asarray(page_ids)
        assert pool_pages is not None
    kv_indptr = _prefix(pages_per_req)
    last = (kv_lens - (pages_per_req - 1) * page_size).astype(np.int32)
    return kv_indptr, np.asarray(page_ids, dtype=np.int32), last, int(pool_pages)


def e4m3_codes(rng: np.random.Generator, shape) -> np.ndarray:
    """Random e4m3 codes of either sign with exponent field 3..8 and any
    mantissa: magnitudes 1/16 .. 3.75, an N(0,1)-like spread that stays away
    from the format's subnormals, its largest values and its NaN."""
    sign = rng.integers(0, 2, size=shape).astype(np.uint8) << 7
    exp = rng.integers(3, 9, size=shape).astype(np.uint8) << 3
    man = rng.integers(0, 8, size=shape).astype(np.uint8)
    return (sign | exp | man).astype(np.uint8)


def fill_pool(rng, kv_lens, kv_indptr, kv_indices, page_size, pool_pages, hk, d, layout,
              kv_dtype="bf16"):
    """Pool tensors with payload in used slots and NaN elsewhere: N(0,1) bf16
    bit patterns, or e4m3 codes (kv_dtype "e4m3")."""
    shape = (pool_pages, page_size, hk, d) if layout == NHD else (pool_pages, hk, page_size, d)
    if kv_dtype == "e4m3":
        k = np.full(shape, E4M3_NAN_CODE, dtype=np.uint8)
        v = np.full(shape, E4M3_NAN_CODE, dtype=np.uint8)
    else:
        k = np.full(shape, BF16_NAN_BITS, dtype=np.uint16)
        v = np.full(shape, BF16_NAN_BITS, dtype=np.uint16)
    fill_pages(rng, k, v, kv_lens, kv_indptr, kv_indices, page_size, layout)
    return k, v


def fill_pages(rng, k, v, kv_lens, kv_indptr, kv_indices, page_size, layout):
    """Write random rows (N(0,1) bf16, or e4m3 codes for a uint8 pool) into
    the slots of each request's pages, in place."""
    draw = e4m3_codes if k.dtype == np.uint8 else normal_bf16_bits
    for r, n in enumerate(np.asarray(kv_lens)):
        n = int(n)
        if n == 0:
            continue
        rows_k = draw(rng, (n,) + k.shape[-2:] if layout == NHD else
                      (n, k.shape[1], k.shape[3]))
        rows_v = draw(rng, rows_k.shape)
        pages = kv_indices[kv_indptr[r]:kv_indptr[r + 1]]
        for j0 in range(0, n, page_size):
            pg = int(pages[j0 // page_size])
            cnt = min(page_size, n - j0)
            if layout == NHD:
                k[pg, :cnt] = rows_k[j0:j0 + cnt]
                v[pg, :cnt] = rows_v[j0:j0 + cnt]
            else:
                k[pg, :, :cnt] = rows_k[j0:j0 + cnt].transpose(1, 0, 2)
                v[pg, :, :cnt] = rows_v[j0:j0 + cnt].transpose(1, 0, 2)


def make_paged_batch(seed, qo_lens, kv_lens, *, page_size, layout=NHD, hq=32, hk=8, d=128,
                     mask_mode="causal", pool_pages=None, page_ids=None, name="paged",
                     is_decode=False, with_payload=True, append_new=False, kv_dtype="bf16",
                     k_scale=1.0, v_scale=1.0):
    """Generic paged batch.  With ``append_new`` only the cached prefix of
    every request (its first ``kv_len - qo_len`` positions) is written into
    the pool; the slots of its last ``qo_len`` positions stay NaN, and the
    rows append_paged_kv_cache will write there are drawn separately into
    ``k_new``/``v_new`` ([nnz_q, Hk, D] bf16 bits)."""
    rng = np.random.default_rng(seed)
    qo_lens = np.asarray(qo_lens, dtype=np.int32)
    kv_lens = np.asarray(kv_lens, dtype=np.int32)
    kv_indptr, kv_indices, last, pool = build_page_table(
        rng, kv_lens, page_size, pool_pages=pool_pages, page_ids=page_ids)
    b = Batch(name=name, num_qo_heads=hq, num_kv_heads=hk, head_dim=d, page_size=page_size,
              layout=layout, mask_mode=mask_mode, qo_lens=qo_lens, kv_lens=kv_lens,
              qo_indptr=_prefix(qo_lens), kv_indptr=kv_indptr, kv_indices=kv_indices,
              last_page_len=last, is_decode=is_decode, kv_dtype=kv_dtype, k_scale=k_scale,
              v_scale=v_scale)
    b.extra["pool_pages"] = pool
    if with_payload:
        b.q = normal_bf16_bits(rng, (b.nnz_q, hq, d))
        filled = kv_lens - qo_lens if append_new else kv_lens
        b.k_pool, b.v_pool = fill_pool(rng, filled, kv_indptr, kv_indices, page_size, pool,
                                       hk, d, layout, kv_dtype)
        if append_new:
            b.k_new = normal_bf16_bits(rng, (b.nnz_q, hk, d))
            b.v_new = normal_bf16_bits(rng, (b.nnz_q, hk, d))
    return b


def make_ragged_batch(seed, lens, *, hq=32, hk=32, d=128, mask_mode="custom", p_keep=0.5,
                      name="ragged", with_payload=True):
    """Ragged K/V (``kv_indptr`` counts tokens), qo_len == kv_len per request.

    The custom mask of each request is Bernoulli(p_keep) OR the causal
    pattern, flattened query-major and concatenated over requests."""
    rng = np.random.default_rng(seed)
    lens = np.asarray(lens, dtype=np.int32)
    indptr = _prefix(lens)
    b = Batch(name=name, num_qo_heads=hq, num_kv_heads=hk, head_dim=d, page_size=1,
              layout=NHD, mask_mode=mask_mode, qo_lens=lens.copy(), kv_lens=lens.copy(),
              qo_indptr=indptr.copy(), kv_indptr=indptr.copy(),
              kv_indices=np.arange(int(indptr[-1]), dtype=np.int32),
              last_page_len=np.ones(len(lens), dtype=np.int32), kv_ragged=True)
    if with_payload:
        total = int(indptr[-1])
        b.q = normal_bf16_bits(rng, (total, hq, d))
        b.k_pool = normal_bf16_bits(rng, (total, hk, d))
        b.v_pool = normal_bf16_bits(rng, (total, hk, d))
    if mask_mode == "custom":
        parts = []
        for n in lens:
            n = int(n)
            keep = rng.random((n, n)) < p_keep
            keep |= np.tri(n, n, dtype=bool)
            parts.append(keep.reshape(-1))
        b.mask_bool = (np.concatenate(parts) if parts else np.zeros(0, bool)).astype(np.uint8)
    return b


@dataclass
class Cascade:
    """Multi-level cascade batch: every level splits the same query rows into
    nodes with their own page lists in one pool ("KV-Cache layouts",
    "Multi-level cascade inference data layout").  ``levels`` runs from the
    root; each entry holds int32 qo_indptr, kv_indptr, kv_indices,
    last_page_len and kv_lens.  A node without keys has no pages (its
    last_page_len is 1 and unused)."""

    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    layout: str
    mask_mode: str
    qo_lens: np.ndarray
    levels: list
    q: np.ndarray | None = None
    k_pool: np.ndarray | None = None
    v_pool: np.ndarray | None = None

    @property
    def nnz_q(self) -> int:
        return int(self.levels[-1]["qo_indptr"][-1])

    @property
    def kv_indices(self) -> np.ndarray:
        """Page ids of all levels, concatenated in level order."""
        return np.concatenate([lv["kv_indices"] for lv in self.levels]).astype(np.int32)


def make_cascade_batch(seed, qo_lens, own_kv_lens, shared, *, page_size, layout=NHD, hq=32,
                       hk=8, d=128, mask_mode="causal", with_payload=True, name="cascade",
                       kv_dtype="bf16"):
    """Cascade over requests with query lengths ``qo_lens`` and own (last-level)
    KV lengths ``own_kv_lens``.  ``shared`` lists the levels above the last,
    root first; each is a list of (requests, kv_len) nodes that partition the
    requests in order.  Page ids are a seeded permutation of a pool with
    exactly the pages needed, consumed level by level; unused slots hold NaN
    (bf16 bits, or the e4m3 NaN code for kv_dtype "e4m3")."""
    rng = np.random.default_rng(seed)
    qo_lens = np.asarray(qo_lens, dtype=np.int64)
    q_ptr = _prefix(qo_lens)
    specs = []
    for nodes in shared:
        counts = [int(c) for c, _ in nodes]
        assert sum(counts) == len(qo_lens), "shared nodes must partition the requests"
        bounds = np.concatenate([[0], np.cumsum(counts)])
        node_qo = [int(q_ptr[bounds[i + 1]] - q_ptr[bounds[i]]) for i in range(len(nodes))]
        specs.append((np.asarray(node_qo), np.asarray([int(k) for _, k in nodes])))
    specs.append((qo_lens, np.asarray(own_kv_lens, dtype=np.int64)))
    pages = [(kv + page_size - 1) // page_size for _, kv in specs]
    total = int(sum(int(p.sum()) for p in pages))
    ids = rng.permutation(total).astype(np.int32)
    levels, used = [], 0
    for (qo, kv), pg in zip(specs, pages):
        n_pages = int(pg.sum())
        last = np.where(kv > 0, kv - (pg - 1) * page_size, 1).astype(np.int32)
        levels.append(dict(qo_indptr=_prefix(qo), kv_indptr=_prefix(pg),
                           kv_indices=ids[used:used + n_pages].copy(), last_page_len=last,
                           kv_lens=kv.astype(np.int32)))
        used += n_pages
    c = Cascade(name=name, num_qo_heads=hq, num_kv_heads=hk, head_dim=d, page_size=page_size,
                layout=layout, mask_mode=mask_mode, qo_lens=qo_lens.astype(np.int32),
                levels=levels)
    if with_payload:
        c.q = normal_bf16_bits(rng, (int(q_ptr[-1]), hq, d))
        shape = (total, page_size, hk, d) if layout == NHD else (total, hk, page_size, d)
        if kv_dtype == "e4m3":
            c.k_pool = np.full(shape, E4M3_NAN_CODE, dtype=np.uint8)
            c.v_pool = np.full(shape, E4M3_NAN_CODE, dtype=np.uint8)
        else:
            c.k_pool = np.full(shape, BF16_NAN_BITS, dtype=np.uint16)
            c.v_pool = np.full(shape, BF16_NAN_BITS, dtype=np.uint16)
        for lv in levels:
            fill_pages(rng, c.k_pool, c.v_pool, lv["kv_lens"], lv["kv_indptr"], lv["kv_indices"],
                       page_size, layout)
    return c


# ---------------------------------------------------------------------------
# The five workloads of the benchmark and parity suite.
# ---------------------------------------------------------------------------

def worked_example(seed=1000, literal_pages=False, hq=4, hk=2, d=64):
    """Three requests: qo_lens 3/1/4, kv_lens 6/2/9, page size 4, causal.

    ``literal_pages`` uses the page ids printed in "Deep Dive - FlashInfer"
    ([7, 2], [11], [3, 14, 6] in a 15-page pool); otherwise the six pages are a
    seeded permutation of a 16-page pool."""
    ids = [7, 2, 11, 3, 14, 6] if literal_pages else None
    pool = 15 if literal_pages else 16
    return make_paged_batch(seed, [3, 1, 4], [6, 2, 9], page_size=4, layout=NHD, hq=hq, hk=hk,
                            d=d, mask_mode="causal", pool_pages=pool, page_ids=ids,
                            name="worked_example")


def batch_decode(seed=1001, n=64, kv_lo=512, kv_hi=4096, page_size=16, layout=NHD, hq=32,
                 hk=8, d=128, with_payload=True, kv_dtype="bf16", k_scale=1.0, v_scale=1.0):
    """64 decode requests, kv_len ~ U[512, 4096], page size 16, 32/8 heads
    (K/V as bf16, or as e4m3 codes with per-pool scales)."""
    rng = np.random.default_rng(seed)
    kv = rng.integers(kv_lo, kv_hi, size=n, endpoint=True)
    return make_paged_batch(seed + 7, np.ones(n, np.int32), kv, page_size=page_size,
                            layout=layout, hq=hq, hk=hk, d=d, mask_mode="causal",
                            name="batch_decode", is_decode=True, with_payload=with_payload,
                            kv_dtype=kv_dtype, k_scale=k_scale, v_scale=v_scale)


def append_prefill(seed=1002, n=16, q_lo=128, q_hi=1024, prefix_hi=4096, page_size=16,
                   layout=NHD, hq=32, hk=8, d=128, with_payload=True, kv_dtype="bf16",
                   k_scale=1.0, v_scale=1.0):
    """16 requests, qo_len ~ U[128,1024], cached prefix ~ U[0,4096], causal.
    New K/V rows come in ``k_new``/``v_new`` (bf16) for append_paged_kv_cache;
    with kv_dtype "e4m3" the cached prefix is e4m3 codes."""
    rng = np.random.default_rng(seed)
    ql = rng.integers(q_lo, q_hi, size=n, endpoint=True)
    pre = rng.integers(0, prefix_hi, size=n, endpoint=True)
    return make_paged_batch(seed + 7, ql, pre + ql, page_size=page_size, layout=layout, hq=hq,
                            hk=hk, d=d, mask_mode="causal", name="append_prefill",
                            with_payload=with_payload, append_new=with_payload,
                            kv_dtype=kv_dtype, k_scale=k_scale, v_scale=v_scale)


def mixed_step(seed=1003, page_size=1, layout=NHD, n_long=8, long_lo=32768, long_hi=131072,
               n_short=120, short_lo=64, short_hi=2048, n_chunk=4, chunk=512, prefix_hi=8192,
               hq=32, hk=8, d=128, with_payload=True):
    """8 long + 120 short decodes and 4 prefill chunks of 512 tokens."""
    rng = np.random.default_rng(seed)
    kv_long = rng.integers(long_lo, long_hi, size=n_long, endpoint=True)
    kv_short = rng.integers(short_lo, short_hi, size=n_short, endpoint=True)
    pre = rng.integers(0, prefix_hi, size=n_chunk, endpoint=True)
    qo = np.concatenate([np.ones(n_long + n_short, np.int64), np.full(n_chunk, chunk)])
    kv = np.concatenate([kv_long, kv_short, pre + chunk])
    return make_paged_batch(seed + 7, qo, kv, page_size=page_size, layout=layout, hq=hq, hk=hk,
                            d=d, mask_mode="causal", name=f"mixed_step_p{page_size}_{layout}",
                            with_payload=with_payload)


def shared_prompt_decode(seed=1005, n=64, prompt=32768, own_lo=512, own_hi=2048, page_size=16,
                         layout=NHD, hq=32, hk=8, d=128, with_payload=True):
    """Two-level cascade: ``n`` decode rows share a ``prompt``-token root node;
    each request's own suffix is U[own_lo, own_hi] tokens (its newest token
    included)."""
    rng = np.random.default_rng(seed)
    own = rng.integers(own_lo, own_hi, size=n, endpoint=True)
    return make_cascade_batch(seed, np.ones(n, np.int64), own, [[(n, prompt)]],
                              page_size=page_size, layout=layout, hq=hq, hk=hk, d=d,
                              with_payload=with_payload, name="shared_prompt_decode")


def ragged_custom_mask(seed=1004, n=8, lo=256, hi=2048, hq=32, hk=32, d=128, with_payload=True):
    """8 requests, qo_len == kv_len ~ U[256, 2048], ragged K/V, custom mask."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(lo, hi, size=n, endpoint=True)
    return make_ragged_batch(seed + 7, lens, hq=hq, hk=hk, d=d, mask_mode="custom",
                             name="ragged_custom_mask", with_payload=with_payload)
