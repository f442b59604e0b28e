"""CPU oracle for batched paged-KV attention — TEST INFRASTRUCTURE ONLY.

Only the test-suite, the smoke check and the CPU-baseline leg of the benchmark
may import this module.  The product path never calls it, and it shares no
code with the CUDA library or its planner.

Everything here is the plain definition, in float64 NumPy, written from the
pages it cites; nothing is blocked, fused or reordered:

* "Deep Dive - FlashInfer" (leetllm.com): sections "Why inference attention
  becomes irregular" (the length contract and the two pointer arrays),
  "Causality uses logical positions, not page numbers" (address of a logical
  token, the bottom-right causal rule j <= K - Q + i), "Core mechanism:
  schedule work around state" and "A worked split-KV example" (the attention
  state (o, b) with b the base-2 log of the natural-exp sum, and the two-way
  state merge with normalised scales and explicit empty states).
* "KV-Cache layouts" (FlashInfer docs, Chinese translation): sections
  "NHD/HND", "Ragged Tensor", "Mask layout (2D Ragged Tensor)" (row-major
  per-request masks, mask_indptr = cumsum(qo_len * kv_len), little-endian bit
  packing) and "Page table layout" (CSR page table, the length contract, 5-D
  and tuple storage).
* "GPU attention backends: FlashInfer and FlashAttention" (mini-sglang):
  sections "FlashInfer: plan and run" (page-size-1 view of a token pool) and
  "FlashAttention: a page-number table" (page-number table to CSR).
* "KV-Cache layouts", section "Multi-level cascade inference data layout"
  (per-level qo_indptr / kv_indptr / kv_indices / last_page_len over one
  pool): cascade_attention.
* 8-bit K/V: the e4m3 format as its published definition states it (OCP
  "8-bit floating point" specification: 1 sign bit, 4 exponent bits with
  bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN), and the pages'
  note that low-precision caches use the HND layout ("KV-Cache layouts",
  "NHD/HND").  The pages give no scale contract; the reading taken is one
  scale per K pool and one per V pool: a stored code c stands for
  e4m3(c) * scale.

Readings where the pages are silent (each is listed in the design notes):
bit 1 of a custom mask keeps a key; the mask is applied after scaling; a row
that sees no key returns a zero vector and lse = -inf; new tokens of a request
occupy its last qo_len logical positions; qo head h reads kv head h // g; in
a cascade, keys of levels above the last are all visible to the rows below
them and only the last level carries the mask.

Pins (tests that tie this module to something other than itself) live in
tests/test_oracle_*.py; every function below has at least one.
"""
from __future__ import annotations

import math

import numpy as np

LN2 = math.log(2.0)


# ---------------------------------------------------------------------------
# bf16 payload decoding (payloads travel as raw uint16 bit patterns)
# ---------------------------------------------------------------------------

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float64 (exact: bf16 is the top half of fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Decode e4m3 codes (uint8) to float64 by the format's definition.

    sign s = bit 7, exponent e = bits 6..3 (bias 7), mantissa m = bits 2..0:
    e = 0 is subnormal, (-1)^s * m/8 * 2^(1-7); otherwise (-1)^s * (1 + m/8) *
    2^(e-7), except e = 15 with m = 7, which is NaN (the format has no
    infinities, so e = 15 with m < 7 are the largest finite values)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    out = sign * mag
    return np.where((e == 15) & (c & 7 == 7), np.nan, out)


def f32_to_e4m3(x) -> np.ndarray:
    """Round float32 values to e4m3 codes: to the nearest value of the format
    (ties to the even code, the one whose lowest mantissa bit is 0), with
    magnitudes above the largest finite value 448 clamped to 448 (saturating:
    nothing finite becomes NaN) and NaN kept as the NaN code 0x7F."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    pos_codes = np.arange(0, 0x7F, dtype=np.uint8)  # +0 .. 448, increasing values
    pos_vals = e4m3_to_f64(pos_codes)
    a = np.minimum(np.abs(np.nan_to_num(x)), 448.0)
    hi = np.clip(np.searchsorted(pos_vals, a, side="left"), 0, len(pos_vals) - 1)
    lo = np.clip(hi - 1, 0, len(pos_vals) - 1)
    d_lo, d_hi = a - pos_vals[lo], pos_vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (pos_codes[hi] % 2 == 0))
    code = np.where(pick_hi, pos_codes[hi], pos_codes[lo]).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def quantize_kv_e4m3(bits: np.ndarray, scale: float) -> np.ndarray:
    """bf16 payload -> e4m3 codes of value / scale: the division in float32
    (correctly rounded), then the one rounding to e4m3 (f32_to_e4m3)."""
    v = bf16_bits_to_f64(bits).astype(np.float32)
    return f32_to_e4m3(v / np.float32(scale))


def kv_payload_to_f64(x, kv_dtype: str, scale: float) -> np.ndarray:
    """K or V payload as float64 values: bf16 bit patterns, or e4m3 codes
    times the pool's scale."""
    if kv_dtype == "bf16":
        return bf16_bits_to_f64(x)
    if kv_dtype == "e4m3":
        return e4m3_to_f64(x) * float(scale)
    raise ValueError(kv_dtype)


# ---------------------------------------------------------------------------
# Metadata: the length contract and the pointer arrays
# ("Deep Dive - FlashInfer", "Why inference attention becomes irregular";
#  "KV-Cache layouts", "Page table layout")
# ---------------------------------------------------------------------------

def kv_len_from_pages(page_ids, last_page_len: int, page_size: int) -> int:
    """KV length of one request: page_size * (num_pages - 1) + last_page_len.

    Rejects an empty page list, negative or non-integer page ids, and a tail
    outside 1..page_size (the documented range of last_page_len)."""
    if len(page_ids) == 0:
        raise ValueError("a request needs at least one page")
    for p in page_ids:
        if not isinstance(p, (int, np.integer)) or p < 0:
            raise ValueError("page ids must be non-negative integers")
    if not isinstance(last_page_len, (int, np.integer)) or not 1 <= last_page_len <= page_size:
        raise ValueError("last_page_len must lie in 1..page_size")
    return page_size * (len(page_ids) - 1) + int(last_page_len)


def indptr_from_lengths(lengths) -> list[int]:
    """[0, l0, l0+l1, ...]: the index-pointer array of a ragged dimension."""
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return out


def kv_lens_from_csr(kv_indptr, kv_indices, last_page_len, page_size) -> list[int]:
    """KV length of every request of a CSR page table (validated per request)."""
    lens = []
    for r in range(len(kv_indptr) - 1):
        pages = [int(p) for p in kv_indices[int(kv_indptr[r]):int(kv_indptr[r + 1])]]
        lens.append(kv_len_from_pages(pages, int(last_page_len[r]), page_size))
    return lens


def token_address(page_ids, j: int, page_size: int) -> tuple[int, int]:
    """Logical token j of a request -> (physical page, slot in page)."""
    return int(page_ids[j // page_size]), j % page_size


def causal_visible(i: int, j: int, qo_len: int, kv_len: int) -> bool:
    """Bottom-right aligned causal rule: query i (local) sees key j iff j <= K - Q + i."""
    return j <= kv_len - qo_len + i


def mask_indptr(qo_lens, kv_lens) -> list[int]:
    """Start of each request's flattened mask: prefix sums of qo_len * kv_len."""
    return indptr_from_lengths([int(a) * int(b) for a, b in zip(qo_lens, kv_lens)])


def packbits_little(bools) -> np.ndarray:
    """Pack 0/1 values 8 per byte, element k -> bit (k & 7) of byte k >> 3.

    Non-zero counts as 1; the high bits of a short last byte are 0."""
    flat = (np.asarray(bools).reshape(-1) != 0).astype(np.uint16)
    padded = np.zeros(((flat.size + 7) // 8) * 8, dtype=np.uint16)
    padded[:flat.size] = flat
    weights = np.array([1 << k for k in range(8)], dtype=np.uint16)  # bit k of each byte
    return (padded.reshape(-1, 8) * weights).sum(axis=1).astype(np.uint8)


def mask_bit(packed, k: int) -> bool:
    """Bit k of a little-endian packed mask."""
    return bool((int(packed[k >> 3]) >> (k & 7)) & 1)


def page_table_to_csr(page_table, seq_lens, page_size):
    """FlashAttention-style page-number table -> CSR (kv_indptr, kv_indices, last_page_len).

    Each request keeps ceil(len / P) leading entries of its row; the tail length
    is len - (pages - 1) * P."""
    indptr, indices, last = [0], [], []
    for row, n in zip(page_table, seq_lens):
        pages = (int(n) + page_size - 1) // page_size
        indices.extend(int(p) for p in row[:pages])
        indptr.append(indptr[-1] + pages)
        last.append(int(n) - (pages - 1) * page_size)
    return indptr, indices, last


def token_locations_to_page_numbers(token_row, seq_len: int, page_size: int) -> list[int]:
    """Every page_size-th token location of a request's row, divided by P."""
    return [int(x) // page_size for x in list(token_row[:seq_len])[::page_size]]


# ---------------------------------------------------------------------------
# Attention states and their merge
# ("Deep Dive - FlashInfer", "Core mechanism" and "A worked split-KV example")
# ---------------------------------------------------------------------------

def direct_state(scores, values):
    """Attention state of one query row over a key set.

    ``scores`` are the scaled logits s_j, ``values`` the value rows.  Returns
    (o, b) with o the softmax-weighted value (normalised over this key set) and
    b = log2(sum_j exp(s_j)).  An empty key set gives a zero vector and -inf."""
    scores = np.asarray(scores, dtype=np.float64).reshape(-1)
    values = np.asarray(values, dtype=np.float64)
    dim = values.shape[-1] if values.ndim == 2 else 0
    if scores.size == 0:
        return np.zeros(dim), -math.inf
    shift = scores.max()
    w = np.exp(scores - shift)
    z = w.sum()
    o = (w[:, None] * values).sum(axis=0) / z
    return o, (shift + math.log(z)) / LN2


def merge_state(o_a, b_a, o_b, b_b):
    """Merge two states over disjoint key sets (base-2 statistics).

    Empty states (zero vector, b = -inf) are the identity.  Otherwise take the
    larger statistic as the shift, form w = 2^(b - shift) for both, normalise
    the two scales before combining the vectors, and return shift + log2(w_a+w_b)."""
    o_a = np.asarray(o_a, dtype=np.float64)
    o_b = np.asarray(o_b, dtype=np.float64)
    if o_a.shape != o_b.shape or o_a.size == 0:
        raise ValueError("state vectors must have the same positive dimension")
    if not (np.all(np.isfinite(o_a)) and np.all(np.isfinite(o_b))):
        raise ValueError("state vectors must be finite")
    for o, b in ((o_a, b_a), (o_b, b_b)):
        if math.isnan(b) or b == math.inf:
            raise ValueError("lse must be finite or -inf")
        if b == -math.inf and np.any(o != 0):
            raise ValueError("an empty state must carry a zero vector")
    if b_a == -math.inf:
        return o_b.copy(), b_b
    if b_b == -math.inf:
        return o_a.copy(), b_a
    shift = max(b_a, b_b)
    w_a = 2.0 ** (b_a - shift)
    w_b = 2.0 ** (b_b - shift)
    z = w_a + w_b
    return (w_a / z) * o_a + (w_b / z) * o_b, shift + math.log2(z)


def merge_states(states):
    """Left fold of merge_state over a list of (o, b) states."""
    it = iter(states)
    o, b = next(it)
    o = np.asarray(o, dtype=np.float64)
    for o2, b2 in it:
        o, b = merge_state(o, b, o2, b2)
    return o, b


# ---------------------------------------------------------------------------
# Gather of logical K/V rows (paged NHD / HND, or ragged)
# ("KV-Cache layouts", "NHD/HND", "Ragged Tensor", "Page table layout")
# ---------------------------------------------------------------------------

def gather_request_kv(pool, *, layout, page_size, kv_indptr, kv_indices, req, kv_len,
                      kv_ragged=False):
    """Logical rows 0..kv_len-1 of request ``req`` as an array [kv_len, Hk, D].

    Paged: token j lives in page kv_indices[kv_indptr[r] + j // P], slot j % P;
    NHD pool [pages, P, Hk, D], HND pool [pages, Hk, P, D].  Ragged: row
    kv_indptr[r] + j of a [tokens, Hk, D] tensor."""
    if kv_ragged:
        base = int(kv_indptr[req])
        return np.stack([pool[base + j] for j in range(kv_len)]) if kv_len else pool[:0]
    page_ids = kv_indices[int(kv_indptr[req]):int(kv_indptr[req + 1])]
    rows = []
    for j in range(kv_len):
        page, slot = token_address(page_ids, j, page_size)
        rows.append(pool[page, slot] if layout == "NHD" else pool[page, :, slot])
    return np.stack(rows) if rows else np.zeros((0,) + pool.shape[-2:], pool.dtype)


def visible_keys(mode, i, qo_len, kv_len, packed_mask=None, mask_start=0):
    """Indices j of the keys query i (local) may see under the given mask mode."""
    if mode == "none":
        return list(range(kv_len))
    if mode == "causal":
        return [j for j in range(kv_len) if causal_visible(i, j, qo_len, kv_len)]
    if mode == "custom":
        return [j for j in range(kv_len) if mask_bit(packed_mask, mask_start + i * kv_len + j)]
    raise ValueError(mode)


# ---------------------------------------------------------------------------
# Batched attention: softmax(Q K^T * scale + mask) V per request and head
# ---------------------------------------------------------------------------

def batch_attention(q_bits, k_pool_bits, v_pool_bits, *, qo_indptr, kv_indptr, kv_indices,
                    last_page_len, page_size, num_qo_heads, num_kv_heads, layout="NHD",
                    mask_mode="causal", packed_mask=None, sm_scale=None, kv_ragged=False,
                    requests=None, kv_range=None, rows=None, kv_dtype="bf16", k_scale=1.0,
                    v_scale=1.0):
    """Reference output of one batch.

    Returns (o, lse2) as float64 arrays [nnz_q, Hq, D] and [nnz_q, Hq]; rows of
    requests not listed in ``requests`` stay NaN.  ``kv_range`` (t0, t1)
    restricts every request to logical keys t0 <= j < t1 (a split-KV chunk).
    ``rows`` (a set of global query rows) computes only those rows.
    ``kv_dtype`` "e4m3": the pools hold e4m3 codes standing for
    e4m3(code) * k_scale (K) and e4m3(code) * v_scale (V)."""
    q = bf16_bits_to_f64(q_bits)
    head_dim = q.shape[-1]
    if num_qo_heads % num_kv_heads:
        raise ValueError("num_qo_heads must be a multiple of num_kv_heads")
    group = num_qo_heads // num_kv_heads
    scale = (1.0 / math.sqrt(head_dim)) if not sm_scale else float(sm_scale)
    nreq = len(kv_indptr) - 1
    if kv_ragged:
        kv_lens = [int(kv_indptr[r + 1]) - int(kv_indptr[r]) for r in range(nreq)]
    else:
        kv_lens = kv_lens_from_csr(kv_indptr, kv_indices, last_page_len, page_size)
    qo_lens = [int(qo_indptr[r + 1]) - int(qo_indptr[r]) for r in range(nreq)]
    m_indptr = mask_indptr(qo_lens, kv_lens)
    o = np.full(q.shape, np.nan)
    lse = np.full(q.shape[:2], np.nan)
    for r in (range(nreq) if requests is None else requests):
        qlen, klen = qo_lens[r], kv_lens[r]
        if qlen == 0:
            continue
        if mask_mode == "causal" and klen < qlen:
            raise ValueError("causal attention needs kv_len >= qo_len")
        if rows is not None and not any(int(qo_indptr[r]) + i in rows for i in range(qlen)):
            continue
        kr = kv_payload_to_f64(gather_request_kv(
            k_pool_bits, layout=layout, page_size=page_size, kv_indptr=kv_indptr,
            kv_indices=kv_indices, req=r, kv_len=klen, kv_ragged=kv_ragged), kv_dtype, k_scale)
        vr = kv_payload_to_f64(gather_request_kv(
            v_pool_bits, layout=layout, page_size=page_size, kv_indptr=kv_indptr,
            kv_indices=kv_indices, req=r, kv_len=klen, kv_ragged=kv_ragged), kv_dtype, v_scale)
        for i in range(qlen):
            row = int(qo_indptr[r]) + i
            if rows is not None and row not in rows:
                continue
            keys = visible_keys(mask_mode, i, qlen, klen, packed_mask, m_indptr[r])
            if kv_range is not None:
                keys = [j for j in keys if kv_range[0] <= j < kv_range[1]]
            for h in range(num_qo_heads):
                kh = h // group
                if keys:
                    s = scale * (kr[keys, kh, :] @ q[row, h])
                    o[row, h], lse[row, h] = direct_state(s, vr[keys, kh, :])
                else:
                    o[row, h], lse[row, h] = np.zeros(head_dim), -math.inf
    return o, lse


# ---------------------------------------------------------------------------
# Multi-level cascade ("KV-Cache layouts", "Multi-level cascade inference data
# layout"; "Deep Dive - FlashInfer", "Core mechanism": the attention state is
# the unit that composes across shared prefixes)
# ---------------------------------------------------------------------------

def _node_of(qo_indptr, row: int) -> int:
    """Index n of the node whose query range [qo_indptr[n], qo_indptr[n+1]) holds ``row``."""
    for n in range(len(qo_indptr) - 1):
        if int(qo_indptr[n]) <= row < int(qo_indptr[n + 1]):
            return n
    raise ValueError(f"row {row} is in no node")


def _node_kv_len(level, n: int, page_size: int) -> int:
    pages = int(level["kv_indptr"][n + 1]) - int(level["kv_indptr"][n])
    if pages == 0:
        return 0  # a node without keys (shared levels only)
    return kv_len_from_pages(range(pages), int(level["last_page_len"][n]), page_size)


def cascade_attention(q_bits, k_pool_bits, v_pool_bits, *, levels, page_size, num_qo_heads,
                      num_kv_heads, layout="NHD", mask_mode="causal", sm_scale=None,
                      kv_dtype="bf16", k_scale=1.0, v_scale=1.0, rows=None):
    """Reference output of a multi-level cascade over one page pool.

    ``levels`` lists, from the root, dicts with the level's own qo_indptr,
    kv_indptr, kv_indices and last_page_len (the page-table semantics of every
    other call).  Every level splits the same query rows into nodes.  A row
    sees, at each level but the last, every key of the node holding it (a
    shared prefix lies wholly before the row's own tokens); at the last level
    the keys of its node that ``mask_mode`` leaves visible, with that node's
    (Q, K) and the row's index inside it.  The state is the softmax over the
    union of those key sets, taken in one pass: no merge.  A shared-level node
    may hold no pages.  ``kv_dtype`` "e4m3": the pool holds e4m3 codes read as
    in batch_attention (code times the pool's scale).  ``rows`` (a set of
    query rows) computes only those rows; the others stay NaN."""
    q = bf16_bits_to_f64(q_bits)
    nnz, _, head_dim = q.shape
    group = num_qo_heads // num_kv_heads
    scale = (1.0 / math.sqrt(head_dim)) if not sm_scale else float(sm_scale)
    last = len(levels) - 1
    for lv in levels:
        if int(lv["qo_indptr"][-1]) != nnz:
            raise ValueError("every level must cover all query rows")
    cache = {}

    def node_kv(li, n):
        if (li, n) not in cache:
            lv = levels[li]
            klen = _node_kv_len(lv, n, page_size)
            kv = [kv_payload_to_f64(gather_request_kv(
                pool, layout=layout, page_size=page_size, kv_indptr=lv["kv_indptr"],
                kv_indices=lv["kv_indices"], req=n, kv_len=klen), kv_dtype, scale_)
                  for pool, scale_ in ((k_pool_bits, k_scale), (v_pool_bits, v_scale))]
            cache[(li, n)] = (klen, kv[0], kv[1])
        return cache[(li, n)]

    o = np.full(q.shape, np.nan)
    lse = np.full(q.shape[:2], np.nan)
    for row in range(nnz):
        if rows is not None and row not in rows:
            continue
        ks, vs = [], []
        for li, lv in enumerate(levels):
            n = _node_of(lv["qo_indptr"], row)
            klen, kr, vr = node_kv(li, n)
            if li < last:
                keys = list(range(klen))
            else:
                qlen = int(lv["qo_indptr"][n + 1]) - int(lv["qo_indptr"][n])
                if mask_mode == "causal" and klen < qlen:
                    raise ValueError("causal attention needs kv_len >= qo_len at the last level")
                keys = visible_keys(mask_mode, row - int(lv["qo_indptr"][n]), qlen, klen)
            ks.append(kr[keys])
            vs.append(vr[keys])
        kc, vc = np.concatenate(ks), np.concatenate(vs)
        for h in range(num_qo_heads):
            kh = h // group
            if len(kc):
                o[row, h], lse[row, h] = direct_state(scale * (kc[:, kh, :] @ q[row, h]),
                                                      vc[:, kh, :])
            else:
                o[row, h], lse[row, h] = np.zeros(head_dim), -math.inf
    return o, lse


# ---------------------------------------------------------------------------
# append_paged_kv_cache: scatter new rows into pre-allocated pages
# ("KV-Cache layouts", "Page table layout", the append API note)
# ---------------------------------------------------------------------------

def append_paged_kv_cache(k_new, v_new, append_indptr, k_pool, v_pool, *, kv_indptr, kv_indices,
                          last_page_len, page_size, layout="NHD", kv_dtype="bf16", k_scale=1.0,
                          v_scale=1.0):
    """Return copies of the pools with the appended rows written.

    Request r appends rows append_indptr[r]..append_indptr[r+1]; its KV length
    (from the CSR page table) already counts them, so appended token t lands at
    logical position kv_len - n_append + t.  e4m3 pools receive each bf16 value
    divided by the pool's scale, rounded to e4m3 (quantize_kv_e4m3)."""
    if kv_dtype == "e4m3":
        k_new = quantize_kv_e4m3(k_new, k_scale)
        v_new = quantize_kv_e4m3(v_new, v_scale)
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    kv_lens = kv_lens_from_csr(kv_indptr, kv_indices, last_page_len, page_size)
    for r in range(len(kv_lens)):
        a0, a1 = int(append_indptr[r]), int(append_indptr[r + 1])
        pages = kv_indices[int(kv_indptr[r]):int(kv_indptr[r + 1])]
        for t in range(a1 - a0):
            pos = kv_lens[r] - (a1 - a0) + t
            if pos < 0:
                raise ValueError("more appended tokens than the request's KV length")
            page, slot = token_address(pages, pos, page_size)
            if layout == "NHD":
                k_out[page, slot] = k_new[a0 + t]
                v_out[page, slot] = v_new[a0 + t]
            else:
                k_out[page, :, slot] = k_new[a0 + t]
                v_out[page, :, slot] = v_new[a0 + t]
    return k_out, v_out
