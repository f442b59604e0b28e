// Host side of the C ABI: metadata validation, the planner (work partition,
// split-KV chunking, merge list) and the run / utility entry points.
//
// The planner follows "Deep Dive - FlashInfer", sections "Plan then run"
// (inspect the irregular metadata once per batch on the host, copy the work
// list to the device asynchronously, run a stable kernel per layer) and
// "Load balancing and split-KV decisions" (partition long key ranges across
// CTAs, merge their partial states).  The pages give no split threshold; the
// policy here is ours (plan_decode and plan_prefill below).
#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstdio>
#include <cstring>
#include <unordered_map>
#include <vector>

#include "pka_internal.h"

using pka::AttnArgs;

namespace pka {

// The planner's lists.  A plan object keeps them from one plan to the next:
// each plan clears them (the capacity stays), so steady-state planning does
// not allocate, which matters for a cascade's tens of thousands of merge slots.
struct PlanLists {
  std::vector<int32_t> dec_cta_ptr{0};
  std::vector<PkaWorkItem> dec_items;
  std::vector<int32_t> pre_cta_ptr{0};
  std::vector<PkaWorkItem> pre_items;
  std::vector<PkaMergeTask> merges;
  std::vector<PkaDecodeJoin> joins;  // split decode units, merged in the decode kernel
  int32_t records = 0;
  int32_t joined_pairs = 0;  // (row, qo head) pairs the decode kernel merges
  int32_t decode_chunk = 0;
  // Cascade: every piece writes partial records and each (row, head) merges
  // the records of all levels, listed in merge_slots.
  bool cascade = false;
  struct Slot { int32_t row, head, rec; };
  std::vector<Slot> slots;
  std::vector<int32_t> merge_slots;
  // e4m3 K/V: requests whose keys are decoded to bf16 for the tensor-core rows
  std::vector<PkaDequantUnit> dequant;
  std::unordered_map<int32_t, int32_t> dequant_row0;  // node page-list start -> first scratch row
  int64_t dequant_rows = 0;

  void reset(bool is_cascade) {
    dec_cta_ptr.assign(1, 0);
    dec_items.clear();
    pre_cta_ptr.assign(1, 0);
    pre_items.clear();
    merges.clear();
    joins.clear();
    records = joined_pairs = decode_chunk = 0;
    cascade = is_cascade;
    slots.clear();
    merge_slots.clear();
    dequant.clear();
    dequant_rows = 0;
  }
};

}  // namespace pka

using pka::PlanLists;

struct pka_plan_s {
  pka_params params{};
  bool planned = false;
  pka_plan_info info{};
  PkaImageHeader hdr{};
  int32_t* int_ws_d = nullptr;
  cudaEvent_t event = nullptr;
  bool copy_pending = false;
  int device = -1;
  int32_t layout_records = 0;  // partial records the float workspace is laid out for
  int32_t merge_capacity = 0;  // graph mode: merge tasks the image has room for
  int32_t dequant_capacity = 0;      // graph mode: dequant units the image has room for
  int64_t scratch_capacity = 0;      // rows the float workspace's bf16 K/V scratch is laid out for
  PlanLists lists;             // the planner's lists, reused by every plan
  pka::MapCache decode_maps{};   // tensor maps of the last run's launches
  pka::MapCache prefill_maps{};
};

namespace {

constexpr int kMinDecodeChunk = 64;

thread_local char g_last_error[256] = "";

pka_status cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(e),
                (int)e);
  return PKA_ERR_CUDA;
}

bool params_ok(const pka_params* p) {
  if (!p) return false;
  if (p->reserved[0] != 0) return false;
  if (p->decode_on_tensor_cores != 0 && p->decode_on_tensor_cores != 1) return false;
  if (p->graph_max_batch < 0 || p->graph_max_qo_rows < 0 || p->graph_max_kv_tokens < 0)
    return false;
  if (p->graph_max_batch == 0 && (p->graph_max_qo_rows || p->graph_max_kv_tokens)) return false;
  if (p->graph_max_batch > 0 && p->graph_max_qo_rows < 1) return false;
  if (p->graph_max_batch > 0 && p->kv_ragged && p->graph_max_kv_tokens < 1) return false;
  if (p->num_qo_heads < 1 || p->num_kv_heads < 1) return false;
  if (p->layout != PKA_NHD && p->layout != PKA_HND) return false;
  if (p->mask_mode < PKA_MASK_NONE || p->mask_mode > PKA_MASK_CUSTOM) return false;
  if (p->split_mode < PKA_SPLIT_OFF || p->split_mode > PKA_SPLIT_FIXED) return false;
  if (p->split_mode == PKA_SPLIT_FIXED && p->fixed_split_pages < 1) return false;
  if (!p->kv_ragged && p->page_size < 1) return false;
  if (p->num_sms < 0) return false;
  if (p->kv_dtype != PKA_KV_BF16 && p->kv_dtype != PKA_KV_FP8_E4M3) return false;
  if (!std::isfinite(p->k_scale) || !std::isfinite(p->v_scale)) return false;
  return true;
}


pka_status check_supported(const pka_params* p) {
  if (p->num_qo_heads % p->num_kv_heads) return PKA_ERR_UNSUPPORTED;
  int g = p->num_qo_heads / p->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return PKA_ERR_UNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 128) return PKA_ERR_UNSUPPORTED;
  if (p->graph_max_batch > 0 && p->split_mode == PKA_SPLIT_FIXED) return PKA_ERR_UNSUPPORTED;
  return PKA_OK;
}

bool graph_mode(const pka_params* p) { return p->graph_max_batch > 0; }

// Graph mode: section capacities of the plan image, from the declared limits.
// Decode: units (request, head block) <= B * Hk / hpc; the AUTO split closes a
// CTA only once it holds more than chunk - 16 >= 3/4 chunk keys, so it makes
// at most 4/3 * num_sms + 2 CTAs and every item either ends a unit or closes
// a CTA.  Tensor-core rows are not split in graph mode: one item per
// (request, kv head, query tile) and sum_r ceil(Q_r / tq) <= ceil(R / tq) + B.
struct GraphCaps {
  int64_t dec_items = 0, pre_items = 0, merges = 0, records = 0, joins = 0;
  int64_t dequant_units = 0, dequant_rows = 0;  // e4m3 K/V: bf16 scratch of tensor-core rows
};

GraphCaps graph_caps(const pka_params* p, int num_sms) {
  GraphCaps c;
  const int64_t B = p->graph_max_batch, R = p->graph_max_qo_rows;
  const int g = p->num_qo_heads / p->num_kv_heads;
  const int hpc = pka::decode_heads_per_cta(p->num_kv_heads, g);
  const int tq = 2 * (pka::kPrefillTileRows / g);
  c.dec_items = B * (p->num_kv_heads / hpc) + 2 * (int64_t)num_sms + 2;
  c.pre_items = (int64_t)p->num_kv_heads * ((R + tq - 1) / tq + B);
  if (p->split_mode == PKA_SPLIT_AUTO) {
    // split decode rows are merged inside the decode kernel (one join per
    // split (request, kv head)); no merge tasks are left for the merge kernel
    c.joins = B * p->num_kv_heads;
    c.records = c.dec_items * hpc * g;
  }
  if (p->kv_dtype == PKA_KV_FP8_E4M3 && p->graph_max_kv_tokens > 0) {
    // one unit per request with qo_len >= 2; its keys count against the
    // declared K/V token capacity
    c.dequant_units = B;
    c.dequant_rows = p->graph_max_kv_tokens;
  }
  return c;
}

struct Batch {
  std::vector<int32_t> qo_len, kv_len, q_row0, kv_base;
  std::vector<int64_t> mask_base;
  int64_t total_kv = 0;
  int32_t nnz_q = 0;
  int mask_mode = PKA_MASK_NONE;  // the mask this batch (or cascade level) applies
  int32_t item_flags = 0;         // PkaWorkItem.flags of its items
};

// Length contract of "Why inference attention becomes irregular" and the
// "Page table layout" section: K = P * (pages - 1) + last, 1 <= last <= P.
// A cascade level above the last (`shared`) may hold nodes without pages; its
// page ids sit at kv_off in the concatenated index array.
pka_status derive(const pka_params* p, int32_t batch, const int32_t* qo, const int32_t* kv,
                  const int32_t* last, Batch* b, int mask_mode, bool shared = false,
                  int64_t kv_off = 0) {
  b->mask_mode = mask_mode;
  if (batch < 0 || !kv || (!p->kv_ragged && !last)) return PKA_ERR_INVALID_ARG;
  if (kv[0] != 0) return PKA_ERR_METADATA;
  if (qo && qo[0] != 0) return PKA_ERR_METADATA;
  b->qo_len.resize(batch);
  b->kv_len.resize(batch);
  b->q_row0.resize(batch);
  b->kv_base.resize(batch);
  b->mask_base.resize(batch + 1);
  b->mask_base[0] = 0;
  int64_t rows = 0;
  for (int32_t r = 0; r < batch; ++r) {
    int64_t npages = (int64_t)kv[r + 1] - kv[r];
    if (npages < 0) return PKA_ERR_METADATA;
    int64_t klen;
    if (p->kv_ragged) {
      klen = npages;
    } else if (npages == 0 && shared) {
      klen = 0;
    } else {
      if (npages < 1) return PKA_ERR_METADATA;
      if (last[r] < 1 || last[r] > p->page_size) return PKA_ERR_METADATA;
      klen = (int64_t)p->page_size * (npages - 1) + last[r];
    }
    if (klen > INT32_MAX) return PKA_ERR_UNSUPPORTED;
    int64_t qlen = qo ? (int64_t)qo[r + 1] - qo[r] : 1;
    if (qlen < 0) return PKA_ERR_METADATA;
    if (mask_mode == PKA_MASK_CAUSAL && klen < qlen) return PKA_ERR_METADATA;
    if (kv_off + kv[r] > INT32_MAX) return PKA_ERR_UNSUPPORTED;
    b->qo_len[r] = (int32_t)qlen;
    b->kv_len[r] = (int32_t)klen;
    b->q_row0[r] = (int32_t)(qo ? qo[r] : r);
    b->kv_base[r] = (int32_t)(kv_off + kv[r]);
    b->total_kv += klen;
    rows += qlen;
    if (rows > INT32_MAX) return PKA_ERR_UNSUPPORTED;
    b->mask_base[r + 1] = b->mask_base[r] + qlen * klen;
  }
  b->nnz_q = (int32_t)rows;
  return PKA_OK;
}

// e4m3 K/V: decode rows read the codes; rows with qo_len >= 2 read a bf16
// scratch decoded in run(), whose size depends on the batch: graph mode
// (fixed workspaces) sizes it by graph_max_kv_tokens and refuses such rows
// when that capacity is not declared.
pka_status check_kv_dtype(const pka_params* p, const Batch& b) {
  if (p->kv_dtype != PKA_KV_FP8_E4M3 || !graph_mode(p) || p->graph_max_kv_tokens > 0)
    return PKA_OK;
  const int32_t tc_rows = p->decode_on_tensor_cores ? 1 : 2;  // rows the tensor-core kernel takes
  for (int32_t q : b.qo_len)
    if (q >= tc_rows) {
      pka::set_last_error("graph mode over e4m3 pools with qo_len >= 2 rows needs graph_max_kv_tokens");
      return PKA_ERR_UNSUPPORTED;
    }
  return PKA_OK;
}

// e4m3 K/V: one dequant unit per request (or cascade node) that tensor-core
// items read, identified by its page-list start kv_base (distinct for every
// node with pages), its scratch rows back to back in the order the items meet
// them; the items' kv_base is rewritten to the node's first scratch row (the
// kernel then reads the scratch as ragged K/V).
void plan_dequant(PlanLists* L) {
  L->dequant_row0.clear();
  for (PkaWorkItem& w : L->pre_items) {
    auto it = L->dequant_row0.find(w.kv_base);
    if (it == L->dequant_row0.end()) {
      it = L->dequant_row0.emplace(w.kv_base, (int32_t)L->dequant_rows).first;
      L->dequant.push_back({w.kv_base, w.kv_len, (int32_t)L->dequant_rows, 0});
      L->dequant_rows += w.kv_len;
    }
    w.kv_base = it->second;
  }
}

PkaWorkItem make_item(const Batch& b, int r, int kv_head0, int n_kv_heads, int q_local0,
                      int q_count, int t0, int t1) {
  PkaWorkItem it{};
  it.req = r;
  it.kv_head0 = kv_head0;
  it.n_kv_heads = n_kv_heads;
  it.q_row0 = b.q_row0[r] + q_local0;
  it.q_local0 = q_local0;
  it.q_count = q_count;
  it.qo_len = b.qo_len[r];
  it.kv_len = b.kv_len[r];
  it.kv_base = b.kv_base[r];
  it.t0 = t0;
  it.t1 = t1;
  it.out_rec = -1;
  it.mask_lo = (int32_t)(uint32_t)(b.mask_base[r] & 0xffffffffu);
  it.mask_hi = (int32_t)(b.mask_base[r] >> 32);
  it.flags = b.item_flags;
  it.join = -1;
  return it;
}

// Give the pieces of one split unit their partial records and merge tasks.
// `pieces` index into `items`; each piece writes q_count * heads records laid
// out [token][qo head]; the heads are heads_total qo heads starting at head0.
// With join_kv_heads > 0 (decode pieces outside a cascade) the unit gets one
// PkaDecodeJoin per kv head instead of merge tasks: the decode kernel merges
// the pieces itself, the last piece to finish doing the work.
void assign_records(PlanLists* L, std::vector<PkaWorkItem>& items,
                    const std::vector<int>& pieces, int q_row0, int q_count, int head0,
                    int heads_total, int join_kv_heads = 0) {
  if (pieces.size() < 2 && !L->cascade) return;
  int per = q_count * heads_total;
  int base = L->records;
  for (size_t k = 0; k < pieces.size(); ++k) items[pieces[k]].out_rec = base + (int)k * per;
  L->records += (int)pieces.size() * per;
  if (join_kv_heads > 0 && !L->cascade) {
    const int g = heads_total / join_kv_heads;
    const int j0 = (int)L->joins.size();
    L->joins.resize((size_t)j0 + join_kv_heads);
    PkaDecodeJoin* jo = L->joins.data() + j0;
    for (int hl = 0; hl < join_kv_heads; ++hl) {
      jo[hl] = PkaDecodeJoin{};
      jo[hl].rec_first = base + hl * g;
      jo[hl].nslots = (int)pieces.size();
      jo[hl].rec_stride = per;
    }
    for (int k : pieces) items[k].join = j0;
    L->joined_pairs += q_count * heads_total;
    return;
  }
  if (L->cascade) {
    // filled through a pointer: a push_back per slot through L measured 5x slower
    const size_t at = L->slots.size();
    L->slots.resize(at + pieces.size() * (size_t)per);
    PlanLists::Slot* o = L->slots.data() + at;
    for (size_t k = 0; k < pieces.size(); ++k)
      for (int i = 0; i < q_count; ++i)
        for (int h = 0; h < heads_total; ++h)
          *o++ = {q_row0 + i, head0 + h, base + (int)k * per + i * heads_total + h};
    return;
  }
  for (int i = 0; i < q_count; ++i)
    for (int h = 0; h < heads_total; ++h) {
      PkaMergeTask t{};
      t.out_row = q_row0 + i;
      t.head = head0 + h;
      t.rec_first = base + i * heads_total + h;
      t.nslots = (int)pieces.size();
      t.rec_stride = per;
      L->merges.push_back(t);
    }
}

// Cascade: one merge task per (row, head) over the records of every level,
// listed contiguously in merge_slots (a counting sort by row and head).
void build_slot_merges(PlanLists* L, int32_t nnz, int32_t heads) {
  const int64_t keys = (int64_t)nnz * heads;
  const size_t n = L->slots.size();
  const PlanLists::Slot* sl = L->slots.data();
  std::vector<int32_t> start(keys + 1, 0);
  int32_t* st = start.data();
  for (size_t i = 0; i < n; ++i) ++st[(int64_t)sl[i].row * heads + sl[i].head + 1];
  int64_t used = 0;  // (row, head) pairs with at least one record
  for (int64_t k = 0; k < keys; ++k) {
    used += st[k + 1] > 0;
    st[k + 1] += st[k];
  }
  L->merge_slots.resize(n);
  int32_t* out = L->merge_slots.data();
  std::vector<int32_t> pos(start.begin(), start.end() - 1);
  int32_t* ps = pos.data();
  for (size_t i = 0; i < n; ++i) out[ps[(int64_t)sl[i].row * heads + sl[i].head]++] = sl[i].rec;
  const size_t m0 = L->merges.size();
  L->merges.resize(m0 + (size_t)used);
  PkaMergeTask* t = L->merges.data() + m0;
  for (int64_t k = 0; k < keys; ++k) {
    if (st[k + 1] == st[k]) continue;
    *t = PkaMergeTask{};
    t->out_row = (int32_t)(k / heads);
    t->head = (int32_t)(k % heads);
    t->rec_first = st[k];
    t->nslots = st[k + 1] - st[k];
    t->rec_stride = 0;  // list mode
    ++t;
  }
}

// Order the items inside each decode CTA so that few split units have more
// than one piece finishing at the end of the kernel.  The last of a unit's
// pieces to finish merges them all: when it runs last in its CTA while
// another piece of the unit also runs last in its own CTA, both finish
// together, neither sees the other done in advance, and the merge takes the
// slow path (fence, count, then the merge) right at the end.  A piece that
// fills a whole CTA always ends last; among the other split pieces, those of
// a CTA that also holds whole units go first, and a CTA with just two split
// pieces runs last the one whose unit has no piece ending last yet (walking
// the CTAs in order).
void order_split_pieces(PlanLists* L) {
  auto& items = L->dec_items;
  const auto& ptr = L->dec_cta_ptr;
  if (L->joins.empty()) return;
  std::vector<int> ends(L->joins.size(), 0);  // pieces ending last, by the unit's first join
  const int ctas = (int)ptr.size() - 1;
  for (int c = 0; c < ctas; ++c)
    if (ptr[c + 1] - ptr[c] == 1 && items[ptr[c]].join >= 0) ++ends[items[ptr[c]].join];
  std::vector<PkaWorkItem> split, whole;
  for (int c = 0; c < ctas; ++c) {
    const int b = ptr[c], e = ptr[c + 1];
    if (e - b < 2) continue;
    split.clear();
    whole.clear();
    for (int i = b; i < e; ++i) (items[i].join >= 0 ? split : whole).push_back(items[i]);
    if (split.empty()) continue;
    if (!whole.empty()) {
      int i = b;
      for (const auto& it : split) items[i++] = it;
      for (const auto& it : whole) items[i++] = it;
      continue;
    }
    if (split.size() != 2) continue;
    // split[0] continues a unit from the previous CTA, split[1] goes on in the
    // next: run split[0] last unless its unit already has a piece ending last
    const int u = split[0].join, v = split[1].join;
    if (ends[u] == 0) {
      items[b] = split[1];
      items[b + 1] = split[0];
      ++ends[u];
    } else {
      ++ends[v];
    }
  }
}

// Decode rows (qo_len == 1): units are (request, block of kv heads); with
// split AUTO the keys of all units are dealt out in equal shares to one
// persistent CTA per SM (a unit may span CTAs, a CTA may hold several units).
// The units of every cascade level go into one list (a plain batch is one level).
void plan_decode(const pka_params* p, const std::vector<Batch>& lv, int num_sms, PlanLists* L) {
  int g = p->num_qo_heads / p->num_kv_heads;
  int hpc = pka::decode_heads_per_cta(p->num_kv_heads, g);
  int hg_count = p->num_kv_heads / hpc;
  struct Unit { int l, r, hg, K; };
  std::vector<Unit> units;
  int64_t total = 0;
  for (int l = 0; l < (int)lv.size(); ++l) {
    const Batch& b = lv[l];
    for (int r = 0; r < (int)b.qo_len.size(); ++r) {
      if (b.qo_len[r] != 1 || p->decode_on_tensor_cores) continue;
      if (L->cascade && b.kv_len[r] == 0) continue;  // an empty node adds no state
      for (int hg = 0; hg < hg_count; ++hg) {
        units.push_back({l, r, hg, b.kv_len[r]});
        total += b.kv_len[r];
      }
    }
  }
  if (units.empty()) return;
  int64_t chunk = 0;
  if (p->split_mode == PKA_SPLIT_FIXED) {
    chunk = (int64_t)p->fixed_split_pages * (p->kv_ragged ? 1 : p->page_size);
  } else if (p->split_mode == PKA_SPLIT_AUTO) {
    int64_t target = (total + num_sms - 1) / num_sms;
    target = (target + pka::kDecodeTileTokens - 1) / pka::kDecodeTileTokens * pka::kDecodeTileTokens;
    chunk = std::max<int64_t>(target, kMinDecodeChunk);
  }
  L->decode_chunk = (int)chunk;
  auto& items = L->dec_items;
  std::vector<int> pieces;  // items of the current unit (reused: the planner runs every step)
  pieces.reserve(64);
  if (p->split_mode != PKA_SPLIT_AUTO) {
    // one CTA per piece
    for (const Unit& u : units) {
      pieces.clear();
      int64_t step = chunk > 0 ? chunk : std::max(u.K, 1);
      int64_t t = 0;
      do {
        int64_t t1 = std::min<int64_t>(u.K, t + step);
        pieces.push_back((int)items.size());
        items.push_back(make_item(lv[u.l], u.r, u.hg * hpc, hpc, 0, 1, (int)t, (int)t1));
        L->dec_cta_ptr.push_back((int)items.size());
        t = t1;
      } while (t < u.K);
      assign_records(L, items, pieces, lv[u.l].q_row0[u.r], 1, u.hg * hpc * g, hpc * g, hpc);
    }
    return;
  }
  items.reserve(units.size() + 2 * (size_t)num_sms + 2);
  L->dec_cta_ptr.reserve(2 * (size_t)num_sms + 2);
  L->joins.reserve(units.size() * hpc);
  int64_t load = 0;
  for (const Unit& u : units) {
    pieces.clear();
    int64_t t = 0;
    do {
      // Cuts inside a request fall on 16-key tile boundaries, so that whole
      // pages stay in one tile of the decode kernel.
      int64_t take = u.K - t;
      if (take > chunk - load) {
        take = (chunk - load) / pka::kDecodeTileTokens * pka::kDecodeTileTokens;
        if (take == 0) {  // no room for a whole tile: close this CTA
          L->dec_cta_ptr.push_back((int)items.size());
          load = 0;
          continue;
        }
      }
      pieces.push_back((int)items.size());
      items.push_back(make_item(lv[u.l], u.r, u.hg * hpc, hpc, 0, 1, (int)t, (int)(t + take)));
      t += take;
      load += take;
      if (load >= chunk) {
        L->dec_cta_ptr.push_back((int)items.size());
        load = 0;
      }
    } while (t < u.K);
    assign_records(L, items, pieces, lv[u.l].q_row0[u.r], 1, u.hg * hpc * g, hpc * g, hpc);
  }
  if (L->dec_cta_ptr.back() != (int)items.size()) L->dec_cta_ptr.push_back((int)items.size());
  order_split_pieces(L);
}

// Greedy dealing (longest first onto the least loaded CTA): for each index in
// `order`, the CTA with the smallest (load, CTA id) takes it.  A min-heap of
// (load, id) pairs with one sift-down per deal (the pairs are distinct, so the
// choice is the same as with any priority queue).  Fills cta_of.
void deal_least_loaded(const std::vector<int>& order, const std::vector<int64_t>& cost, int ctas,
                       std::vector<int>& cta_of) {
  using Slot = std::pair<int64_t, int>;
  std::vector<Slot> hp(ctas);
  for (int c = 0; c < ctas; ++c) hp[c] = {0, c};  // ascending ids: already a min-heap
  const size_t m = hp.size();
  for (int i : order) {
    const Slot v{hp[0].first + cost[i], hp[0].second};
    cta_of[i] = hp[0].second;
    size_t k = 0;
    for (;;) {
      size_t c = 2 * k + 1;
      if (c >= m) break;
      if (c + 1 < m && hp[c + 1] < hp[c]) ++c;
      if (!(hp[c] < v)) break;
      hp[k] = hp[c];
      k = c;
    }
    hp[k] = v;
  }
}

// Rows of requests with qo_len >= 2 go to the tensor-core kernel: units are
// (request, kv head, 2 x 128 / g query tokens): the g qo heads of one kv head
// pack with the tokens into two 128-row tiles that share every K/V load.  Causal
// units only visit keys up to the tile's last visible one.  Items are dealt
// to CTAs longest-first onto the least loaded CTA.
void plan_prefill(const pka_params* p, const std::vector<Batch>& lv, int num_sms, PlanLists* L) {
  int g = p->num_qo_heads / p->num_kv_heads;
  int tq = 2 * (pka::kPrefillTileRows / g);
  struct Unit { int l, r, h, q0, qc, kend; };
  std::vector<Unit> units;
  int64_t total_tiles = 0;
  for (int l = 0; l < (int)lv.size(); ++l) {
    const Batch& b = lv[l];
    for (int r = 0; r < (int)b.qo_len.size(); ++r) {
      int Q = b.qo_len[r], K = b.kv_len[r];
      if (Q < (p->decode_on_tensor_cores ? 1 : 2)) continue;
      if (L->cascade && K == 0) continue;  // an empty node adds no state
      for (int h = 0; h < p->num_kv_heads; ++h)
        for (int q0 = 0; q0 < Q; q0 += tq) {
          int qc = std::min(tq, Q - q0);
          int kend = K;
          if (b.mask_mode == PKA_MASK_CAUSAL) kend = K - Q + (q0 + qc - 1) + 1;
          units.push_back({l, r, h, q0, qc, kend});
          total_tiles += (kend + pka::kPrefillTileKeys - 1) / pka::kPrefillTileKeys;
        }
    }
  }
  if (units.empty()) return;
  int64_t chunk = 0;  // keys per piece, 0 = whole range
  if (p->split_mode == PKA_SPLIT_FIXED) {
    chunk = (int64_t)p->fixed_split_pages * (p->kv_ragged ? 1 : p->page_size);
  } else if (p->split_mode == PKA_SPLIT_AUTO && !graph_mode(p) &&
             (int64_t)units.size() < 2 * num_sms) {
    int64_t per_cta = std::max<int64_t>(4, (total_tiles + num_sms - 1) / num_sms);
    chunk = per_cta * pka::kPrefillTileKeys;
  }
  auto& items = L->pre_items;
  std::vector<int64_t> cost;
  cost.reserve(units.size());
  items.reserve(units.size());
  std::vector<int> pieces;  // items of the current unit (reused)
  for (const Unit& u : units) {
    pieces.clear();
    int64_t step = chunk > 0 ? chunk : std::max(u.kend, 1);
    int64_t t = 0;
    do {
      int64_t t1 = std::min<int64_t>(u.kend, t + step);
      pieces.push_back((int)items.size());
      items.push_back(make_item(lv[u.l], u.r, u.h, 1, u.q0, u.qc, (int)t, (int)t1));
      cost.push_back((t1 - t) + 64);
      t = t1;
    } while (t < u.kend);
    assign_records(L, items, pieces, lv[u.l].q_row0[u.r] + u.q0, u.qc, u.h * g, g);
  }
  int n = (int)items.size();
  int ctas = std::min(n, num_sms);
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int a, int c) { return cost[a] > cost[c]; });
  // The CTA of each item; then the items grouped by CTA, each CTA's in
  // dealing order (a counting sort).
  std::vector<int> cta_of(n), start(ctas + 1, 0);
  deal_least_loaded(order, cost, ctas, cta_of);
  for (int i = 0; i < n; ++i) ++start[cta_of[i] + 1];
  for (int c = 0; c < ctas; ++c) start[c + 1] += start[c];
  std::vector<PkaWorkItem> sorted(n);
  std::vector<int> pos(start.begin(), start.end() - 1);
  for (int i : order) sorted[pos[cta_of[i]]++] = items[i];
  for (int c = 0; c < ctas; ++c) L->pre_cta_ptr.push_back(start[c + 1]);
  items.swap(sorted);
}

// Graph mode: deal the planner's CTAs onto exactly `ctas` CTAs, heaviest
// first onto the least loaded one, so that the grid never changes.
void fold_ctas(std::vector<int32_t>& cta_ptr, std::vector<PkaWorkItem>& items, int ctas) {
  const int n = (int)cta_ptr.size() - 1;
  if (n <= ctas) {
    cta_ptr.resize(ctas + 1, cta_ptr.back());
    return;
  }
  std::vector<int64_t> cost(n, 0);
  for (int c = 0; c < n; ++c)
    for (int i = cta_ptr[c]; i < cta_ptr[c + 1]; ++i) cost[c] += (items[i].t1 - items[i].t0) + 64;
  std::vector<int> order(n);
  for (int c = 0; c < n; ++c) order[c] = c;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return cost[x] > cost[y]; });
  std::vector<int> cta_of(n);
  deal_least_loaded(order, cost, ctas, cta_of);
  std::vector<std::vector<int>> per(ctas);
  for (int c : order) per[cta_of[c]].push_back(c);
  std::vector<PkaWorkItem> sorted;
  sorted.reserve(items.size());
  std::vector<int32_t> ptr{0};
  for (int c = 0; c < ctas; ++c) {
    for (int v : per[c])
      for (int i = cta_ptr[v]; i < cta_ptr[v + 1]; ++i) sorted.push_back(items[i]);
    ptr.push_back((int32_t)sorted.size());
  }
  items.swap(sorted);
  cta_ptr.swap(ptr);
}

size_t align_words(size_t w) { return (w + 15) & ~size_t(15); }

// Bytes of one bf16 K (or V) scratch of `rows` rows [rows, Hk, D], rounded
// up to 256.
size_t kv_scratch_bytes(const pka_params* p, int64_t rows) {
  const size_t b = (size_t)rows * p->num_kv_heads * p->head_dim * 2;
  return (b + 255) & ~size_t(255);
}

}  // namespace

void pka::set_last_error(const char* msg) {
  std::snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
}

pka_status pka::cuda_failure(cudaError_t e, const char* where) { return cuda_fail(e, where); }

namespace {

// Plan the levels (one for a plain batch) into the image and start its copy.
pka_status plan_levels(pka_plan_t plan, const pka_params* p, const std::vector<Batch>& lv,
                       int32_t batch, bool cascade, void* int_ws_d, size_t int_ws_bytes,
                       void* pinned_h, size_t pinned_bytes, void* stream) {
  const int32_t nnz = lv.back().nnz_q;
  int64_t total_kv = 0;
  for (const Batch& b : lv) total_kv += b.total_kv;
  int num_sms = p->num_sms;
  if (num_sms == 0) {
    if (int_ws_d) {
      int dev = 0;
      cudaError_t e = cudaGetDevice(&dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return cuda_fail(e, "device query");
    } else {
      num_sms = 152;
    }
  }

  const bool graph = graph_mode(p);
  if (graph && (batch > p->graph_max_batch || nnz > p->graph_max_qo_rows ||
                (p->kv_ragged && total_kv > p->graph_max_kv_tokens))) {
    pka::set_last_error("batch exceeds the graph-mode capacities");
    return PKA_ERR_WORKSPACE;
  }

  PlanLists& L = plan->lists;
  L.reset(cascade);
  plan_decode(p, lv, num_sms, &L);
  plan_prefill(p, lv, num_sms, &L);
  if (cascade) build_slot_merges(&L, nnz, p->num_qo_heads);
  if (p->kv_dtype == PKA_KV_FP8_E4M3 && !L.pre_items.empty()) plan_dequant(&L);
  if (L.dequant_rows > INT32_MAX) return PKA_ERR_UNSUPPORTED;
  GraphCaps caps;
  if (graph) {
    caps = graph_caps(p, num_sms);
    fold_ctas(L.dec_cta_ptr, L.dec_items, num_sms);
    fold_ctas(L.pre_cta_ptr, L.pre_items, num_sms);
    if ((int64_t)L.dec_items.size() > caps.dec_items ||
        (int64_t)L.pre_items.size() > caps.pre_items || (int64_t)L.merges.size() > caps.merges ||
        L.records > caps.records || (int64_t)L.joins.size() > caps.joins ||
        (int64_t)L.dequant.size() > caps.dequant_units || L.dequant_rows > caps.dequant_rows) {
      pka::set_last_error("plan outgrew the graph-mode image capacities");
      return PKA_ERR_WORKSPACE;
    }
  }
  // Section sizes: what this plan holds, or the fixed capacities in graph mode.
  const int64_t n_dec_ptr = (int64_t)L.dec_cta_ptr.size(), n_pre_ptr = (int64_t)L.pre_cta_ptr.size();
  const int64_t n_dec = graph ? caps.dec_items : (int64_t)L.dec_items.size();
  const int64_t n_pre = graph ? caps.pre_items : (int64_t)L.pre_items.size();
  const int64_t n_merge = graph ? caps.merges : (int64_t)L.merges.size();
  const int64_t n_join = graph ? caps.joins : (int64_t)L.joins.size();
  const int64_t n_dequant = graph ? caps.dequant_units : (int64_t)L.dequant.size();
  const int64_t scratch_rows = graph ? caps.dequant_rows : L.dequant_rows;
  const int64_t layout_records = graph ? caps.records : L.records;

  PkaImageHeader h{};
  h.magic = PKA_IMAGE_MAGIC;
  h.num_decode_ctas = (int)L.dec_cta_ptr.size() - 1;
  h.num_decode_items = (int)L.dec_items.size();
  h.num_prefill_ctas = (int)L.pre_cta_ptr.size() - 1;
  h.num_prefill_items = (int)L.pre_items.size();
  h.num_merge_tasks = (int)L.merges.size();
  h.num_partial_records = L.records;
  h.num_decode_joins = (int)L.joins.size();
  h.decode_heads_per_cta =
      pka::decode_heads_per_cta(p->num_kv_heads, p->num_qo_heads / p->num_kv_heads);
  h.graph_mode = graph ? 1 : 0;
  constexpr size_t kItemWords = sizeof(PkaWorkItem) / 4, kMergeWords = sizeof(PkaMergeTask) / 4;
  size_t w = align_words(sizeof(PkaImageHeader) / 4);
  h.off_decode_cta_ptr = (int)w;
  w = align_words(w + n_dec_ptr);
  h.off_decode_items = (int)w;
  w = align_words(w + n_dec * kItemWords);
  h.off_prefill_cta_ptr = (int)w;
  w = align_words(w + n_pre_ptr);
  h.off_prefill_items = (int)w;
  w = align_words(w + n_pre * kItemWords);
  h.off_merge_tasks = (int)w;
  w = align_words(w + n_merge * kMergeWords);
  h.off_merge_slots = L.merge_slots.empty() ? 0 : (int)w;
  w = align_words(w + L.merge_slots.size());
  constexpr size_t kJoinWords = sizeof(PkaDecodeJoin) / 4;
  h.off_decode_joins = n_join > 0 ? (int)w : 0;
  w = align_words(w + n_join * kJoinWords);
  constexpr size_t kDequantWords = sizeof(PkaDequantUnit) / 4;
  h.num_dequant_units = (int)L.dequant.size();
  h.off_dequant_units = n_dequant > 0 ? (int)w : 0;
  h.dequant_rows = (int)L.dequant_rows;
  w = align_words(w + n_dequant * kDequantWords);
  if (w > (size_t)INT32_MAX || layout_records > INT32_MAX / 256) {
    pka::set_last_error("plan image or partial records exceed 2^31");
    return PKA_ERR_UNSUPPORTED;
  }
  h.total_words = (int)w;

  pka_plan_info info{};
  info.int_ws_bytes = (uint64_t)w * 4;
  size_t rec_o = (size_t)layout_records * p->head_dim * 4;
  size_t rec_o_al = (rec_o + 255) & ~size_t(255);
  info.float_ws_bytes =
      layout_records ? rec_o_al + (((size_t)layout_records * 4 + 255) & ~size_t(255)) : 0;
  // e4m3 K/V: the bf16 K and V scratch follow the partial states
  info.float_ws_bytes += 2 * kv_scratch_bytes(p, scratch_rows);
  info.kv_scratch_rows = (int32_t)L.dequant_rows;
  info.num_requests = batch;
  info.nnz_qo = nnz;
  info.total_kv = total_kv;
  info.num_decode_ctas = h.num_decode_ctas;
  info.num_decode_items = h.num_decode_items;
  info.num_prefill_ctas = h.num_prefill_ctas;
  info.num_prefill_items = h.num_prefill_items;
  info.num_merge_tasks = h.num_merge_tasks + L.joined_pairs;
  info.num_decode_joins = h.num_decode_joins;
  info.num_partial_records = L.records;
  info.decode_chunk_tokens = L.decode_chunk;
  plan->info = info;
  if (!pinned_h || pinned_bytes < info.int_ws_bytes) return PKA_ERR_WORKSPACE;
  if (int_ws_d && int_ws_bytes < info.int_ws_bytes) return PKA_ERR_WORKSPACE;

  // The pinned buffer may still feed a previous copy of this plan object.
  if (plan->copy_pending && plan->event) {
    if (cudaEventSynchronize(plan->event) != cudaSuccess) return PKA_ERR_CUDA;
    plan->copy_pending = false;
  }
  // Word ranges of the image that carry this plan: all of it, or in graph mode
  // the used head of each fixed-size section (the kernels read no further).
  std::vector<std::pair<size_t, size_t>> ranges;
  if (graph) {
    ranges.push_back({0, h.off_decode_items + L.dec_items.size() * kItemWords});
    ranges.push_back({(size_t)h.off_prefill_cta_ptr,
                      h.off_prefill_items + L.pre_items.size() * kItemWords - h.off_prefill_cta_ptr});
    if (!L.merges.empty())
      ranges.push_back({(size_t)h.off_merge_tasks, L.merges.size() * kMergeWords});
    if (!L.joins.empty())
      ranges.push_back({(size_t)h.off_decode_joins, L.joins.size() * kJoinWords});
    if (!L.dequant.empty())
      ranges.push_back({(size_t)h.off_dequant_units, L.dequant.size() * kDequantWords});
  } else {
    ranges.push_back({0, w});
  }
  int32_t* img = static_cast<int32_t*>(pinned_h);
  for (const auto& r : ranges) std::memset(img + r.first, 0, r.second * 4);
  std::memcpy(img, &h, sizeof(h));
  std::memcpy(img + h.off_decode_cta_ptr, L.dec_cta_ptr.data(), L.dec_cta_ptr.size() * 4);
  if (!L.dec_items.empty())
    std::memcpy(img + h.off_decode_items, L.dec_items.data(), L.dec_items.size() * sizeof(PkaWorkItem));
  std::memcpy(img + h.off_prefill_cta_ptr, L.pre_cta_ptr.data(), L.pre_cta_ptr.size() * 4);
  if (!L.pre_items.empty())
    std::memcpy(img + h.off_prefill_items, L.pre_items.data(), L.pre_items.size() * sizeof(PkaWorkItem));
  if (!L.merges.empty())
    std::memcpy(img + h.off_merge_tasks, L.merges.data(), L.merges.size() * sizeof(PkaMergeTask));
  if (!L.merge_slots.empty())
    std::memcpy(img + h.off_merge_slots, L.merge_slots.data(), L.merge_slots.size() * 4);
  if (!L.joins.empty())
    std::memcpy(img + h.off_decode_joins, L.joins.data(), L.joins.size() * sizeof(PkaDecodeJoin));
  if (!L.dequant.empty())
    std::memcpy(img + h.off_dequant_units, L.dequant.data(),
                L.dequant.size() * sizeof(PkaDequantUnit));

  plan->params = *p;
  plan->hdr = h;
  plan->int_ws_d = static_cast<int32_t*>(int_ws_d);
  plan->layout_records = (int32_t)layout_records;
  plan->merge_capacity = (int32_t)n_merge;
  plan->dequant_capacity = (int32_t)n_dequant;
  plan->scratch_capacity = scratch_rows;
  if (int_ws_d) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (!plan->event) e = cudaEventCreateWithFlags(&plan->event, cudaEventDisableTiming);
    for (const auto& r : ranges)
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(static_cast<int32_t*>(int_ws_d) + r.first, img + r.first, r.second * 4,
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaEventRecord(plan->event, st);
    if (e != cudaSuccess) return cuda_fail(e, "plan copy");
    plan->copy_pending = true;
  }
  plan->planned = true;
  return PKA_OK;
}

}  // namespace

extern "C" {

const char* pka_status_str(pka_status s) {
  switch (s) {
    case PKA_OK: return "ok";
    case PKA_ERR_INVALID_ARG: return "invalid argument";
    case PKA_ERR_METADATA: return "metadata violates the indptr / page-table contract";
    case PKA_ERR_UNSUPPORTED: return "unsupported head_dim, head ratio or mode";
    case PKA_ERR_WORKSPACE: return "workspace or staging buffer too small";
    case PKA_ERR_STALE_PLAN: return "run parameters differ from the planned ones";
    case PKA_ERR_CUDA: return "CUDA runtime error";
    case PKA_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting on a barrier";
  }
  return "unknown status";
}

pka_status pka_version(int32_t* major, int32_t* minor) {
  if (!major || !minor) return PKA_ERR_INVALID_ARG;
  *major = PKA_VERSION_MAJOR;
  *minor = PKA_VERSION_MINOR;
  return PKA_OK;
}

pka_status pka_validate(const pka_params* p, int32_t batch, const int32_t* qo,
                        const int32_t* kv, const int32_t* last) {
  if (!params_ok(p)) return PKA_ERR_INVALID_ARG;
  pka_status s = check_supported(p);
  if (s != PKA_OK) return s;
  Batch b;
  s = derive(p, batch, qo, kv, last, &b, p->mask_mode);
  return s != PKA_OK ? s : check_kv_dtype(p, b);
}

pka_status pka_plan_create(pka_plan_t* plan) {
  if (!plan) return PKA_ERR_INVALID_ARG;
  *plan = new (std::nothrow) pka_plan_s();
  return *plan ? PKA_OK : PKA_ERR_INVALID_ARG;
}

void pka_plan_destroy(pka_plan_t plan) {
  if (!plan) return;
  if (plan->event) {
    cudaEventSynchronize(plan->event);
    cudaEventDestroy(plan->event);
  }
  delete plan;
}

pka_status pka_plan(pka_plan_t plan, const pka_params* p, int32_t batch, const int32_t* qo,
                    const int32_t* kv, const int32_t* last, void* int_ws_d, size_t int_ws_bytes,
                    void* pinned_h, size_t pinned_bytes, void* stream) {
  if (!plan || !params_ok(p)) return PKA_ERR_INVALID_ARG;
  plan->planned = false;
  plan->info = pka_plan_info{};
  pka_status s = check_supported(p);
  if (s != PKA_OK) return s;
  std::vector<Batch> lv(1);
  s = derive(p, batch, qo, kv, last, &lv[0], p->mask_mode);
  if (s == PKA_OK) s = check_kv_dtype(p, lv[0]);
  if (s != PKA_OK) return s;
  return plan_levels(plan, p, lv, batch, false, int_ws_d, int_ws_bytes, pinned_h, pinned_bytes,
                     stream);
}

pka_status pka_plan_cascade(pka_plan_t plan, const pka_params* p, int32_t num_levels,
                            const int32_t* num_nodes, const int32_t* const* qo,
                            const int32_t* const* kv, const int32_t* const* last, void* int_ws_d,
                            size_t int_ws_bytes, void* pinned_h, size_t pinned_bytes,
                            void* stream) {
  if (!plan || !params_ok(p)) return PKA_ERR_INVALID_ARG;
  plan->planned = false;
  plan->info = pka_plan_info{};
  pka_status s = check_supported(p);
  if (s != PKA_OK) return s;
  if (p->kv_ragged || p->mask_mode == PKA_MASK_CUSTOM || graph_mode(p)) return PKA_ERR_UNSUPPORTED;
  if (num_levels < 1 || num_levels > PKA_MAX_CASCADE_LEVELS || !num_nodes || !qo || !kv || !last)
    return PKA_ERR_INVALID_ARG;
  std::vector<Batch> lv(num_levels);
  int64_t kv_off = 0;
  for (int l = 0; l < num_levels; ++l) {
    if (!qo[l] || !kv[l] || !last[l] || num_nodes[l] < 0) return PKA_ERR_INVALID_ARG;
    const bool shared = l + 1 < num_levels;
    s = derive(p, num_nodes[l], qo[l], kv[l], last[l], &lv[l],
               shared ? (int)PKA_MASK_NONE : p->mask_mode, shared, kv_off);
    if (s != PKA_OK) return s;
    if (lv[l].nnz_q != lv[0].nnz_q) return PKA_ERR_METADATA;  // levels split the same rows
    if (shared && p->mask_mode != PKA_MASK_NONE) lv[l].item_flags = PKA_ITEM_ALL_VISIBLE;
    kv_off += kv[l][num_nodes[l]];
  }
  if (kv_off > INT32_MAX) return PKA_ERR_UNSUPPORTED;
  return plan_levels(plan, p, lv, num_nodes[num_levels - 1], true, int_ws_d, int_ws_bytes,
                     pinned_h, pinned_bytes, stream);
}

pka_status pka_plan_get_info(pka_plan_t plan, pka_plan_info* info) {
  if (!plan || !info) return PKA_ERR_INVALID_ARG;
  *info = plan->info;
  return PKA_OK;
}

pka_status pka_plan_wait(pka_plan_t plan) {
  if (!plan) return PKA_ERR_INVALID_ARG;
  if (plan->copy_pending && plan->event) {
    if (cudaEventSynchronize(plan->event) != cudaSuccess) return PKA_ERR_CUDA;
    plan->copy_pending = false;
  }
  return PKA_OK;
}

pka_status pka_run(pka_plan_t plan, const pka_params* p, const void* q, const void* k,
                   const void* v, int64_t page_stride, const int32_t* kv_indices,
                   const uint8_t* mask, void* o, float* lse, void* float_ws, size_t float_ws_bytes,
                   void* stream) {
  if (!plan || !p || !plan->planned) return PKA_ERR_INVALID_ARG;
  if (std::memcmp(&plan->params, p, sizeof(pka_params)) != 0) return PKA_ERR_STALE_PLAN;
  if (!plan->int_ws_d) return PKA_ERR_INVALID_ARG;  // a host-only (dry-run) plan cannot run
  // no query rows (an empty batch, or only qo_len == 0 requests): nothing to
  // compute, and the (empty) buffers may be null
  if (plan->info.nnz_qo == 0 && !graph_mode(p)) return PKA_OK;
  if (!q || !k || !v || !o) return PKA_ERR_INVALID_ARG;
  if (!p->kv_ragged && (!kv_indices || page_stride <= 0)) return PKA_ERR_INVALID_ARG;
  // 16-byte alignment of every row the kernels move with vector or bulk copies
  const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  const bool fp8 = p->kv_dtype == PKA_KV_FP8_E4M3;
  // page stride in elements: 16 bytes for bf16 (8 elements) or e4m3 (16)
  if ((mis & 15) || (!p->kv_ragged && (page_stride & (fp8 ? 15 : 7)))) return PKA_ERR_INVALID_ARG;
  if (p->mask_mode == PKA_MASK_CUSTOM && !mask) return PKA_ERR_INVALID_ARG;
  if (float_ws_bytes < plan->info.float_ws_bytes || (plan->info.float_ws_bytes && !float_ws))
    return PKA_ERR_WORKSPACE;
  const PkaImageHeader& h = plan->hdr;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int g = p->num_qo_heads / p->num_kv_heads;
  float scale = p->sm_scale > 0.f ? p->sm_scale : 1.0f / std::sqrt((float)p->head_dim);
  const bool graph = graph_mode(p);
  size_t rec_o = (size_t)plan->layout_records * p->head_dim * 4;
  size_t rec_o_al = (rec_o + 255) & ~size_t(255);

  AttnArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.k = static_cast<const uint16_t*>(k);
  a.v = static_cast<const uint16_t*>(v);
  a.page_stride = page_stride;
  a.kv_indices = kv_indices;
  a.mask = mask;
  a.o = static_cast<uint16_t*>(o);
  a.lse = lse;
  a.part_o = static_cast<float*>(float_ws);
  a.part_lse = float_ws ? reinterpret_cast<float*>(static_cast<char*>(float_ws) + rec_o_al) : nullptr;
  a.num_qo_heads = p->num_qo_heads;
  a.num_kv_heads = p->num_kv_heads;
  a.page_size = p->kv_ragged ? 1 : p->page_size;
  a.layout = p->layout;
  a.kv_ragged = p->kv_ragged;
  a.mask_mode = p->mask_mode;
  a.heads_per_cta = h.decode_heads_per_cta;
  // e4m3 K/V: K's scale multiplies every score, V's scale the output
  const float k_scale = fp8 && p->k_scale > 0.f ? p->k_scale : 1.f;
  a.scale_log2 = scale * k_scale * 1.4426950408889634f;
  a.kv_fp8 = fp8 ? 1 : 0;
  a.v_scale = fp8 && p->v_scale > 0.f ? p->v_scale : 1.f;

  // Graph mode launches every kernel on its fixed grid, whatever this plan
  // holds, so that a captured run() serves every later plan.
  if (graph || h.num_decode_items > 0) {
    a.cta_ptr = plan->int_ws_d + h.off_decode_cta_ptr;
    a.items = reinterpret_cast<const PkaWorkItem*>(plan->int_ws_d + h.off_decode_items);
    a.joins = h.off_decode_joins
                  ? reinterpret_cast<PkaDecodeJoin*>(plan->int_ws_d + h.off_decode_joins)
                  : nullptr;
    cudaError_t e = pka::launch_decode(a, h.num_decode_ctas, p->head_dim, g, &plan->decode_maps, st);
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  }
  if (graph || h.num_prefill_items > 0) {
    a.cta_ptr = plan->int_ws_d + h.off_prefill_cta_ptr;
    a.items = reinterpret_cast<const PkaWorkItem*>(plan->int_ws_d + h.off_prefill_items);
    // the Q (and ragged K/V) tensor maps span the buffers' declared rows
    const int rows = graph ? p->graph_max_qo_rows : plan->info.nnz_qo;
    int64_t kv_rows = graph ? p->graph_max_kv_tokens : plan->info.total_kv;
    pka::AttnArgs pa = a;
    if (graph ? plan->dequant_capacity > 0 : h.num_dequant_units > 0) {
      // e4m3 K/V: decode the keys of the tensor-core requests to bf16 in the
      // float workspace (after the partial states); the tensor-core kernel
      // then reads them as ragged K/V.  Graph mode lays the scratch out for
      // its capacity and launches on that fixed size; the dequant kernel
      // reads this plan's unit and row counts from the device image.
      const size_t rec_lse = plan->layout_records
                                 ? (((size_t)plan->layout_records * 4 + 255) & ~size_t(255))
                                 : 0;
      char* base = static_cast<char*>(float_ws) + (plan->layout_records ? rec_o_al : 0) + rec_lse;
      uint16_t* sk = reinterpret_cast<uint16_t*>(base);
      uint16_t* sv = reinterpret_cast<uint16_t*>(base + kv_scratch_bytes(p, plan->scratch_capacity));
      const int32_t* counts =
          graph ? plan->int_ws_d + offsetof(PkaImageHeader, num_dequant_units) / 4 : nullptr;
      cudaError_t e = pka::launch_dequant(
          reinterpret_cast<const PkaDequantUnit*>(plan->int_ws_d + h.off_dequant_units),
          graph ? plan->dequant_capacity : h.num_dequant_units,
          graph ? plan->scratch_capacity : h.dequant_rows, counts, kv_indices, k, v, page_stride,
          p->page_size, p->layout, p->kv_ragged, p->num_kv_heads, p->head_dim, sk, sv, st);
      if (e != cudaSuccess) return cuda_fail(e, "dequant launch");
      pa.k = sk;
      pa.v = sv;
      pa.kv_ragged = 1;
      pa.page_size = 1;
      pa.kv_fp8 = 0;
      kv_rows = plan->scratch_capacity;
    }
    cudaError_t e = pka::launch_prefill(pa, h.num_prefill_ctas, p->head_dim, g, rows, kv_rows,
                                         &plan->prefill_maps, st);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  }
  if (graph ? plan->merge_capacity > 0 : h.num_merge_tasks > 0) {
    pka::MergeArgs m{};
    m.tasks = reinterpret_cast<const PkaMergeTask*>(plan->int_ws_d + h.off_merge_tasks);
    m.num_tasks = graph ? plan->merge_capacity : h.num_merge_tasks;
    if (graph) m.num_tasks_dev = plan->int_ws_d + offsetof(PkaImageHeader, num_merge_tasks) / 4;
    if (h.off_merge_slots) m.slots = plan->int_ws_d + h.off_merge_slots;
    m.heads = p->num_qo_heads;
    m.part_o = a.part_o;
    m.part_lse = a.part_lse;
    m.o = a.o;
    m.lse = lse;
    m.head_dim = p->head_dim;
    cudaError_t e = pka::launch_merge(m, st);
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  }
  return PKA_OK;
}

pka_status pka_append_paged_kv_cache(const pka_params* p, int32_t batch, const void* k_new,
                                     const void* v_new, const int32_t* append_indptr,
                                     int64_t nnz_new, const int32_t* kv_indptr,
                                     const int32_t* kv_indices, const int32_t* last_page_len,
                                     void* k, void* v, int64_t page_stride, void* stream) {
  if (!params_ok(p) || batch < 0 || nnz_new < 0) return PKA_ERR_INVALID_ARG;
  if (p->head_dim != 64 && p->head_dim != 128) return PKA_ERR_UNSUPPORTED;

  if (p->kv_ragged) return PKA_ERR_UNSUPPORTED;
  if (nnz_new == 0 || batch == 0) return PKA_OK;
  if (!k_new || !v_new || !append_indptr || !kv_indptr || !kv_indices || !last_page_len || !k ||
      !v || page_stride <= 0)
    return PKA_ERR_INVALID_ARG;
  // 16-byte row pieces move per thread: 16-byte aligned buffers, and a page
  // stride of whole 16-byte units (8 bf16 or 16 e4m3 elements)
  const uintptr_t mis = reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
                        reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v);
  if ((mis & 15) || (page_stride & (p->kv_dtype == PKA_KV_FP8_E4M3 ? 15 : 7)))
    return PKA_ERR_INVALID_ARG;
  cudaError_t e = pka::launch_append(*p, batch, static_cast<const uint16_t*>(k_new),
                                     static_cast<const uint16_t*>(v_new), append_indptr, nnz_new,
                                     kv_indptr, kv_indices, last_page_len, k, v, page_stride,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : cuda_fail(e, "append launch");
}

pka_status pka_merge_states(const float* v, const float* lse, const int32_t* indptr,
                            int32_t rows, int32_t heads, int32_t dim, void* v_out,
                            float* lse_out, void* stream) {
  if (rows < 0 || heads < 1) return PKA_ERR_INVALID_ARG;
  if (dim != 64 && dim != 128) return PKA_ERR_UNSUPPORTED;
  if (rows == 0) return PKA_OK;
  if (!v || !lse || !indptr || !v_out) return PKA_ERR_INVALID_ARG;
  pka::MergeArgs m{};
  m.indptr = indptr;
  m.rows = rows;
  m.heads = heads;
  m.part_o = v;
  m.part_lse = lse;
  m.o = static_cast<uint16_t*>(v_out);
  m.lse = lse_out;
  m.head_dim = dim;
  cudaError_t e = pka::launch_merge(m, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : cuda_fail(e, "merge launch");
}

pka_status pka_packbits(const uint8_t* in, int64_t n, uint8_t* out, void* stream) {
  if (n < 0) return PKA_ERR_INVALID_ARG;
  if (n == 0) return PKA_OK;
  if (!in || !out) return PKA_ERR_INVALID_ARG;
  cudaError_t e = pka::launch_packbits(in, n, out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : cuda_fail(e, "packbits launch");
}

pka_status pka_get_device_error(int32_t* code, void* stream) {
  if (!code) return PKA_ERR_INVALID_ARG;
  cudaError_t e = pka::read_and_clear_device_error(code, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : cuda_fail(e, "device error read");
}

pka_status pka_selftest_bounded_wait(int32_t arrive, int32_t polls, void* stream) {
  if ((arrive != 0 && arrive != 1) || polls < 1 || polls > 1000) return PKA_ERR_INVALID_ARG;
  cudaError_t e = pka::launch_wait_selftest(arrive, polls, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKA_OK : cuda_fail(e, "wait self-test launch");
}

const char* pka_last_error(void) { return g_last_error; }

}  // extern "C"
