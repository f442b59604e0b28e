// pka_check_indices: a host check of a batch's page table against the pool
// and against the slots the batch appends to.
//
// "Deep Dive - FlashInfer", "Where FlashInfer sits in a serving stack": the
// allocator boundary is where page-table bugs come from: a page reused while
// another request still reads it, or a page table that disagrees with
// last_page_len.  The kernels read kv_indices as given, so an id outside the
// pool is an unchecked read of whatever memory lies there.  This call checks,
// on the host and before anything runs:
//   - the length contract (as pka_validate does);
//   - every page id a request uses lies in [0, num_pool_pages);
//   - with append counts: no (page, slot) that one request appends to this
//     step is appended to by another request or read by another request as
//     part of its history (the appended slots of request r are its last
//     append_len[r] logical positions, "KV-Cache layouts", "Page table
//     layout": lengths already count the appended tokens).
// Pages shared read-only between requests (a common prefix) are allowed.
#include <cstdint>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pka_internal.h"

extern "C" pka_status pka_check_indices(const pka_params* params, int32_t batch,
                                        const int32_t* append_indptr_h,
                                        const int32_t* kv_indptr_h, const int32_t* kv_indices_h,
                                        int64_t num_indices, const int32_t* last_page_len_h,
                                        int64_t num_pool_pages, int64_t* bad_index) {
  if (bad_index) *bad_index = -1;
  if (!params || batch < 0 || !kv_indptr_h || num_indices < 0 || num_pool_pages < 0)
    return PKA_ERR_INVALID_ARG;
  if (params->kv_ragged) return PKA_ERR_UNSUPPORTED;  // ragged K/V has no page table
  // the length contract and, with appends, append_len <= kv_len (the causal
  // check of pka_validate with the append counts as query rows)
  pka_params p = *params;
  p.mask_mode = append_indptr_h ? PKA_MASK_CAUSAL : PKA_MASK_NONE;
  pka_status s = pka_validate(&p, batch, append_indptr_h, kv_indptr_h, last_page_len_h);
  if (s != PKA_OK) return s;
  if (batch > 0 && (int64_t)kv_indptr_h[batch] > num_indices) return PKA_ERR_INVALID_ARG;
  if (batch > 0 && !kv_indices_h) return PKA_ERR_INVALID_ARG;
  const int64_t P = params->page_size;
  auto fail = [&](int64_t idx) {
    if (bad_index) *bad_index = idx;
    return PKA_ERR_METADATA;
  };
  for (int32_t r = 0; r < batch; ++r)
    for (int64_t i = kv_indptr_h[r]; i < kv_indptr_h[r + 1]; ++i)
      if (kv_indices_h[i] < 0 || (int64_t)kv_indices_h[i] >= num_pool_pages) return fail(i);
  if (!append_indptr_h) return PKA_OK;

  // (page, slot) -> appending request, and the pages that hold appended slots
  std::unordered_map<int64_t, int32_t> written;
  std::unordered_set<int32_t> written_pages;
  std::vector<int64_t> kv_len(batch);
  for (int32_t r = 0; r < batch; ++r) {
    const int64_t npages = (int64_t)kv_indptr_h[r + 1] - kv_indptr_h[r];
    kv_len[r] = P * (npages - 1) + last_page_len_h[r];
    const int64_t n_app = (int64_t)append_indptr_h[r + 1] - append_indptr_h[r];
    for (int64_t pos = kv_len[r] - n_app; pos < kv_len[r]; ++pos) {
      const int64_t at = kv_indptr_h[r] + pos / P;
      const int64_t key = (int64_t)kv_indices_h[at] * P + pos % P;
      if (!written.emplace(key, r).second) return fail(at);  // appended by two requests
      written_pages.insert(kv_indices_h[at]);
    }
  }
  // history positions of every request must not be another request's appends
  for (int32_t r = 0; r < batch; ++r) {
    const int64_t n_app = (int64_t)append_indptr_h[r + 1] - append_indptr_h[r];
    const int64_t hist = kv_len[r] - n_app;
    for (int64_t pi = 0; pi * P < hist; ++pi) {
      const int64_t at = kv_indptr_h[r] + pi;
      if (!written_pages.count(kv_indices_h[at])) continue;
      const int64_t slots = hist - pi * P < P ? hist - pi * P : P;
      for (int64_t sl = 0; sl < slots; ++sl) {
        auto it = written.find((int64_t)kv_indices_h[at] * P + sl);
        if (it != written.end() && it->second != r) return fail(at);
      }
    }
  }
  return PKA_OK;
}
