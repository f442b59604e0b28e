// Layout of the plan image that pka_plan writes into the pinned staging
// buffer and copies into the caller's device int workspace.  Shared by the
// host planner and the kernels (both are the product path).
//
// image := header | decode_cta_ptr | decode_items | prefill_cta_ptr |
//          prefill_items | merge_tasks | merge_slots | decode_joins |
//          dequant_units (offsets in int32 units)
#pragma once
#include <stdint.h>

#define PKA_IMAGE_MAGIC 0x31414B50  // "PKA1"

struct PkaImageHeader {
  int32_t magic;
  int32_t total_words;           // size of the whole image in int32 words
  int32_t num_decode_ctas;
  int32_t num_decode_items;
  int32_t num_prefill_ctas;
  int32_t num_prefill_items;
  int32_t num_merge_tasks;
  int32_t num_partial_records;
  int32_t off_decode_cta_ptr;    // int32[num_decode_ctas + 1]
  int32_t off_decode_items;      // PkaWorkItem[num_decode_items]
  int32_t off_prefill_cta_ptr;   // int32[num_prefill_ctas + 1]
  int32_t off_prefill_items;     // PkaWorkItem[num_prefill_items]
  int32_t off_merge_tasks;       // PkaMergeTask[num_merge_tasks]
  int32_t decode_heads_per_cta;  // kv heads one decode CTA covers
  int32_t graph_mode;            // 1: fixed layout sized by the graph capacities
  int32_t off_merge_slots;       // int32[num_partial_records] record lists, 0 if none
  int32_t num_decode_joins;      // split decode (request, kv head) pairs merged in the decode kernel
  int32_t off_decode_joins;      // PkaDecodeJoin[num_decode_joins], 0 if none
  int32_t num_dequant_units;     // e4m3 K/V: requests whose keys the tensor-core rows read
  int32_t off_dequant_units;     // PkaDequantUnit[num_dequant_units], 0 if none
  int32_t dequant_rows;          // rows of the bf16 K/V scratch (sum of their kv_len)
  int32_t reserved[11];
};

// One unit of attention work: a block of kv heads (decode) or one kv head
// (tensor-core path), a tile of query tokens of one request, and a key range.
struct PkaWorkItem {
  int32_t req;
  int32_t kv_head0;    // first kv head
  int32_t n_kv_heads;  // kv heads covered
  int32_t q_row0;      // global row of the tile's first query token
  int32_t q_local0;    // its index i inside the request (0..qo_len-1)
  int32_t q_count;     // query tokens in the tile
  int32_t qo_len;      // Q of the request
  int32_t kv_len;      // K of the request
  int32_t kv_base;     // kv_indptr[req]: first page id slot (or first token if ragged)
  int32_t t0;          // first key of the range (logical position)
  int32_t t1;          // one past the last key
  int32_t out_rec;     // -1: write O/LSE; else first partial record ([token][qo head])
  int32_t mask_lo;     // mask_indptr[req] (bit offset), low/high words
  int32_t mask_hi;
  int32_t flags;
  int32_t join;        // decode piece of a split: first PkaDecodeJoin of its unit, else -1
};

// One (query row, qo head) whose partial states are merged after a split.
// Record k (0 <= k < nslots) of the task is rec_first + k * rec_stride, or,
// with rec_stride == 0 (cascade plans), merge_slots[rec_first + k].
struct PkaMergeTask {
  int32_t out_row;
  int32_t head;
  int32_t rec_first;
  int32_t nslots;
  int32_t rec_stride;
  int32_t reserved[3];
};

// One kv head of a split decode unit (request, block of kv heads).  Every
// piece of the unit writes its partial states, then counts itself in
// `arrived`; the piece that brings the count to nslots merges the states of
// the kv head's g qo heads (records rec_first + k * rec_stride + h, k <
// nslots, h < g) and sets `arrived` back to 0 for the next run.
struct PkaDecodeJoin {
  int32_t arrived;     // pieces finished so far in the current run (0 between runs)
  int32_t rec_first;   // record of qo head 0 of this kv head in piece 0
  int32_t nslots;      // pieces of the unit (>= 2)
  int32_t rec_stride;  // records between consecutive pieces
};

// e4m3 K/V, one request whose keys the tensor-core rows read: its logical
// keys 0 .. kv_len - 1 (page ids from kv_base in kv_indices) are decoded to
// bf16 rows dst_row0 .. dst_row0 + kv_len - 1 of a [rows, Hk, D] scratch in
// the float workspace, which those rows then read as ragged K/V.
struct PkaDequantUnit {
  int32_t kv_base;   // first page id slot of the request in kv_indices
  int32_t kv_len;    // its keys
  int32_t dst_row0;  // first scratch row
  int32_t reserved;
};

// Item flags
#define PKA_ITEM_ALL_VISIBLE 1  // every key of the range is visible (cascade levels above the last)

static_assert(sizeof(PkaImageHeader) == 128, "header size");
static_assert(sizeof(PkaDecodeJoin) == 16, "join size");
static_assert(sizeof(PkaWorkItem) == 64, "work item size");
static_assert(sizeof(PkaMergeTask) == 32, "merge task size");
static_assert(sizeof(PkaDequantUnit) == 16, "dequant unit size");
