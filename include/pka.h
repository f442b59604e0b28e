/*
 * pka.h — batched attention between a ragged query tensor and a paged KV
 * cache in CSR form, as a plan/run C ABI for NVIDIA GB300 (sm_103a).
 *
 * The operation (sources are cited by page title and section):
 *
 *   For request r with Q = qo_len[r] query rows and K = kv_len[r] keys,
 *     O[i, h]   = sum_j softmax_j(scale * q_i,h . k_j,h/g + mask) v_j,h/g
 *     LSE[i, h] = log2( sum_{visible j} exp(scale * q_i,h . k_j,h/g) )
 *   with g = num_qo_heads / num_kv_heads (qo head h reads kv head h / g).
 *   - "Deep Dive - FlashInfer", "Why inference attention becomes irregular":
 *     qo_indptr counts query rows; kv_indptr counts page ids; the length
 *     contract K = page_size * (pages - 1) + last_page_len, 1 <= last <= P;
 *     K already includes the tokens appended this step.
 *   - same page, "Causality uses logical positions, not page numbers":
 *     logical key j lives in page kv_indices[kv_indptr[r] + j / P], slot
 *     j % P; causal rows see keys j <= K - Q + i (bottom-right aligned).
 *   - same page, "Core mechanism" and "A worked split-KV example": the state
 *     (o, b) with b the base-2 log of the natural-exp sum; states over
 *     disjoint key ranges merge exactly (normalised scales first).
 *   - same page, "Plan then run": a host plan per batch, a run per layer.
 *   - "KV-Cache layouts" (FlashInfer docs): "NHD/HND" page layouts, "Ragged
 *     Tensor" (kv_indptr over tokens), "Mask layout (2D Ragged Tensor)"
 *     (per-request row-major masks at mask_indptr = cumsum(qo_len * kv_len),
 *     bit-packed 8 per byte, little-endian), "Page table layout" (5-D or
 *     tuple K/V storage; the caller owns the page table).
 *
 * Conventions for every call:
 *   - Payloads (q, k, v, o, k_new, v_new) are bfloat16; lse is float32 in
 *     base-2 units; index arrays are int32.
 *   - "_h" pointers are host memory, "_d" and payload pointers device memory.
 *   - The library allocates no device memory and no pinned memory.  The
 *     caller owns every buffer; pka_plan_create allocates the host plan
 *     object (and one CUDA event on the first pka_plan with a device
 *     workspace).  The plan object keeps the planner's host work lists from
 *     one plan to the next (their size follows the largest plan so far)
 *     until pka_plan_destroy, so steady-state planning does not allocate.
 *   - All device work is ordered on the caller's stream, passed as a
 *     cudaStream_t cast to void* (NULL = legacy default stream).
 *   - Every call returns a pka_status; nothing throws across the ABI and no
 *     kernel traps.  Kernels that wait on a barrier give up after a bounded
 *     number of polls and record PKA_ERR_DEVICE_TIMEOUT, readable with
 *     pka_get_device_error.
 */
#ifndef PKA_H_
#define PKA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKA_VERSION_MAJOR 1
#define PKA_VERSION_MINOR 0

typedef enum pka_status {
  PKA_OK = 0,
  PKA_ERR_INVALID_ARG = 1,    /* null pointer, negative size, bad enum        */
  PKA_ERR_METADATA = 2,       /* indptr / last_page_len violate the contract  */
  PKA_ERR_UNSUPPORTED = 3,    /* head_dim, head ratio or mode not built       */
  PKA_ERR_WORKSPACE = 4,      /* a workspace or staging buffer is too small   */
  PKA_ERR_STALE_PLAN = 5,     /* run() parameters differ from plan()'s        */
  PKA_ERR_CUDA = 6,           /* a CUDA runtime call failed                   */
  PKA_ERR_DEVICE_TIMEOUT = 7  /* a kernel gave up waiting on a barrier        */
} pka_status;

typedef enum pka_layout { PKA_NHD = 0, PKA_HND = 1 } pka_layout;
typedef enum pka_mask_mode {
  PKA_MASK_NONE = 0,
  PKA_MASK_CAUSAL = 1,  /* key j visible to local row i iff j <= K - Q + i   */
  PKA_MASK_CUSTOM = 2   /* bit mask_indptr[r] + i*K + j of the packed mask; */
                        /* 1 keeps the key, 0 drops it                       */
} pka_mask_mode;
/* K/V element type.  PKA_KV_FP8_E4M3: the pools hold 8-bit e4m3 codes (the
 * OCP 8-bit float format: 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits); code c of the K pool stands for e4m3(c) * k_scale, of the V pool for
 * e4m3(c) * v_scale.  The pages tie low-precision caches to the HND layout
 * ("KV-Cache layouts", "NHD/HND") but fix no scale contract: one scale per
 * pool is the plainest reading.  Any layout and page size; page_stride (in
 * elements = bytes) a multiple of 16.  Decode rows read the codes directly;
 * for rows with qo_len >= 2 (tensor cores) run() first decodes each such
 * request's keys to bf16 (exact) into a scratch in the float workspace
 * (info.kv_scratch_rows rows of K and of V; in a cascade, each node's keys
 * once), then reads that scratch.  In graph mode the scratch is laid out for
 * graph_max_kv_tokens rows (the keys of all rows with qo_len >= 2 of any
 * plan must fit); without that capacity graph mode refuses such rows
 * (PKA_ERR_UNSUPPORTED), and a plan whose rows outgrow it gets
 * PKA_ERR_WORKSPACE. */
typedef enum pka_kv_dtype { PKA_KV_BF16 = 0, PKA_KV_FP8_E4M3 = 1 } pka_kv_dtype;
typedef enum pka_split_mode {
  PKA_SPLIT_OFF = 0,    /* one work item per (request, head block, q tile)   */
  PKA_SPLIT_AUTO = 1,   /* planner balances keys across CTAs, merges splits  */
  PKA_SPLIT_FIXED = 2   /* every key range cut into fixed_split_pages pages  */
} pka_split_mode;

typedef struct pka_params {
  int32_t num_qo_heads;      /* Hq >= 1                                        */
  int32_t num_kv_heads;      /* Hk >= 1, Hq % Hk == 0, Hq / Hk in {1,2,4,8}    */
  int32_t head_dim;          /* D in {64, 128}                                 */
  int32_t page_size;         /* P >= 1 (ignored when kv_ragged)               */
  int32_t layout;            /* pka_layout of the K/V pages                    */
  int32_t mask_mode;         /* pka_mask_mode                                  */
  float sm_scale;            /* <= 0 selects 1/sqrt(D)                         */
  int32_t kv_ragged;         /* 1: K/V are ragged [tokens, Hk, D] tensors and  */
                             /*    kv_indptr counts tokens ("Ragged Tensor")   */
  int32_t split_mode;        /* pka_split_mode                                 */
  int32_t fixed_split_pages; /* pages per chunk for PKA_SPLIT_FIXED (>= 1)     */
  int32_t num_sms;           /* 0: query the current device; > 0: plan for it  */
  /* CUDA-graph mode (graph_max_batch > 0): the plan image gets a fixed layout
   * sized by these capacities and run() launches fixed grids, so a run()
   * captured in a CUDA graph stays valid when later plans (same params,
   * same workspaces) rewrite the image in place.  Split mode FIXED is not
   * available in graph mode; prefill rows are not split. */
  int32_t graph_max_batch;     /* the most requests of any plan                */
  int32_t graph_max_qo_rows;   /* the most query rows; q and o hold this many   */
  int32_t graph_max_kv_tokens; /* ragged K/V: the most K/V rows; e4m3 pools:    */
                               /* the most keys of rows with qo_len >= 2       */
  int32_t kv_dtype;            /* pka_kv_dtype of the K/V pools                 */
  float k_scale;               /* PKA_KV_FP8_E4M3: scale of K codes (<= 0: 1)    */
  float v_scale;               /* PKA_KV_FP8_E4M3: scale of V codes (<= 0: 1)    */
  /* 1: rows with qo_len == 1 also go to the tensor-core (tcgen05) kernel, the
   * g qo heads of a row packed into its 128-row tile ("Deep Dive -
   * FlashInfer": decode through the tensor-core tile for grouped heads);
   * 0: they go to the decode kernel (warp-level MMAs, faster for decode on
   * GB300).  Over e4m3 pools such rows read the bf16 scratch like the other
   * tensor-core rows (and count against graph_max_kv_tokens in graph mode). */
  int32_t decode_on_tensor_cores;
  int32_t reserved[1];         /* must be zero                                  */
} pka_params;

/* Summary of a plan, filled by pka_plan (also when it fails with
 * PKA_ERR_WORKSPACE, so a caller can size its buffers and call again). */
typedef struct pka_plan_info {
  uint64_t int_ws_bytes;     /* device int workspace and pinned staging bytes  */
  uint64_t float_ws_bytes;   /* float workspace pka_run needs (split states)   */
  int32_t num_requests;
  int32_t nnz_qo;            /* qo_indptr[batch]                               */
  int64_t total_kv;          /* sum of kv_len over requests                    */
  int32_t num_decode_ctas;   /* CTAs of the decode launch (qo_len == 1 rows)   */
  int32_t num_decode_items;
  int32_t num_prefill_ctas;  /* CTAs of the tensor-core launch (qo_len >= 2)   */
  int32_t num_prefill_items;
  int32_t num_merge_tasks;   /* (row, qo head) pairs merged after a split     */
  int32_t num_partial_records;
  int32_t decode_chunk_tokens; /* keys per decode CTA (0: no split)            */
  int32_t num_decode_joins;  /* split (decode row, kv head) pairs that the     */
                             /* decode kernel merges itself (their g qo heads  */
                             /* are among num_merge_tasks)                     */
  int32_t kv_scratch_rows;   /* e4m3 K/V: bf16 rows decoded for the tensor-core */
                             /* rows in the float workspace (0 otherwise)       */
  int32_t reserved[3];
} pka_plan_info;

typedef struct pka_plan_s* pka_plan_t;

/* Static description of an error code. Never NULL. */
const char* pka_status_str(pka_status status);

/* Library version (PKA_VERSION_MAJOR / MINOR). */
pka_status pka_version(int32_t* major, int32_t* minor);

/* Check the batch description against the contract without planning.
 * qo_indptr_h may be NULL (decode: one row per request).  Host only; needs
 * no GPU.  Returns PKA_ERR_METADATA for: indptr[0] != 0, a decreasing
 * indptr, a request with no page, last_page_len outside 1..P, causal rows
 * with kv_len < qo_len; PKA_ERR_UNSUPPORTED for head_dim not in {64,128} or a
 * head ratio not in {1,2,4,8}; PKA_ERR_INVALID_ARG for bad enums or sizes. */
pka_status pka_validate(const pka_params* params, int32_t batch, const int32_t* qo_indptr_h,
                        const int32_t* kv_indptr_h, const int32_t* last_page_len_h);

/* Create / destroy the host plan object. */
pka_status pka_plan_create(pka_plan_t* plan);
void pka_plan_destroy(pka_plan_t plan);

/* In graph mode pka_plan returns PKA_ERR_WORKSPACE when the batch exceeds the
 * declared capacities (requests, query rows, ragged K/V rows). */

/* plan(): inspect one batch on the host ("Deep Dive - FlashInfer", "Plan
 * then run"; "Load balancing and split-KV decisions").
 *   Validates the metadata, derives kv_len, mask offsets, query tiles with
 *   GQA row packing, split-KV chunks and the merge list, writes the plan
 *   image into pinned_h and copies it into int_ws_d with cudaMemcpyAsync on
 *   `stream`.  kv_indices is not read here: pka_run reads it on the device, so
 *   pages may be remapped between runs without a new plan as long as the
 *   lengths stay the same.
 *   int_ws_d == NULL: host-only dry run (no CUDA call; pinned_h may be any
 *   host memory).  Needs info.int_ws_bytes of both int_ws_d and pinned_h; on
 *   a short buffer returns PKA_ERR_WORKSPACE with the sizes in the plan info.
 *   pinned_h must stay untouched until the copy completes: call
 *   pka_plan_wait before reusing it for another plan. */
pka_status pka_plan(pka_plan_t plan, const pka_params* params, int32_t batch,
                    const int32_t* qo_indptr_h, const int32_t* kv_indptr_h,
                    const int32_t* last_page_len_h, void* int_ws_d, size_t int_ws_bytes,
                    void* pinned_h, size_t pinned_bytes, void* stream);

/* Multi-level cascade plan ("KV-Cache layouts", "Multi-level cascade
 * inference data layout"; "Deep Dive - FlashInfer", "Core mechanism": the
 * (o, lse) state composes across shared prefixes).
 *   Level l (0 = root, num_levels - 1 = last) has num_nodes[l] nodes with its
 *   own host arrays qo_indptr[l] [num_nodes[l] + 1], kv_indptr[l]
 *   [num_nodes[l] + 1] and last_page_len[l] [num_nodes[l]], with the meaning
 *   they have in pka_plan.  Every level splits the same query rows
 *   (qo_indptr[l][num_nodes[l]] equal for all l).  A row attends to the keys
 *   of the node holding it at every level: all of them at the levels above
 *   the last (a shared prefix lies before the row's own tokens), and at the
 *   last level those params->mask_mode leaves visible, with that node's
 *   (qo_len, kv_len).  A node above the last may have no pages (its
 *   last_page_len is then ignored); last-level nodes follow pka_plan's
 *   contract.
 *   pka_run then takes as kv_indices the page ids of all levels concatenated
 *   in level order: level l's kv_indptr indexes its own part, which starts
 *   after the sum of kv_indptr[l'][num_nodes[l']] over l' < l.  Each level's
 *   work writes fp32 partial states to the float workspace and the merge
 *   kernel combines every row's states into O and LSE in the same pka_run.
 *   Supported: paged K/V (bf16 or e4m3 pools), mask none or causal, split
 *   off/auto/fixed, up to PKA_MAX_CASCADE_LEVELS levels; ragged K/V, custom
 *   masks and graph mode return PKA_ERR_UNSUPPORTED.  Workspace rules and errors as in pka_plan;
 *   rows split differently between levels give PKA_ERR_METADATA. */
#define PKA_MAX_CASCADE_LEVELS 16
pka_status pka_plan_cascade(pka_plan_t plan, const pka_params* params, int32_t num_levels,
                            const int32_t* num_nodes, const int32_t* const* qo_indptr_h,
                            const int32_t* const* kv_indptr_h,
                            const int32_t* const* last_page_len_h, void* int_ws_d,
                            size_t int_ws_bytes, void* pinned_h, size_t pinned_bytes,
                            void* stream);

/* Copy the plan's summary into *info. */
pka_status pka_plan_get_info(pka_plan_t plan, pka_plan_info* info);

/* Block until the plan's host-to-device copy has completed. */
pka_status pka_plan_wait(pka_plan_t plan);

/* run(): execute the plan for one layer.
 *   q   [nnz_qo, Hq, D] bf16, o [nnz_qo, Hq, D] bf16, lse [nnz_qo, Hq] fp32
 *   (lse may be NULL).
 *   Paged K/V: k and v point at page 0 of the K and V pools; page p starts
 *   page_stride elements after page p-1 (NHD page [P, Hk, D], HND page
 *   [Hk, P, D]).  5-D storage [pages, 2, ...] passes k = base, v = base +
 *   P*Hk*D and page_stride = 2*P*Hk*D; tuple storage passes page_stride =
 *   P*Hk*D.  Ragged K/V: k, v are [kv_indptr[batch], Hk, D]; page_stride and
 *   kv_indices_d are ignored.
 *   packed_mask_d: little-endian bit array, read only for PKA_MASK_CUSTOM.
 *   float_ws_d: at least info.float_ws_bytes (may be NULL when that is 0).
 *   A plan without query rows (info.nnz_qo == 0, not graph mode) returns
 *   PKA_OK at once; its buffers may be NULL.
 *   Split decode rows are merged inside the decode kernel: each piece counts
 *   itself in a counter of the device plan image, and the last one merges.
 *   The counters return to zero by the end of every run, so one plan serves
 *   any number of runs; two runs of one plan must not overlap on the GPU
 *   (they would share the counters and the float workspace).  After
 *   PKA_ERR_DEVICE_TIMEOUT a counter may be left non-zero: call pka_plan
 *   again (it rewrites the image) before the next run.
 *   Returns PKA_ERR_STALE_PLAN when *params differs from the planned one. */
pka_status pka_run(pka_plan_t plan, const pka_params* params, const void* q, const void* k,
                   const void* v, int64_t page_stride, const int32_t* kv_indices_d,
                   const uint8_t* packed_mask_d, void* o, float* lse, void* float_ws_d,
                   size_t float_ws_bytes, void* stream);

/* append_paged_kv_cache ("KV-Cache layouts", "Page table layout": pages of
 * the appended rows are allocated beforehand by the caller).
 *   Request r appends rows append_indptr_d[r] .. append_indptr_d[r+1] of
 *   k_new/v_new [nnz_new, Hk, D]; its kv_len (from kv_indptr_d and
 *   last_page_len_d) already counts them, so row t lands at logical position
 *   kv_len - n_append + t.  Uses params->num_kv_heads, head_dim, page_size and
 *   layout.  Device metadata is trusted (not validated); nnz_new must equal
 *   append_indptr_d[batch].  k_new / v_new are bf16; e4m3 pools
 *   (params->kv_dtype) store each value divided by k_scale / v_scale, rounded
 *   to the nearest e4m3 value (ties to even), magnitudes above 448 clamped to
 *   448.  Buffers 16-byte aligned, page_stride a multiple of 16 bytes;
 *   PKA_ERR_INVALID_ARG otherwise. */
pka_status pka_append_paged_kv_cache(const pka_params* params, int32_t batch, const void* k_new,
                                     const void* v_new, const int32_t* append_indptr_d,
                                     int64_t nnz_new, const int32_t* kv_indptr_d,
                                     const int32_t* kv_indices_d,
                                     const int32_t* last_page_len_d, void* k, void* v,
                                     int64_t page_stride, void* stream);

/* merge_states ("Deep Dive - FlashInfer", "A worked split-KV example"):
 *   For every row r and head h, merge the states s = indptr_d[r] ..
 *   indptr_d[r+1]-1 of v [S, heads, dim] (fp32, each normalised over its own
 *   keys) with statistics lse [S, heads] (base 2).  Empty states (lse = -inf)
 *   are skipped; a row with no finite state yields zeros and -inf.  Writes
 *   v_out [rows, heads, dim] bf16 and lse_out [rows, heads] fp32 (may be
 *   NULL).  dim in {64, 128}. */
pka_status pka_merge_states(const float* v, const float* lse, const int32_t* indptr_d,
                            int32_t rows, int32_t heads, int32_t dim, void* v_out,
                            float* lse_out, void* stream);

/* packbits ("KV-Cache layouts", "Mask layout (2D Ragged Tensor)"): element
 * k of bools_d (non-zero = 1) becomes bit (k & 7) of byte k >> 3 of out_d;
 * the unused high bits of the last byte are 0.  out_d holds (n + 7) / 8 bytes. */
pka_status pka_packbits(const uint8_t* bools_d, int64_t n, uint8_t* out_d, void* stream);

/* pka_run for callers that cannot allocate device memory when they run
 * (no cudaMalloc while a stream is captured into a CUDA graph, engines that
 * give a kernel library no allocator and own every byte of device memory, or
 * hosts where all allocation happens at start-up).  The paper has no
 * counterpart to this call.
 *   Same arguments and results as pka_run, except that the split-KV partial
 *   states live in a fixed 16 MiB array inside the library's device memory
 *   (held by every GPU that loads the library until the process exits)
 *   instead of a caller float workspace.  Allocates nothing: no cudaMalloc,
 *   cudaFree or allocating library routine.
 *   A plan whose info.float_ws_bytes exceeds 16 MiB is rejected with
 *   PKA_ERR_WORKSPACE before anything is launched (pka_last_error says why).
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.
 *   Every call on a device shares the one array and it keeps the last call's
 *   contents (nothing in it needs to start at zero: each state is written
 *   before it is read).  Calls whose kernels overlap on the GPU — on two
 *   streams, or from two threads — race on the array; order them on one
 *   stream or with events. */
pka_status pka_run_static_scratch(pka_plan_t plan, const pka_params* params, const void* q,
                                  const void* k, const void* v, int64_t page_stride,
                                  const int32_t* kv_indices_d, const uint8_t* packed_mask_d,
                                  void* o, float* lse, void* stream);

/* Text of the last CUDA failure behind a PKA_ERR_CUDA returned on the
 * calling thread (empty if none).  Owned by the library; valid until the
 * next call on the same thread. */
const char* pka_last_error(void);

/* Read and clear the device error word written by kernels that gave up on a
 * barrier (0 = none, else a pka_status).  Synchronises `stream`. */
pka_status pka_get_device_error(int32_t* code, void* stream);

/* Host check of a page table ("Deep Dive - FlashInfer", "Where FlashInfer
 * sits in a serving stack": pages reused while another request still reads
 * them, and page tables that disagree with last_page_len, are the bugs of
 * the allocator boundary).  The kernels read kv_indices as given and do not
 * bound-check page ids, so a caller that cannot vouch for its page table
 * calls this first.  Host memory only; no CUDA call.
 *   Checks the length contract (as pka_validate), that kv_indptr_h[batch] <=
 *   num_indices, and that every page id kv_indices_h[kv_indptr_h[r] ..
 *   kv_indptr_h[r+1]) lies in [0, num_pool_pages).  With append_indptr_h
 *   (the rows each request appends this step, as pka_append_paged_kv_cache
 *   takes them; NULL: no appends), it also checks that no (page, slot) that
 *   one request appends to is appended to by another request, or lies in
 *   another request's history (its first kv_len - append_len positions).
 *   Pages that several requests only read (a shared prefix) are allowed.
 *   Returns PKA_ERR_METADATA on the first violation, with *bad_index (may be
 *   NULL) set to the position in kv_indices_h of the offending page id (-1
 *   for a length-contract violation); PKA_ERR_INVALID_ARG for null arrays or
 *   a short kv_indices_h; PKA_ERR_UNSUPPORTED for ragged K/V. */
pka_status pka_check_indices(const pka_params* params, int32_t batch,
                             const int32_t* append_indptr_h, const int32_t* kv_indptr_h,
                             const int32_t* kv_indices_h, int64_t num_indices,
                             const int32_t* last_page_len_h, int64_t num_pool_pages,
                             int64_t* bad_index);

/* Self-test of the bounded barrier waits behind PKA_ERR_DEVICE_TIMEOUT
 * (failure detection; the pages have no counterpart).  Launches one small
 * kernel whose waits use the same code as the attention kernels: two warps
 * wait together (a warp-wide decision, so a timeout never splits a warp) and
 * one thread waits alone, on a barrier with `polls` polls of at most 1 ms
 * each (1 <= polls <= 1000).
 *   arrive == 0: nothing arrives on the barrier; every wait gives up and the
 *     kernel records PKA_ERR_DEVICE_TIMEOUT in the device error word (read
 *     and clear it with pka_get_device_error), then returns normally.
 *   arrive == 1: one thread arrives first; no wait runs out and nothing is
 *     recorded.
 * Either way the kernel ends by itself and the CUDA context stays usable.
 * PKA_ERR_INVALID_ARG for other arrive or polls values. */
pka_status pka_selftest_bounded_wait(int32_t arrive, int32_t polls, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKA_H_ */
