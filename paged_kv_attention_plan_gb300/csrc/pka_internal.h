// Internal declarations shared by the host entry points and the kernels.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <cstring>

#include "pka.h"
#include "pka_plan_image.h"

namespace pka {

// Everything one attention launch needs besides its work list.
struct AttnArgs {
  const int32_t* cta_ptr;     // [num_ctas + 1] item ranges per CTA
  const PkaWorkItem* items;
  PkaDecodeJoin* joins;       // decode: joins of split units (plan image), or null
  const uint16_t* q;          // bf16 bits [nnz_q, Hq, D]
  const uint16_t* k;          // bf16 bits, pool or ragged tensor
  const uint16_t* v;
  int64_t page_stride;        // elements between consecutive pages
  const int32_t* kv_indices;  // page ids (paged only)
  const uint8_t* mask;        // packed custom mask (custom mode only)
  uint16_t* o;                // bf16 bits [nnz_q, Hq, D]
  float* lse;                 // [nnz_q, Hq] or null
  float* part_o;              // [records, D] partial outputs (normalised)
  float* part_lse;            // [records]
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  int32_t page_size;
  int32_t layout;             // PKA_NHD / PKA_HND
  int32_t kv_ragged;
  int32_t mask_mode;
  int32_t heads_per_cta;      // decode: kv heads a CTA covers
  float scale_log2;           // sm_scale * log2(e) (times the K scale for e4m3 K/V)
  int32_t kv_fp8;             // 1: k and v hold e4m3 codes (decode kernel only)
  float v_scale;              // e4m3 V: scale of the codes (1 otherwise)
  int32_t* err;               // device error word (bounded waits that gave up)
};

struct MergeArgs {
  const PkaMergeTask* tasks;  // plan merge list (tasks == null -> indptr mode)
  int32_t num_tasks;          // tasks, or the list's capacity when num_tasks_dev is set
  const int32_t* num_tasks_dev;  // graph mode: the task count in the device plan image
  const int32_t* slots;       // record lists of tasks with rec_stride == 0 (cascade)
  const int32_t* indptr;      // merge_states mode: [rows + 1]
  int32_t rows;
  int32_t heads;
  const float* part_o;        // [records, D]
  const float* part_lse;      // [records]
  uint16_t* o;                // bf16 bits [rows, heads, D]
  float* lse;                 // [rows, heads] or null
  int32_t head_dim;
};

// Tensor maps of one attention launch, kept in the plan object between runs:
// a launch encodes its maps again only when something they describe (a
// buffer address, a stride, a shape) differs from the cached key.
struct MapCache {
  static constexpr int kKeyWords = 16;
  static constexpr int kMaps = 5;
  uint64_t key[kKeyWords];
  int valid;
  int aux;  // a launch setting derived with the maps
  alignas(64) unsigned char maps[kMaps * 128];  // CUtensorMap objects (128 bytes each)

  bool hit(const uint64_t (&k)[kKeyWords]) const {
    if (!valid) return false;
    for (int i = 0; i < kKeyWords; ++i)
      if (key[i] != k[i]) return false;
    return true;
  }
  void store(const uint64_t (&k)[kKeyWords], const void* m, size_t bytes, int aux_value) {
    for (int i = 0; i < kKeyWords; ++i) key[i] = k[i];
    std::memcpy(maps, m, bytes);
    aux = aux_value;
    valid = 1;
  }
};

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for `Kernel` only when
// the current device has not yet been given at least `bytes` (a larger limit
// set earlier covers every smaller launch).
template <auto Kernel>
cudaError_t ensure_dynamic_smem(int bytes) {
  static std::atomic<int> set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < 64;
  if (tracked && set[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && tracked) {
    int cur = set[dev].load(std::memory_order_relaxed);
    while (cur < bytes && !set[dev].compare_exchange_weak(cur, bytes, std::memory_order_acq_rel)) {
    }
  }
  return e;
}

cudaError_t launch_decode(const AttnArgs& a, int num_ctas, int head_dim, int group,
                          MapCache* cache, cudaStream_t stream);
cudaError_t launch_prefill(const AttnArgs& a, int num_ctas, int head_dim, int group, int nnz_q,
                           int64_t total_kv, MapCache* cache, cudaStream_t stream);
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);
cudaError_t launch_packbits(const uint8_t* in, int64_t n, uint8_t* out, cudaStream_t stream);
cudaError_t launch_append(const pka_params& p, int32_t batch, const uint16_t* k_new,
                          const uint16_t* v_new, const int32_t* append_indptr, int64_t nnz,
                          const int32_t* kv_indptr, const int32_t* kv_indices,
                          const int32_t* last_page_len, void* k, void* v,
                          int64_t page_stride, cudaStream_t stream);
cudaError_t launch_wait_selftest(int arrive, int polls, cudaStream_t stream);
cudaError_t launch_dequant(const PkaDequantUnit* units, int n_units, int64_t rows,
                           const int32_t* counts,
                           const int32_t* kv_indices, const void* k8, const void* v8,
                           int64_t page_stride, int page_size, int layout, int ragged, int hk,
                           int d, uint16_t* out_k, uint16_t* out_v, cudaStream_t stream);
cudaError_t read_and_clear_device_error(int32_t* code, cudaStream_t stream);
// Device address of the error word on the current device (null on failure).
int32_t* device_error_word();
// Set the text pka_last_error returns on this thread.
void set_last_error(const char* msg);
// Record a failed CUDA call (its error text and code, after `where`) as the
// text pka_last_error returns on this thread; returns PKA_ERR_CUDA.
pka_status cuda_failure(cudaError_t e, const char* where);
// Multiprocessor count of the current device (cached per device; 0 if the
// query fails).
int current_device_sms();

// Decode launch geometry shared by the planner and the kernel: a decode CTA
// covers `heads_per_cta` kv heads (at most 8, one consumer warp each, so that
// a 16-key stage of K and V stays near 64 KiB); each warp serves all g <= 8
// qo heads of its kv head.
inline int decode_heads_per_cta(int num_kv_heads, int group) {
  (void)group;
  int h = num_kv_heads < 8 ? num_kv_heads : 8;
  while (h > 1 && num_kv_heads % h) --h;
  return h;
}

constexpr int kDecodeTileTokens = 16;   // keys per pipeline stage of the decode kernel
constexpr int kPrefillTileKeys = 128;   // keys per tensor-core tile
constexpr int kPrefillTileRows = 128;   // packed (token, qo head) rows per tile

}  // namespace pka
