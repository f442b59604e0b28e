// pka_run_static_scratch: pka_run without a caller-provided float workspace.
//
// Some callers cannot call cudaMalloc at the point where they run attention:
// code that runs while a stream is being captured into a CUDA graph, engines
// that hand out all device memory from their own pre-reserved pool and give
// a kernel library no allocator, or hosts where every allocation must happen
// at start-up.  For them this entry point keeps the only scratch the run
// needs — the normalised partial states of split-KV chunks, later combined
// by the merge kernel — in a fixed array in the library's own device memory.
#include <mutex>

#include "pka_internal.h"

namespace pka {
namespace {

// Scratch for split-KV partial states.  Every GPU that loads the library
// holds this array until the process exits.
constexpr size_t kStaticScratchBytes = size_t(16) << 20;
__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device.  Host code must
// not pass the symbol itself to a kernel: on the host it names a stand-in,
// not device memory.  Set up once per device, with that device current.
void* static_scratch_address(cudaError_t* err) {
  static std::mutex mu;
  static void* cache[64] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_static_scratch);
    if (*err != cudaSuccess) return nullptr;
    cache[dev] = p;
  }
  return cache[dev];
}

}  // namespace
}  // namespace pka

extern "C" pka_status pka_run_static_scratch(pka_plan_t plan, const pka_params* params,
                                             const void* q, const void* k, const void* v,
                                             int64_t page_stride, const int32_t* kv_indices_d,
                                             const uint8_t* packed_mask_d, void* o, float* lse,
                                             void* stream) {
  if (!plan || !params) return PKA_ERR_INVALID_ARG;
  pka_plan_info info;
  pka_status s = pka_plan_get_info(plan, &info);
  if (s != PKA_OK) return s;
  if (info.float_ws_bytes > pka::kStaticScratchBytes) {
    pka::set_last_error(
        "pka_run_static_scratch: the plan's split-KV states need more than the 16 MiB static "
        "scratch; use pka_run with a caller workspace or a coarser split");
    return PKA_ERR_WORKSPACE;
  }
  cudaError_t e = cudaSuccess;
  void* scratch = pka::static_scratch_address(&e);
  if (!scratch) {
    // clear the failed call's error, so that it does not surface later as the
    // failure of an unrelated launch
    cudaGetLastError();
    return pka::cuda_failure(e, "pka_run_static_scratch: device address of the static scratch");
  }
  return pka_run(plan, params, q, k, v, page_stride, kv_indices_d, packed_mask_d, o, lse, scratch,
                 pka::kStaticScratchBytes, stream);
}
