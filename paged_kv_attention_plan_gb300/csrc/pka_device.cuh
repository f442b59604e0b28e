// Device helpers: mbarriers, bulk async copies, bf16 packing, bounded waits.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace pka {

// A barrier wait suspends the warp (up to kSuspendNs per poll) until the
// phase completes; after kWaitPolls polls (a few seconds) it gives up, the
// caller records PKA_ERR_DEVICE_TIMEOUT in the device error word and the CTA
// leaves.
constexpr uint32_t kSuspendNs = 1000000;  // 1 ms
constexpr uint32_t kWaitPolls = 4000;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that may suspend the thread for up to `ns` nanoseconds.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded wait of one thread for the completion of the phase with the given
// parity (for waits that a single lane of its warp makes).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint32_t polls = kWaitPolls) {
  if (mbar_try_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < polls; ++i)
    if (mbar_try_wait_suspend(bar, parity, kSuspendNs)) return true;
  return false;
}

// Bounded wait made by a whole warp (all 32 lanes converged).  The warp
// decides together: it goes on once every lane has seen the phase complete,
// and gives up, all lanes at once, when the common poll count runs out, so
// a timeout can never leave some lanes waiting and others gone (which would
// hang the warp at its next shuffle or __syncwarp).  A completed phase stays
// complete for its parity until the barrier completes the next one, which
// needs this warp's own later arrival, so lanes that saw it early keep
// seeing it.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity,
                                               uint32_t polls = kWaitPolls) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  for (uint32_t i = 0; i < polls; ++i)
    if (__all_sync(0xffffffffu, mbar_try_wait_suspend(bar, parity, kSuspendNs))) return true;
  return false;
}

// Warp-uniform read of a CTA-wide abort flag (all 32 lanes converged).
__device__ __forceinline__ bool warp_any(volatile int* flag) {
  return __any_sync(0xffffffffu, *flag != 0);
}

// Global -> shared bulk copy completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Two bf16 packed in a 32-bit word -> (low, high) as floats.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Round two floats to bf16 (nearest even) and pack them (low = a).
__device__ __forceinline__ uint32_t float2_to_bf16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

}  // namespace pka
