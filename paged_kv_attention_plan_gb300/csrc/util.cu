// Bandwidth kernels around the attention launches: the state merge,
// append_paged_kv_cache, packbits, and the device error word.
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>

#include "pka_device.cuh"
#include "pka_internal.h"

namespace pka {

// Written by kernels whose bounded barrier waits gave up (0 = no error).
__device__ int32_t g_device_error;

int32_t* device_error_word() {
  static std::mutex mu;
  static int32_t* cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<int32_t*>(p);
  }
  return cache[dev];
}

int current_device_sms() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

cudaError_t read_and_clear_device_error(int32_t* code, cudaStream_t stream) {
  int32_t* p = device_error_word();
  if (!p) return cudaErrorInvalidDevice;
  int32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, p, sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  *code = host;
  if (host != 0) {
    e = cudaMemsetAsync(p, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
  }
  return e;
}

namespace {

// ---------------------------------------------------------------------------
// State merge ("Deep Dive - FlashInfer", "A worked split-KV example"): the
// n-way form of the two-way merge.  Shift by the largest finite statistic,
// weight each state by 2^(b - shift), normalise the weights before the
// weighted sum, and return shift + log2(sum of weights).  States with
// b = -inf (no visible key) carry no weight; if every state is empty the
// result is a zero vector and -inf.  One warp per (row, head): lane k takes
// the statistics of slots k, k + 32, ... (warp reductions for the shift and
// the sum of weights; the first 32 slots' records and statistics stay in
// registers), then the warp adds the weighted rows slot by slot in slot
// order, eight rows in flight.
// ---------------------------------------------------------------------------
template <int D>
__device__ __forceinline__ void merge_one(const MergeArgs& a, const int task, const int lane) {
  constexpr int PER = D / 32;  // dims per lane
  int out_row, head, rec_first, nslots, stride;
  if (a.tasks) {
    const PkaMergeTask t = a.tasks[task];
    out_row = t.out_row;
    head = t.head;
    rec_first = t.rec_first;
    nslots = t.nslots;
    stride = t.rec_stride;
  } else {
    out_row = task / a.heads;
    head = task % a.heads;
    const int s0 = a.indptr[out_row], s1 = a.indptr[out_row + 1];
    rec_first = s0 * a.heads + head;
    nslots = s1 - s0;
    stride = a.heads;
  }
  // record of slot k: strided, or listed (stride 0)
  auto rec_of = [&](int k) -> int {
    return stride ? rec_first + k * stride : a.slots[rec_first + k];
  };
  // slot `lane` (the first 32 slots) stays in registers for all three steps
  int rec0 = 0;
  float b0 = -INFINITY;
  if (lane < nslots) {
    rec0 = rec_of(lane);
    b0 = a.part_lse[rec0];
  }
  float shift = b0;
  for (int k = lane + 32; k < nslots; k += 32) shift = fmaxf(shift, a.part_lse[rec_of(k)]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    shift = fmaxf(shift, __shfl_xor_sync(0xffffffffu, shift, off));
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float z = 0.f;
  if (shift != -INFINITY) {
    z = exp2f(b0 - shift);  // 0 for an empty or absent slot
    for (int k = lane + 32; k < nslots; k += 32) z += exp2f(a.part_lse[rec_of(k)] - shift);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
    const float inv_z = 1.f / z;
    constexpr int R = 8;  // rows in flight
    for (int base = 0; base < nslots; base += 32) {
      // this lane's slot of the chunk: its record and normalised weight
      int rec = rec0;
      float b = b0;
      if (base > 0) {
        rec = 0;
        b = -INFINITY;
        if (base + lane < nslots) {
          rec = rec_of(base + lane);
          b = a.part_lse[rec];
        }
      }
      const float wgt = b == -INFINITY ? 0.f : exp2f(b - shift) * inv_z;
      const int cnt = min(32, nslots - base);
      for (int j = 0; j < cnt; j += R) {
        float x[R][PER];
        float wr[R];
#pragma unroll
        for (int q = 0; q < R; ++q) {
          wr[q] = __shfl_sync(0xffffffffu, wgt, (j + q) & 31);
          const int r = __shfl_sync(0xffffffffu, rec, (j + q) & 31);
          if (j + q < cnt && wr[q] != 0.f) {
            const float* src = a.part_o + (int64_t)r * D + lane * PER;
            if constexpr (PER == 4) {
              const float4 v = *reinterpret_cast<const float4*>(src);
              x[q][0] = v.x;
              x[q][1] = v.y;
              x[q][2] = v.z;
              x[q][3] = v.w;
            } else {
              const float2 v = *reinterpret_cast<const float2*>(src);
              x[q][0] = v.x;
              x[q][1] = v.y;
            }
          } else {
            wr[q] = 0.f;
#pragma unroll
            for (int e = 0; e < PER; ++e) x[q][e] = 0.f;
          }
        }
#pragma unroll
        for (int q = 0; q < R; ++q)
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[e] += wr[q] * x[q][e];
      }
    }
  }
  uint16_t* dst = a.o + ((int64_t)out_row * a.heads + head) * D + lane * PER;
  if constexpr (PER == 4) {
    uint2 pk;
    pk.x = float2_to_bf16x2(acc[0], acc[1]);
    pk.y = float2_to_bf16x2(acc[2], acc[3]);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = float2_to_bf16x2(acc[0], acc[1]);
  }
  if (lane == 0 && a.lse)
    a.lse[(int64_t)out_row * a.heads + head] = shift == -INFINITY ? -INFINITY : shift + log2f(z);
}

// Warps stride over the tasks.  With num_tasks_dev set (graph mode) the count
// is read from the device plan image, bounded by the list's capacity.
template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const MergeArgs a) {
  int n = a.tasks ? a.num_tasks : a.rows * a.heads;
  if (a.tasks && a.num_tasks_dev) n = min(max(*a.num_tasks_dev, 0), a.num_tasks);
  const int lane = threadIdx.x & 31;
  for (int task = blockIdx.x * 8 + (threadIdx.x >> 5); task < n; task += gridDim.x * 8)
    merge_one<D>(a, task, lane);
}

// ---------------------------------------------------------------------------
// packbits ("KV-Cache layouts", "Mask layout (2D Ragged Tensor)"): element k
// -> bit (k & 7) of byte k >> 3, little-endian within the byte.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) packbits_kernel(const uint8_t* __restrict__ in, int64_t n,
                                                       uint8_t* __restrict__ out) {
  const int64_t nbytes = (n + 7) >> 3;
  for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nbytes;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t k0 = b << 3;
    uint32_t byte = 0;
    if (k0 + 8 <= n && ((reinterpret_cast<uintptr_t>(in + k0) & 7) == 0)) {
      const uint2 x = *reinterpret_cast<const uint2*>(in + k0);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        byte |= (((x.x >> (8 * i)) & 0xffu) != 0u) << i;
        byte |= (((x.y >> (8 * i)) & 0xffu) != 0u) << (i + 4);
      }
    } else {
      for (int i = 0; i < 8 && k0 + i < n; ++i) byte |= (in[k0 + i] != 0) << i;
    }
    out[b] = static_cast<uint8_t>(byte);
  }
}

// ---------------------------------------------------------------------------
// append_paged_kv_cache ("KV-Cache layouts", "Page table layout"): appended
// row t of request r goes to logical position kv_len - n_append + t, i.e.
// page kv_indices[kv_indptr[r] + pos / P], slot pos % P.  One warp per
// appended row: the request (a binary search of append_indptr), page and
// slot are warp-uniform, and the lanes move the row's Hk * D elements of K
// and of V in 16-byte pieces (coalesced loads of the row; stores of whole
// head rows, contiguous across heads in NHD pages).
// ---------------------------------------------------------------------------
// e4m3 pools: 8 values, each divided by the pool's scale (correctly rounded
// float32 division), then rounded to nearest even e4m3 with saturation at the
// largest finite value (cvt .satfinite), 8 codes packed little-endian.
// A power-of-two scale divides exactly by a multiplication with its
// reciprocal (both give the correctly rounded x / scale), so `inv` > 0 takes
// that path and inv == 0 the division.
__device__ __forceinline__ uint2 bf16x8_to_e4m3x8(uint4 x, float scale, float inv) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t pk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = bf16x2_to_float2(w[i]);
    const float lo = inv > 0.f ? f.x * inv : __fdiv_rn(f.x, scale);
    const float hi = inv > 0.f ? f.y * inv : __fdiv_rn(f.y, scale);
    uint32_t r;
    asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n cvt.u32.u16 %0, t;\n}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    pk[i] = r;
  }
  return make_uint2(pk[0] | (pk[1] << 16), pk[2] | (pk[3] << 16));
}

template <bool F8>
__global__ void __launch_bounds__(256) append_kernel(
    const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
    const int32_t* __restrict__ append_indptr, int32_t batch, int64_t nnz,
    const int32_t* __restrict__ kv_indptr, const int32_t* __restrict__ kv_indices,
    const int32_t* __restrict__ last_page_len, void* __restrict__ k, void* __restrict__ v,
    int64_t page_stride, int hk, int d, int P, int layout, float k_scale, float v_scale,
    float k_inv, float v_inv) {
  constexpr int U = 4;  // 16-byte pieces per lane in flight
  const int lane = threadIdx.x & 31;
  const int vsh = d == 128 ? 4 : 3;  // log2 of the 16-byte pieces of one head row
  const int per_head = 1 << vsh;
  const int per_row = hk * per_head;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); row < nnz;
       row += nwarps) {
    int lo = 0, hi = batch - 1;  // last r with append_indptr[r] <= row
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (append_indptr[mid] <= row) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const int n_app = append_indptr[r + 1] - append_indptr[r];
    const int npages = kv_indptr[r + 1] - kv_indptr[r];
    const int kv_len = (npages - 1) * P + last_page_len[r];
    const int pos = kv_len - n_app + (int)(row - append_indptr[r]);
    const int page = kv_indices[kv_indptr[r] + pos / P];
    const int slot = pos % P;
    const int64_t page_off = (int64_t)page * page_stride;
    const uint4* ks = reinterpret_cast<const uint4*>(k_new + row * (int64_t)per_row * 8);
    const uint4* vs = reinterpret_cast<const uint4*>(v_new + row * (int64_t)per_row * 8);
    for (int c0 = lane; c0 < per_row; c0 += 32 * U) {
      uint4 kx[U], vx[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c < per_row) {
          kx[u] = ks[c];
          vx[u] = vs[c];
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c >= per_row) continue;
        const int h = c >> vsh, cc = c & (per_head - 1);
        const int64_t dst = page_off +
                            (layout == PKA_NHD ? ((int64_t)slot * hk + h) * d
                                               : ((int64_t)h * P + slot) * d) +
                            cc * 8;
        if constexpr (F8) {  // element offsets are byte offsets in e4m3 pools
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(k) + dst) =
              bf16x8_to_e4m3x8(kx[u], k_scale, k_inv);
          *reinterpret_cast<uint2*>(static_cast<uint8_t*>(v) + dst) =
              bf16x8_to_e4m3x8(vx[u], v_scale, v_inv);
        } else {
          *reinterpret_cast<uint4*>(static_cast<uint16_t*>(k) + dst) = kx[u];
          *reinterpret_cast<uint4*>(static_cast<uint16_t*>(v) + dst) = vx[u];
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// e4m3 K/V for the tensor-core rows: decode the keys of each listed request
// (logical position j -> page kv_indices[kv_base + j / P], slot j % P, the
// addressing of "Causality uses logical positions, not page numbers"; ragged
// K/V: row kv_base + j, "KV-Cache layouts", "Ragged Tensor") from
// the e4m3 pools into bf16 rows dst_row0 + j of [rows, Hk, D] scratch
// tensors.  e4m3 -> f16 is exact (cvt), and so is f16 -> f32 -> bf16 for
// every e4m3 value; the pool scales are not applied here (K's is folded into
// the softmax scale, V's into the output).  One thread converts 16 codes of
// K and of V; the unit of a row comes from a binary search of dst_row0.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two_codes) {
  uint32_t h2;
  asm("{\n .reg .b16 c;\n cvt.u16.u32 c, %1;\n cvt.rn.f16x2.e4m3x2 %0, c;\n}"
      : "=r"(h2)
      : "r"(two_codes));
  const float lo = __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
  const float hi = __half2float(__ushort_as_half((unsigned short)(h2 >> 16)));
  return float2_to_bf16x2(lo, hi);
}

// `counts` (graph mode): the plan's unit count and row count, read from the
// device image (its num_dequant_units and dequant_rows words), bounded by the
// capacities n_units and rows the launch was sized for.
__global__ void __launch_bounds__(256) dequant_kernel(
    const PkaDequantUnit* __restrict__ units, int n_units, int64_t rows,
    const int32_t* __restrict__ counts, const int32_t* __restrict__ kv_indices,
    const uint8_t* __restrict__ k8, const uint8_t* __restrict__ v8, int64_t page_stride, int P,
    int layout, int ragged, int hk, int d, uint16_t* __restrict__ out_k,
    uint16_t* __restrict__ out_v) {
  if (counts) {
    n_units = min(max(counts[0], 0), n_units);
    rows = min((int64_t)max(counts[2], 0), rows);
  }
  if (n_units <= 0) return;
  const int vec_per_head = d / 16;  // 16 codes per thread
  const int64_t vec_per_row = (int64_t)hk * vec_per_head;
  const int64_t total = rows * vec_per_row;
  for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
       x += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = x / vec_per_row;
    const int rem = (int)(x - row * vec_per_row);
    const int h = rem / vec_per_head;
    const int c = rem - h * vec_per_head;
    int lo = 0, hi = n_units - 1;  // last unit with dst_row0 <= row
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (units[mid].dst_row0 <= row) lo = mid; else hi = mid - 1;
    }
    const PkaDequantUnit u = units[lo];
    const int j = (int)(row - u.dst_row0);
    int64_t src;
    if (ragged) {  // ragged K/V: key j of the request is row kv_base + j
      src = ((int64_t)(u.kv_base + j) * hk + h) * d;
    } else {
      const int page = kv_indices[u.kv_base + j / P];
      const int slot = j % P;
      src = (int64_t)page * page_stride;
      src += layout == PKA_NHD ? ((int64_t)slot * hk + h) * d : ((int64_t)h * P + slot) * d;
    }
    src += c * 16;
    const int64_t dst = (row * hk + h) * d + c * 16;
    const uint4 kc = *reinterpret_cast<const uint4*>(k8 + src);
    const uint4 vc = *reinterpret_cast<const uint4*>(v8 + src);
    const uint32_t kw[4] = {kc.x, kc.y, kc.z, kc.w}, vw[4] = {vc.x, vc.y, vc.z, vc.w};
    uint32_t ko[8], vo[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      ko[2 * i] = e4m3x2_to_bf16x2(kw[i] & 0xffffu);
      ko[2 * i + 1] = e4m3x2_to_bf16x2(kw[i] >> 16);
      vo[2 * i] = e4m3x2_to_bf16x2(vw[i] & 0xffffu);
      vo[2 * i + 1] = e4m3x2_to_bf16x2(vw[i] >> 16);
    }
    uint4* dk = reinterpret_cast<uint4*>(out_k + dst);
    uint4* dv = reinterpret_cast<uint4*>(out_v + dst);
    dk[0] = make_uint4(ko[0], ko[1], ko[2], ko[3]);
    dk[1] = make_uint4(ko[4], ko[5], ko[6], ko[7]);
    dv[0] = make_uint4(vo[0], vo[1], vo[2], vo[3]);
    dv[1] = make_uint4(vo[4], vo[5], vo[6], vo[7]);
  }
}

// Self-test of the bounded barrier waits: warps 0 and 1 wait with the
// warp-wide wait, lane 0 of warp 2 with the single-thread wait, all on one
// mbarrier of count 1 and with `polls` polls.  With `arrive` set, lane 0 of
// warp 1 arrives first and no wait runs out; otherwise nothing arrives, every
// wait gives up, and the kernel records PKA_ERR_DEVICE_TIMEOUT as the real
// kernels do, then returns.
__global__ void __launch_bounds__(96) wait_selftest_kernel(int arrive, uint32_t polls,
                                                           int32_t* err) {
  __shared__ uint64_t bar;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (arrive && threadIdx.x == 32) mbar_arrive(smem_u32(&bar));
  bool ok = true;
  if (warp < 2)
    ok = mbar_wait_warp(smem_u32(&bar), 0, polls);
  else if (lane == 0)
    ok = mbar_wait(smem_u32(&bar), 0, polls);
  if (!ok && err) atomicExch(err, (int32_t)PKA_ERR_DEVICE_TIMEOUT);
}

// Grid of a grid-stride kernel: enough blocks for the work, at most 32 per
// multiprocessor of the current device.
int grid_for(int64_t work, int block) {
  int64_t g = (work + block - 1) / block;
  int sms = current_device_sms();
  const int64_t cap = 32 * (int64_t)(sms > 0 ? sms : 1);
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int tasks = a.tasks ? a.num_tasks : a.rows * a.heads;
  if (tasks <= 0) return cudaSuccess;
  const int blocks = grid_for(tasks, 8);
  if (a.head_dim == 128)
    merge_kernel<128><<<blocks, 256, 0, stream>>>(a);
  else
    merge_kernel<64><<<blocks, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const PkaDequantUnit* units, int n_units, int64_t rows,
                           const int32_t* counts,
                           const int32_t* kv_indices, const void* k8, const void* v8,
                           int64_t page_stride, int page_size, int layout, int ragged, int hk,
                           int d, uint16_t* out_k, uint16_t* out_v, cudaStream_t stream) {
  if (n_units <= 0 || rows <= 0) return cudaSuccess;
  const int64_t work = rows * hk * (d / 16);
  dequant_kernel<<<grid_for(work, 256), 256, 0, stream>>>(
      units, n_units, rows, counts, kv_indices, static_cast<const uint8_t*>(k8),
      static_cast<const uint8_t*>(v8), page_stride, page_size, layout, ragged, hk, d, out_k,
      out_v);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int arrive, int polls, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 96, 0, stream>>>(arrive, (uint32_t)polls, device_error_word());
  return cudaGetLastError();
}

cudaError_t launch_packbits(const uint8_t* in, int64_t n, uint8_t* out, cudaStream_t stream) {
  packbits_kernel<<<grid_for((n + 7) / 8, 256), 256, 0, stream>>>(in, n, out);
  return cudaGetLastError();
}

cudaError_t launch_append(const pka_params& p, int32_t batch, const uint16_t* k_new,
                          const uint16_t* v_new, const int32_t* append_indptr, int64_t nnz,
                          const int32_t* kv_indptr, const int32_t* kv_indices,
                          const int32_t* last_page_len, void* k, void* v,
                          int64_t page_stride, cudaStream_t stream) {
  const int64_t threads = nnz * 32;  // one warp per appended row
  const float ks = p.k_scale > 0.f ? p.k_scale : 1.f, vs = p.v_scale > 0.f ? p.v_scale : 1.f;
  // reciprocal of a power-of-two scale (exact), else 0: divide
  auto pow2_inv = [](float s) {
    int e = 0;
    return std::frexp(s, &e) == 0.5f ? std::ldexp(1.0f, 1 - e) : 0.f;
  };
  if (p.kv_dtype == PKA_KV_FP8_E4M3)
    append_kernel<true><<<grid_for(threads, 256), 256, 0, stream>>>(
        k_new, v_new, append_indptr, batch, nnz, kv_indptr, kv_indices, last_page_len, k, v,
        page_stride, p.num_kv_heads, p.head_dim, p.page_size, p.layout, ks, vs, pow2_inv(ks),
        pow2_inv(vs));
  else
    append_kernel<false><<<grid_for(threads, 256), 256, 0, stream>>>(
        k_new, v_new, append_indptr, batch, nnz, kv_indptr, kv_indices, last_page_len, k, v,
        page_stride, p.num_kv_heads, p.head_dim, p.page_size, p.layout, 1.f, 1.f, 1.f, 1.f);
  return cudaGetLastError();
}

}  // namespace pka
