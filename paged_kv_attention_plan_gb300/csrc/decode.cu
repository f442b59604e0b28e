// Decode attention (one query row per request) over a paged KV cache.
//
// Bandwidth-bound path ("Deep Dive - FlashInfer", "Ragged prefill and paged
// decode": decode reads a long history per query).  One persistent CTA per
// SM walks its share of (request, key range) items from the plan.  Warp 0
// also acts as producer: it streams 16-key tiles of K and V for all kv heads
// of the CTA into shared memory with bulk async copies (whole NHD pages or runs of
// slots, completion counted on an mbarrier); the consumer warps of a kv head
// (one per pair of its g query heads) serve those heads from each tile, so
// every K/V byte is read from HBM once ("GQA head grouping").  Scores and the online
// softmax run in fp32 on CUDA cores with packed f32x2 FMAs: eight lanes share
// one key (16 dims each), four keys per pass.  A CTA writes the final bf16
// output and base-2 LSE of a request, or, when the plan split the request,
// a normalised fp32 partial state for the merge kernel.
#include "pka_device.cuh"
#include "pka_internal.h"

namespace pka {
namespace {

constexpr int TS = kDecodeTileTokens;
constexpr int kMaxStages = 6;
constexpr int kStageBudget = 200 * 1024;

struct Bars {
  uint64_t* base;
  int stages;
  __device__ uint32_t full(int s) const { return smem_u32(base + s); }
  __device__ uint32_t empty(int s) const { return smem_u32(base + stages + s); }
};

__device__ __forceinline__ void record_timeout(int32_t* err, volatile int* abort_flag) {
  *abort_flag = 1;
  if (err) atomicExch(err, (int32_t)PKA_ERR_DEVICE_TIMEOUT);
}

template <int D>
__device__ __forceinline__ void issue_tile_copies(const AttnArgs& a, const PkaWorkItem& w,
                                                  int a0, int n, int hpc, bool head_major,
                                                  uint32_t dK, uint32_t dV, uint32_t bar,
                                                  int lane) {
  const int Hk = a.num_kv_heads;
  const int P = a.page_size;
  const int64_t row = (int64_t)Hk * D;  // elements of one token across all kv heads
  const int t = lane;
  if (t >= n) return;
  const int j = a0 + t;
  if (a.kv_ragged) {
    if (hpc == Hk) {
      if (t == 0) {
        const int64_t off = (int64_t)(w.kv_base + a0) * row;
        bulk_g2s(dK, a.k + off, (uint32_t)(n * row * 2), bar);
        bulk_g2s(dV, a.v + off, (uint32_t)(n * row * 2), bar);
      }
    } else {
      const int64_t off = (int64_t)(w.kv_base + j) * row + (int64_t)w.kv_head0 * D;
      const uint32_t d = (uint32_t)(t * hpc * D * 2);
      bulk_g2s(dK + d, a.k + off, (uint32_t)(hpc * D * 2), bar);
      bulk_g2s(dV + d, a.v + off, (uint32_t)(hpc * D * 2), bar);
    }
    return;
  }
  const int page = a.kv_indices[w.kv_base + j / P];
  const int slot = j % P;
  const int64_t pg = (int64_t)page * a.page_stride;
  const bool run_start = (t == 0) || (slot == 0);
  if (!head_major) {
    // NHD page [P, Hk, D] (also HND with P == 1, which is byte-identical)
    if (hpc == Hk) {
      if (run_start) {
        const int run = min(P - slot, n - t);
        const int64_t off = pg + (int64_t)slot * row;
        const uint32_t d = (uint32_t)(t * hpc * D * 2);
        bulk_g2s(dK + d, a.k + off, (uint32_t)(run * row * 2), bar);
        bulk_g2s(dV + d, a.v + off, (uint32_t)(run * row * 2), bar);
      }
    } else {
      const int64_t off = pg + (int64_t)slot * row + (int64_t)w.kv_head0 * D;
      const uint32_t d = (uint32_t)(t * hpc * D * 2);
      bulk_g2s(dK + d, a.k + off, (uint32_t)(hpc * D * 2), bar);
      bulk_g2s(dV + d, a.v + off, (uint32_t)(hpc * D * 2), bar);
    }
    return;
  }
  // HND page [Hk, P, D]: stage layout [kv head][TS][D]
  if (!run_start) return;
  const int run = min(P - slot, n - t);
  if (hpc == Hk && P == TS && run == TS) {
    bulk_g2s(dK, a.k + pg, (uint32_t)(Hk * P * D * 2), bar);
    bulk_g2s(dV, a.v + pg, (uint32_t)(Hk * P * D * 2), bar);
    return;
  }
  for (int h = 0; h < hpc; ++h) {
    const int64_t off = pg + ((int64_t)(w.kv_head0 + h) * P + slot) * D;
    const uint32_t d = (uint32_t)((h * TS + t) * D * 2);
    bulk_g2s(dK + d, a.k + off, (uint32_t)(run * D * 2), bar);
    bulk_g2s(dV + d, a.v + off, (uint32_t)(run * D * 2), bar);
  }
}

// Producer cursor over the CTA's (item, 16-key tile) stream.  Warp 0 owns it
// and keeps `stages` tiles in flight; before refilling a slot it waits until
// every consumer warp has released it.
struct Producer {
  int item;
  int a0;
  uint32_t it;
};

template <int D>
__device__ __forceinline__ bool produce_one(const AttnArgs& a, Producer& pr, int i1, int stages,
                                            int hpc, bool head_major, uint16_t* sK, uint16_t* sV,
                                            int stage_elems, const Bars& bars, int lane,
                                            volatile int* abort_flag) {
  while (pr.item < i1) {
    const PkaWorkItem w = a.items[pr.item];
    if (pr.a0 < w.t0) pr.a0 = w.t0;
    if (pr.a0 >= w.t1) {
      ++pr.item;
      pr.a0 = -1;
      continue;
    }
    const int s = pr.it % stages;
    if (!mbar_wait(bars.empty(s), ((pr.it / stages) & 1) ^ 1)) {
      record_timeout(a.err, abort_flag);
      return false;
    }
    const int n = min(TS, w.t1 - pr.a0);
    if (lane == 0) mbar_arrive_expect_tx(bars.full(s), (uint32_t)(2 * n * hpc * D * 2));
    __syncwarp();
    issue_tile_copies<D>(a, w, pr.a0, n, hpc, head_major, smem_u32(sK + s * stage_elems),
                         smem_u32(sV + s * stage_elems), bars.full(s), lane);
    pr.a0 += TS;
    ++pr.it;
    return true;
  }
  return false;
}

template <int D, int GW>
__global__ void __launch_bounds__(512, 1) decode_kernel(const AttnArgs a, const int stages) {
  extern __shared__ __align__(1024) uint8_t smem[];
  __shared__ volatile int abort_flag;
  constexpr int NC = D / 64;  // 64-dim chunks; lane u owns dims c*64 + 8u .. +7
  const int hpc = a.heads_per_cta;
  const int group = a.num_qo_heads / a.num_kv_heads;
  const int wph = group / GW;
  const int n_cons = hpc * wph;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int stage_elems = TS * hpc * D;
  uint16_t* sK = reinterpret_cast<uint16_t*>(smem);
  uint16_t* sV = sK + stages * stage_elems;
  const Bars bars{reinterpret_cast<uint64_t*>(sV + stages * stage_elems), stages};
  const bool head_major = a.layout == PKA_HND && a.page_size > 1 && !a.kv_ragged;
  const int ts = head_major ? D : hpc * D;  // element stride between keys in a stage
  const int hs = head_major ? TS * D : D;   // element stride between kv heads in a stage

  const int i0 = a.cta_ptr[blockIdx.x], i1 = a.cta_ptr[blockIdx.x + 1];
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bars.full(s), 1);
      mbar_init(bars.empty(s), n_cons);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (warp >= n_cons) return;

  const bool producer = warp == 0;
  Producer prod{i0, -1, 0};
  if (producer)
    for (int k = 0; k < stages; ++k)
      if (!produce_one<D>(a, prod, i1, stages, hpc, head_major, sK, sV, stage_elems, bars, lane,
                          &abort_flag))
        break;

  // ---------------- consumer warps ----------------
  const int hl = warp / wph;     // kv head inside the CTA's block
  const int sub = warp % wph;    // which GW-slice of the group
  const int tg = lane >> 3;      // key of the pass (0..3)
  const int u = lane & 7;        // dim slice
  const int Hq = a.num_qo_heads;
  uint32_t it = 0;
  for (int ii = i0; ii < i1 && !abort_flag; ++ii) {
    const PkaWorkItem w = a.items[ii];
    const int qo_head0 = (w.kv_head0 + hl) * group + sub * GW;
    float2 qf[GW][NC][4];
#pragma unroll
    for (int g = 0; g < GW; ++g)
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const uint4 raw = *reinterpret_cast<const uint4*>(
            a.q + ((int64_t)w.q_row0 * Hq + qo_head0 + g) * D + c * 64 + u * 8);
        const uint32_t wd[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = bf16x2_to_float2(wd[e]);
          qf[g][c][e] = make_float2(f.x * a.scale_log2, f.y * a.scale_log2);
        }
      }
    float m[GW], l[GW];
    float2 acc[GW][NC][4];
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[g][c][e] = make_float2(0.f, 0.f);
    }
    const int64_t mrow = ((int64_t)w.mask_hi << 32 | (uint32_t)w.mask_lo) +
                         (int64_t)w.q_local0 * w.kv_len;

    for (int a0 = w.t0; a0 < w.t1; a0 += TS, ++it) {
      const int s = it % stages;
      if (!mbar_wait(bars.full(s), (it / stages) & 1)) {
        record_timeout(a.err, &abort_flag);
        break;
      }
      const int n = min(TS, w.t1 - a0);
      const uint16_t* kt = sK + s * stage_elems + hl * hs;
      const uint16_t* vt = sV + s * stage_elems + hl * hs;
      float sc[4][GW];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint16_t* krow = kt + (p * 4 + tg) * ts + u * 8;
        float2 part[GW];
#pragma unroll
        for (int g = 0; g < GW; ++g) part[g] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          const uint4 kr = *reinterpret_cast<const uint4*>(krow + c * 64);
          const float2 k0 = bf16x2_to_float2(kr.x), k1 = bf16x2_to_float2(kr.y);
          const float2 k2 = bf16x2_to_float2(kr.z), k3 = bf16x2_to_float2(kr.w);
#pragma unroll
          for (int g = 0; g < GW; ++g) {
            part[g] = __ffma2_rn(qf[g][c][0], k0, part[g]);
            part[g] = __ffma2_rn(qf[g][c][1], k1, part[g]);
            part[g] = __ffma2_rn(qf[g][c][2], k2, part[g]);
            part[g] = __ffma2_rn(qf[g][c][3], k3, part[g]);
          }
        }
#pragma unroll
        for (int g = 0; g < GW; ++g) sc[p][g] = part[g].x + part[g].y;
      }
#pragma unroll
      for (int off = 1; off < 8; off <<= 1)
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
          for (int g = 0; g < GW; ++g) sc[p][g] += __shfl_xor_sync(0xffffffffu, sc[p][g], off);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int t = p * 4 + tg;
        bool ok = t < n;
        if (ok && a.mask_mode == PKA_MASK_CUSTOM) {
          const int64_t bit = mrow + a0 + t;
          ok = (a.mask[bit >> 3] >> (bit & 7)) & 1;
        }
        if (!ok)
#pragma unroll
          for (int g = 0; g < GW; ++g) sc[p][g] = -INFINITY;
      }
      float alpha[GW];
      bool rescale = false;
#pragma unroll
      for (int g = 0; g < GW; ++g) {
        float mt = fmaxf(fmaxf(sc[0][g], sc[1][g]), fmaxf(sc[2][g], sc[3][g]));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 8));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 16));
        const float m_new = fmaxf(m[g], mt);
        alpha[g] = (m_new == -INFINITY || m_new == m[g]) ? 1.f : exp2f(m[g] - m_new);
        rescale |= alpha[g] != 1.f;
        m[g] = m_new;
      }
      if (rescale) {
#pragma unroll
        for (int g = 0; g < GW; ++g) {
          l[g] *= alpha[g];
          const float2 al = make_float2(alpha[g], alpha[g]);
#pragma unroll
          for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[g][c][e] = __fmul2_rn(acc[g][c][e], al);
        }
      }
      float pr[4][GW];
#pragma unroll
      for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int g = 0; g < GW; ++g) {
          pr[p][g] = (m[g] == -INFINITY) ? 0.f : exp2f(sc[p][g] - m[g]);
          l[g] += pr[p][g];
        }
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int t = p * 4 + tg;
        if (t < n) {
          const uint16_t* vrow = vt + t * ts + u * 8;
#pragma unroll
          for (int c = 0; c < NC; ++c) {
            const uint4 vr = *reinterpret_cast<const uint4*>(vrow + c * 64);
            const float2 v0 = bf16x2_to_float2(vr.x), v1 = bf16x2_to_float2(vr.y);
            const float2 v2 = bf16x2_to_float2(vr.z), v3 = bf16x2_to_float2(vr.w);
#pragma unroll
            for (int g = 0; g < GW; ++g) {
              const float2 pp = make_float2(pr[p][g], pr[p][g]);
              acc[g][c][0] = __ffma2_rn(pp, v0, acc[g][c][0]);
              acc[g][c][1] = __ffma2_rn(pp, v1, acc[g][c][1]);
              acc[g][c][2] = __ffma2_rn(pp, v2, acc[g][c][2]);
              acc[g][c][3] = __ffma2_rn(pp, v3, acc[g][c][3]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.empty(s));
      if (producer)
        produce_one<D>(a, prod, i1, stages, hpc, head_major, sK, sV, stage_elems, bars, lane,
                       &abort_flag);
    }
    if (abort_flag) break;

    // Combine the four key groups of the warp (lane bits 3 and 4).
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      l[g] += __shfl_xor_sync(0xffffffffu, l[g], 8);
      l[g] += __shfl_xor_sync(0xffffffffu, l[g], 16);
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          acc[g][c][e].x += __shfl_xor_sync(0xffffffffu, acc[g][c][e].x, 8);
          acc[g][c][e].y += __shfl_xor_sync(0xffffffffu, acc[g][c][e].y, 8);
          acc[g][c][e].x += __shfl_xor_sync(0xffffffffu, acc[g][c][e].x, 16);
          acc[g][c][e].y += __shfl_xor_sync(0xffffffffu, acc[g][c][e].y, 16);
        }
    }
#pragma unroll
    for (int g = 0; g < GW; ++g) {
      if ((g & 3) != tg) continue;
      const int head = qo_head0 + g;
      const bool any = l[g] > 0.f;
      const float inv = any ? 1.f / l[g] : 0.f;
      const float lse_v = any ? m[g] + log2f(l[g]) : -INFINITY;
      if (w.out_rec < 0) {
        uint16_t* orow = a.o + ((int64_t)w.q_row0 * Hq + head) * D + u * 8;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          uint4 pk;
          pk.x = float2_to_bf16x2(acc[g][c][0].x * inv, acc[g][c][0].y * inv);
          pk.y = float2_to_bf16x2(acc[g][c][1].x * inv, acc[g][c][1].y * inv);
          pk.z = float2_to_bf16x2(acc[g][c][2].x * inv, acc[g][c][2].y * inv);
          pk.w = float2_to_bf16x2(acc[g][c][3].x * inv, acc[g][c][3].y * inv);
          *reinterpret_cast<uint4*>(orow + c * 64) = pk;
        }
        if (u == 0 && a.lse) a.lse[(int64_t)w.q_row0 * Hq + head] = lse_v;
      } else {
        const int rec = w.out_rec + (head - w.kv_head0 * group);
        float* prow = a.part_o + (int64_t)rec * D + u * 8;
#pragma unroll
        for (int c = 0; c < NC; ++c) {
          float4* dst = reinterpret_cast<float4*>(prow + c * 64);
          dst[0] = make_float4(acc[g][c][0].x * inv, acc[g][c][0].y * inv,
                               acc[g][c][1].x * inv, acc[g][c][1].y * inv);
          dst[1] = make_float4(acc[g][c][2].x * inv, acc[g][c][2].y * inv,
                               acc[g][c][3].x * inv, acc[g][c][3].y * inv);
        }
        if (u == 0) a.part_lse[rec] = lse_v;
      }
    }
  }
  if (producer) {
    // Every issued tile's copies must land before the CTA leaves.
    const uint32_t first = prod.it > (uint32_t)stages ? prod.it - stages : 0;
    for (uint32_t k = first; k < prod.it; ++k)
      if (!mbar_wait(bars.full(k % stages), (k / stages) & 1)) record_timeout(a.err, &abort_flag);
  }
}

template <int D, int GW>
cudaError_t launch_t(const AttnArgs& a, int num_ctas, int group, cudaStream_t stream) {
  const int hpc = a.heads_per_cta;
  const int n_cons = hpc * (group / GW);
  const int stage_bytes = 2 * TS * hpc * D * 2;
  int stages = kStageBudget / stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  const size_t smem = (size_t)stages * stage_bytes + 2 * stages * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, GW>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_kernel<D, GW><<<num_ctas, 32 * n_cons, smem, stream>>>(a, stages);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const AttnArgs& a0, int num_ctas, int head_dim, int group,
                          cudaStream_t stream) {
  AttnArgs a = a0;
  a.err = device_error_word();
  const int gw = decode_heads_per_warp(group);
  if (head_dim == 128) {
    if (gw == 1) return launch_t<128, 1>(a, num_ctas, group, stream);
    return launch_t<128, 2>(a, num_ctas, group, stream);
  }
  if (gw == 1) return launch_t<64, 1>(a, num_ctas, group, stream);
  return launch_t<64, 2>(a, num_ctas, group, stream);
}

}  // namespace pka
