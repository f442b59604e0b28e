// Decode attention (one query row per request) over a paged KV cache.
//
// Bandwidth-bound path ("Deep Dive - FlashInfer", "Ragged prefill and paged
// decode": decode reads a long history per query).  One persistent CTA per
// SM walks its share of (request, key range) items from the plan.  A
// producer warp streams 16-key tiles of K and V for all kv heads of the CTA
// into shared memory with bulk async copies (one copy per key row, completion
// counted on an mbarrier); each key row is padded by 16 bytes so that the
// eight rows an ldmatrix reads fall in eight different bank groups.
//
// One consumer warp serves one kv head and all g query heads that read it
// ("GQA head grouping": every K/V byte comes from HBM once).  The g <= 8
// query heads are the N = 8 side of warp-level tensor-core MMAs
// (mma.sync m16n8k16, bf16 in, fp32 accumulate):
//   S^T[16 keys x 8 heads]  = K[16 x D] . Q^T[D x 8]
//   online softmax in fp32 on the accumulator fragments (max over keys with
//   warp shuffles, exp2 of the scores multiplied by scale * log2 e)
//   O^T[D x 8 heads]       += V^T[D x 16 keys] . P^T[16 keys x 8]
// P^T comes from the S^T fragments by an in-register 8x8 transpose
// (movmatrix).  A CTA writes the final bf16 output and base-2 LSE of a
// request, or, when the plan split the request, a normalised fp32 partial
// state for the merge kernel.
//
// HND pages of 8 or a multiple of 16 slots take a second staging layout: each
// kv head's 16 keys arrive by TMA as [16 rows x 128 B] blocks with the
// 128-byte swizzle (16-byte chunk c of row r stored at chunk c ^ (r & 7)),
// and the ldmatrix addresses follow the swizzle; rows of a partial page are
// gathered with 16-byte cp.async into the same layout.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "pka_internal.h"
#include "tc_device.cuh"

namespace pka {
namespace {

constexpr int TS = kDecodeTileTokens;  // keys per stage = one m16 MMA block
constexpr int kMaxStages = 4;
constexpr int kStageBudget = 200 * 1024;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

struct Bars {
  uint64_t* base;
  int stages;
  __device__ uint32_t full(int s) const { return smem_u32(base + s); }
  __device__ uint32_t empty(int s) const { return smem_u32(base + stages + s); }
};

// Bytes of one key row in a stage: the CTA's kv heads, plus 16 bytes of pad.
__host__ __device__ constexpr int row_bytes(int hpc, int D) { return hpc * D * 2 + 16; }

// Swizzled staging: one [16 keys x 64 dims] block is 2 KiB.
constexpr int SWZ_BLK = TS * 128;

struct DecodeMaps {
  CUtensorMap k;  // HND pool {D, P, Hk, pages}, box {64, min(P, 16), 1, 1}
  CUtensorMap v;
};

// Tiles start at multiples of 16 keys inside a request (the planner cuts
// there) or at page boundaries, so with P = 8 or P a multiple of 16 every
// box of min(P, 16) rows stays inside one page.
__host__ __device__ inline bool use_swizzled(int layout, int P, int ragged) {
  return layout == PKA_HND && !ragged && (P == 8 || P % 16 == 0);
}

__device__ __forceinline__ void record_timeout(int32_t* err, volatile int* abort_flag) {
  *abort_flag = 1;
  if (err) atomicExch(err, (int32_t)PKA_ERR_DEVICE_TIMEOUT);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// d += a . b for a 16x16 (row) and 16x8 (col) bf16 fragment pair.
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Issue the bulk copies of keys [a0, a0 + n) of item w (K and V) into a stage.
template <int D>
__device__ __forceinline__ void issue_tile_copies(const AttnArgs& a, const PkaWorkItem& w,
                                                  int a0, int n, int hpc, uint32_t dK,
                                                  uint32_t dV, uint32_t bar, int lane) {
  const int Hk = a.num_kv_heads;
  const int P = a.page_size;
  const int RS = row_bytes(hpc, D);
  const int64_t row = (int64_t)Hk * D;  // elements of one token across all kv heads
  const bool head_major = a.layout == PKA_HND && P > 1 && !a.kv_ragged;
  if (!head_major) {
    // one copy per key row (NHD page, ragged row, or a one-token HND page)
    const int t = lane & 15;
    if (t >= n) return;
    const int j = a0 + t;
    int64_t off;
    if (a.kv_ragged) {
      off = (int64_t)(w.kv_base + j) * row;
    } else {
      const int page = a.kv_indices[w.kv_base + j / P];
      off = (int64_t)page * a.page_stride + (int64_t)(j % P) * row;
    }
    off += (int64_t)w.kv_head0 * D;
    if (lane < 16)
      bulk_g2s(dK + t * RS, a.k + off, (uint32_t)(hpc * D * 2), bar);
    else
      bulk_g2s(dV + t * RS, a.v + off, (uint32_t)(hpc * D * 2), bar);
    return;
  }
  // HND page [Hk, P, D]: one copy per (key, kv head, K or V)
  for (int x = lane; x < n * hpc * 2; x += 32) {
    const int kv = x & 1, h = (x >> 1) % hpc, t = (x >> 1) / hpc;
    const int j = a0 + t;
    const int page = a.kv_indices[w.kv_base + j / P];
    const int64_t off =
        (int64_t)page * a.page_stride + ((int64_t)(w.kv_head0 + h) * P + (j % P)) * D;
    const uint32_t d = (kv ? dV : dK) + t * RS + h * D * 2;
    bulk_g2s(d, (kv ? a.v : a.k) + off, (uint32_t)(D * 2), bar);
  }
}

// Swizzled staging of keys [a0, a0 + n) (a0 is a multiple of 16): whole
// boxes of R = min(P, 16) rows by TMA, the rest gathered with cp.async.
// Rows of a tile of n keys that arrive by TMA (for expect_tx).
__device__ __forceinline__ int swz_tma_rows(int P, int n) {
  const int R = P < TS ? P : TS;
  return (n / R) * R;
}

template <int D>
__device__ __forceinline__ void issue_tile_swizzled(const AttnArgs& a, const DecodeMaps& maps,
                                                    const PkaWorkItem& w, int a0, int n, int hpc,
                                                    uint32_t dK, uint32_t dV, uint32_t bar,
                                                    int lane) {
  constexpr int NB = D / 64;
  const int P = a.page_size;
  const int R = P < TS ? P : TS;
  const int full_rows = (n / R) * R;
  // TMA: box i covers tile rows [i R, (i + 1) R) of one kv head and one 64-dim block
  const int nbox = full_rows / R;
  for (int x = lane; x < nbox * hpc * NB * 2; x += 32) {
    const int kv = x & 1, c = (x >> 1) % NB, h = ((x >> 1) / NB) % hpc, i = (x >> 1) / NB / hpc;
    const int j = a0 + i * R;
    const int page = a.kv_indices[w.kv_base + j / P];
    const uint32_t dst = (kv ? dV : dK) + (h * NB + c) * SWZ_BLK + i * R * 128;
    tc::tma_load_4d(dst, kv ? &maps.v : &maps.k, c * 64, j % P, w.kv_head0 + h, page, bar);
  }
  // cp.async: rows [full_rows, n), 16-byte chunks, swizzled by hand
  constexpr int CH = D / 8;
  const int rest = n - full_rows;
  for (int x = lane; x < rest * hpc * CH * 2; x += 32) {
    const int kv = x & 1, ch = (x >> 1) % CH, h = ((x >> 1) / CH) % hpc;
    const int r = full_rows + (x >> 1) / CH / hpc;
    const int j = a0 + r;
    const int page = a.kv_indices[w.kv_base + j / P];
    const int64_t off = (int64_t)page * a.page_stride +
                        ((int64_t)(w.kv_head0 + h) * P + (j % P)) * D + ch * 8;
    const uint32_t dst = (kv ? dV : dK) + (h * NB + ch / 8) * SWZ_BLK + r * 128 +
                         (((ch % 8) ^ (r & 7)) * 16);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                 "l"((kv ? a.v : a.k) + off)
                 : "memory");
  }
}

template <int D>
__global__ void __launch_bounds__(288, 1)
    decode_kernel(const __grid_constant__ DecodeMaps maps, const AttnArgs a, const int stages) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ volatile int abort_flag;
  constexpr int KS = D / 16;  // k-steps of the QK^T product
  constexpr int MT = D / 16;  // 16-dim blocks of the P V product
  const int hpc = a.heads_per_cta;
  const int G = a.num_qo_heads / a.num_kv_heads;
  const int n_cons = hpc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool swz = use_swizzled(a.layout, a.page_size, a.kv_ragged);
  const int RS = row_bytes(hpc, D);
  const int stage_bytes = swz ? hpc * (D / 64) * SWZ_BLK : TS * RS;
  uint8_t* sK = smem;
  uint8_t* sV = smem + stages * stage_bytes;
  const Bars bars{reinterpret_cast<uint64_t*>(smem + 2 * stages * stage_bytes), stages};

  const int i0 = a.cta_ptr[blockIdx.x], i1 = a.cta_ptr[blockIdx.x + 1];
  if (i0 >= i1) return;  // an empty CTA of a fixed (graph mode) grid
  // Rows of a partial tile that no copy writes must hold finite values (their
  // P is 0, and 0 * NaN would poison O): zero the stages once.
  for (int x = threadIdx.x; x < 2 * stages * stage_bytes / 16; x += blockDim.x)
    reinterpret_cast<uint4*>(smem)[x] = make_uint4(0, 0, 0, 0);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bars.full(s), 33);  // expect_tx by lane 0 + the 32 producer lanes
      mbar_init(bars.empty(s), n_cons);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == n_cons) {
    // ---------------- producer warp ----------------
    uint32_t it = 0;
    for (int ii = i0; ii < i1 && !abort_flag; ++ii) {
      const PkaWorkItem w = a.items[ii];
      for (int a0 = w.t0; a0 < w.t1; a0 += TS, ++it) {
        const int s = it % stages;
        if (!mbar_wait(bars.empty(s), ((it / stages) & 1) ^ 1)) {
          record_timeout(a.err, &abort_flag);
          break;
        }
        const int n = min(TS, w.t1 - a0);
        const int tx_rows = swz ? swz_tma_rows(a.page_size, n) : n;
        if (lane == 0) mbar_arrive_expect_tx(bars.full(s), (uint32_t)(2 * tx_rows * hpc * D * 2));
        __syncwarp();
        if (swz) {
          issue_tile_swizzled<D>(a, maps, w, a0, n, hpc, smem_u32(sK + s * stage_bytes),
                                 smem_u32(sV + s * stage_bytes), bars.full(s), lane);
          // gathered rows are generic-proxy writes: land, fence, then arrive
          asm volatile("cp.async.wait_all;" ::: "memory");
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        } else {
          issue_tile_copies<D>(a, w, a0, n, hpc, smem_u32(sK + s * stage_bytes),
                               smem_u32(sV + s * stage_bytes), bars.full(s), lane);
        }
        mbar_arrive(bars.full(s));
      }
    }
    // Drain: every issued tile's copies must land before the CTA leaves.
    const uint32_t first = it > (uint32_t)stages ? it - stages : 0;
    for (uint32_t k = first; k < it; ++k)
      if (!mbar_wait(bars.full(k % stages), (k / stages) & 1)) record_timeout(a.err, &abort_flag);
    return;
  }
  if (warp > n_cons) return;

  // ---------------- consumer warps: warp hl serves kv head kv_head0 + hl ----------------
  const int hl = warp;
  const int qd = lane & 3;    // thread in quad: heads 2qd, 2qd + 1 of S^T
  const int grp = lane >> 2;  // group: key row of S^T; head of the Q^T / P^T fragments
  const int Hq = a.num_qo_heads;
  // ldmatrix row addresses (bytes inside a stage) of this lane
  const int mi = lane >> 3, mr = lane & 7;
  const uint32_t k_lane = (uint32_t)((mr + 8 * (mi & 1)) * RS + hl * D * 2 + 16 * (mi >> 1));
  const uint32_t v_lane = (uint32_t)((mr + 8 * (mi >> 1)) * RS + hl * D * 2 + 16 * (mi & 1));
  // swizzled staging: chunk c (16 bytes) of key row r of kv head hl
  const uint32_t hb = (uint32_t)(hl * (D / 64) * SWZ_BLK);
  const int k_key = mr + 8 * (mi & 1), v_key = mr + 8 * (mi >> 1);
  auto swz_addr = [&](int key, int c) -> uint32_t {
    return hb + (uint32_t)((c >> 3) * SWZ_BLK + key * 128 + (((c & 7) ^ (key & 7)) << 4));
  };
  const uint32_t sK0 = smem_u32(sK), sV0 = smem_u32(sV);
  const float sc = a.scale_log2;
  uint32_t it = 0;
  for (int ii = i0; ii < i1 && !abort_flag; ++ii) {
    const PkaWorkItem w = a.items[ii];
    const int head_base = (w.kv_head0 + hl) * G;  // first qo head of this kv head
    // Q^T fragments (k = dims, n = heads): head grp, dims 16ks + 2qd (+1, +8, +9)
    uint32_t qf[KS][2];
    {
      const bool real = grp < G;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          a.q + ((int64_t)w.q_row0 * Hq + head_base + (real ? grp : 0)) * D);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qf[ks][0] = real ? qrow[8 * ks + qd] : 0u;
        qf[ks][1] = real ? qrow[8 * ks + 4 + qd] : 0u;
      }
    }
    float acc[MT][4];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY;  // running max of heads 2qd, 2qd + 1 (log2 units)
    float l0 = 0.f, l1 = 0.f;              // this lane's share of the exp sums
    const int64_t mrow = ((int64_t)w.mask_hi << 32 | (uint32_t)w.mask_lo) +
                         (int64_t)w.q_local0 * w.kv_len;

    for (int a0 = w.t0; a0 < w.t1; a0 += TS, ++it) {
      const int s = it % stages;
      if (!mbar_wait(bars.full(s), (it / stages) & 1)) {
        record_timeout(a.err, &abort_flag);
        break;
      }
      const int n = min(TS, w.t1 - a0);
      const uint32_t kb = sK0 + s * stage_bytes, vb = sV0 + s * stage_bytes;
      // S^T = K . Q^T
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        uint32_t af[4];
        ldsm_x4(kb + (swz ? swz_addr(k_key, 2 * ks + (mi >> 1)) : k_lane + 32 * ks), af);
        mma16816(sacc, af, qf[ks][0], qf[ks][1]);
      }
      // keys grp and grp + 8 of the tile; heads 2qd, 2qd + 1
      bool ok0 = grp < n, ok1 = grp + 8 < n;
      if (a.mask_mode == PKA_MASK_CUSTOM) {
        if (ok0) {
          const int64_t bit = mrow + a0 + grp;
          ok0 = (a.mask[bit >> 3] >> (bit & 7)) & 1;
        }
        if (ok1) {
          const int64_t bit = mrow + a0 + grp + 8;
          ok1 = (a.mask[bit >> 3] >> (bit & 7)) & 1;
        }
      }
      const float s00 = ok0 ? sacc[0] * sc : -INFINITY, s01 = ok0 ? sacc[1] * sc : -INFINITY;
      const float s10 = ok1 ? sacc[2] * sc : -INFINITY, s11 = ok1 ? sacc[3] * sc : -INFINITY;
      float t0 = fmaxf(s00, s10), t1 = fmaxf(s01, s11);
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, off));
        t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, off));
      }
      float al0 = 1.f, al1 = 1.f;
      if (m0 == -INFINITY) {
        m0 = t0;
      } else if (t0 > m0 + kRescaleThreshold) {
        al0 = ex2(m0 - t0);
        m0 = t0;
      }
      if (m1 == -INFINITY) {
        m1 = t1;
      } else if (t1 > m1 + kRescaleThreshold) {
        al1 = ex2(m1 - t1);
        m1 = t1;
      }
      if (al0 != 1.f || al1 != 1.f) {
        l0 *= al0;
        l1 *= al1;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          acc[mt][0] *= al0;
          acc[mt][1] *= al1;
          acc[mt][2] *= al0;
          acc[mt][3] *= al1;
        }
      }
      const float p00 = m0 == -INFINITY ? 0.f : ex2(s00 - m0);
      const float p10 = m0 == -INFINITY ? 0.f : ex2(s10 - m0);
      const float p01 = m1 == -INFINITY ? 0.f : ex2(s01 - m1);
      const float p11 = m1 == -INFINITY ? 0.f : ex2(s11 - m1);
      l0 += p00 + p10;
      l1 += p01 + p11;
      // P^T fragments: transpose the (key x head) 8x8 blocks to (head x key)
      const uint32_t pb0 = transpose8x8(float2_to_bf16x2(p00, p01));
      const uint32_t pb1 = transpose8x8(float2_to_bf16x2(p10, p11));
      // O^T += V^T . P^T
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t af[4];
        ldsm_x4_t(vb + (swz ? swz_addr(v_key, 2 * mt + (mi & 1)) : v_lane + 32 * mt), af);
        mma16816(acc[mt], af, pb0, pb1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.empty(s));
    }
    if (abort_flag) break;

    // Sum the exp shares over the 8 key groups; normalise and write.
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int h = 2 * qd + hh;  // head of this lane's accumulator columns
      if (h >= G) continue;
      const float l = hh ? l1 : l0, m = hh ? m1 : m0;
      const bool any = l > 0.f;
      const float inv = any ? 1.f / l : 0.f;
      const float lse_v = any ? m + log2f(l) : -INFINITY;
      const int head = head_base + h;
      if (w.out_rec < 0) {
        uint16_t* orow = a.o + ((int64_t)w.q_row0 * Hq + head) * D;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const uint32_t pk = float2_to_bf16x2(acc[mt][hh] * inv, acc[mt][2 + hh] * inv);
          orow[16 * mt + grp] = (uint16_t)(pk & 0xffffu);
          orow[16 * mt + grp + 8] = (uint16_t)(pk >> 16);
        }
        if (grp == 0 && a.lse) a.lse[(int64_t)w.q_row0 * Hq + head] = lse_v;
      } else {
        const int rec = w.out_rec + (head - w.kv_head0 * G);
        float* prow = a.part_o + (int64_t)rec * D;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          prow[16 * mt + grp] = acc[mt][hh] * inv;
          prow[16 * mt + grp + 8] = acc[mt][2 + hh] * inv;
        }
        if (grp == 0) a.part_lse[rec] = lse_v;
      }
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// HND page pool {D, P, Hk, pages}: one box = min(P, 16) slots of one kv head
// and 64 dims, 128-byte swizzle.
bool encode_hnd(CUtensorMap* m, const void* base, const AttnArgs& a, int D) {
  auto fn = encode_fn();
  if (!fn) return false;
  const uint64_t P = a.page_size, Hk = a.num_kv_heads;
  cuuint64_t dims[4] = {(cuuint64_t)D, P, Hk, (cuuint64_t)1 << 31};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, P * D * 2, (cuuint64_t)a.page_stride * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)(P < (uint64_t)TS ? P : TS), 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_t(const AttnArgs& a, int num_ctas, cudaStream_t stream) {
  const int hpc = a.heads_per_cta;
  const bool swz = use_swizzled(a.layout, a.page_size, a.kv_ragged);
  DecodeMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (swz && (!encode_hnd(&maps.k, a.k, a, D) || !encode_hnd(&maps.v, a.v, a, D)))
    return cudaErrorInvalidValue;
  const int stage_bytes = 2 * (swz ? hpc * (D / 64) * SWZ_BLK : TS * row_bytes(hpc, D));
  int stages = kStageBudget / stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  // the swizzled blocks need 1024-byte alignment: pad the dynamic allocation
  const size_t smem = 1024 + (size_t)stages * stage_bytes + 2 * stages * sizeof(uint64_t);
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  decode_kernel<D><<<num_ctas, 32 * (hpc + 1), smem, stream>>>(maps, a, stages);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const AttnArgs& a0, int num_ctas, int head_dim, int group,
                          cudaStream_t stream) {
  AttnArgs a = a0;
  a.err = device_error_word();
  (void)group;
  if (head_dim == 128) return launch_t<128>(a, num_ctas, stream);
  return launch_t<64>(a, num_ctas, stream);
}

}  // namespace pka
