// Append / prefill attention (qo_len >= 2 rows) on the 5th-generation tensor
// cores: tcgen05.mma with TMEM accumulators, operands staged by TMA.
//
// A work item is (request, kv head, tile of 128/g query tokens, key range).
// The g qo heads of the kv head pack with the tokens into 128 rows
// (row = token * g + head), so one K/V tile serves all of them ("Deep Dive -
// FlashInfer", GPU smoke check: qo head h reads kv head h / g).  Per 128-key
// tile:  S = Q K^T (tcgen05, fp32 in TMEM) -> mask (bottom-right causal
// j <= K - Q + i of "Causality uses logical positions, not page numbers", or
// the packed custom mask of "KV-Cache layouts", "Mask layout (2D Ragged
// Tensor)") -> online softmax in fp32 registers, one row per thread -> P
// (bf16, shared memory) -> O += P V (tcgen05, fp32 in TMEM).  The epilogue
// writes bf16 O and the base-2 LSE, or a normalised fp32 partial state that
// the merge kernel combines ("A worked split-KV example").
//
// Warp roles (192 threads): warps 0-3 softmax and epilogue (thread = row =
// TMEM lane), warp 4 TMA producer, warp 5 TMEM allocator and MMA issuer.
// S is double-buffered in TMEM so that QK^T of tile k+1 overlaps the softmax
// of tile k; K/V tiles use a two-stage ring.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "pka_internal.h"
#include "tc_device.cuh"

namespace pka {
namespace {

constexpr int BM = kPrefillTileRows;  // 128 packed rows
constexpr int BN = kPrefillTileKeys;  // 128 keys
constexpr int STAGES = 2;
constexpr uint32_t BLK = 16384;       // one [128 rows x 128 B] swizzled block
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

struct Maps {
  CUtensorMap q;     // 3-D {D, Hq, nnz_q}, box {64, g, 128/g}
  CUtensorMap kv_k;  // paged: 4-D, box = one whole page; ragged: 3-D, box 128 rows
  CUtensorMap kv_v;
};

struct PrefillParams {
  AttnArgs a;
  int group;
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[STAGES], v_full[STAGES], kv_empty[STAGES];
  uint64_t s_full[2];
  uint64_t p_full, o_done, o_free;
};

__device__ __forceinline__ void fail(const AttnArgs& a, volatile int* abort_flag) {
  *abort_flag = 1;
  if (a.err) atomicExch(a.err, (int32_t)PKA_ERR_DEVICE_TIMEOUT);
}

__device__ __forceinline__ int num_tiles(const PkaWorkItem& w) {
  return w.t1 > w.t0 ? (w.t1 - w.t0 + BN - 1) / BN : 0;
}

// Split of a tile window [kb, vend) into whole pages loaded by TMA and rows
// gathered with cp.async.  TMA takes the pages [p_lo, p_hi) that lie fully
// inside the window when the page size is a multiple of 8 rows (up to 128)
// and the first of them lands on a 1024-byte boundary of the tile (the
// alignment of a 128-byte swizzled TMA destination); the rows before and
// after them ([kb, p_lo*P) and [p_hi*P, vend)) are gathered 16 bytes at a time.
struct TileSplit {
  int p_lo, p_hi;   // TMA pages (empty when p_lo >= p_hi)
  int head_rows;    // cp.async rows at the start of the window
  int tail_start;   // first cp.async row of the tail (relative to kb)
  int nrows;        // vend - kb
};

__device__ __forceinline__ TileSplit split_tile(int P, int kb, int vend) {
  TileSplit t;
  t.nrows = vend - kb;
  t.p_lo = (kb + P - 1) / P;
  t.p_hi = vend / P;
  const bool ok = (P % 8) == 0 && P <= BN && t.p_lo < t.p_hi && ((t.p_lo * P - kb) % 8) == 0;
  if (!ok) {
    t.p_lo = t.p_hi = 0;
    t.head_rows = t.nrows;
    t.tail_start = t.nrows;
  } else {
    t.head_rows = t.p_lo * P - kb;
    t.tail_start = t.p_hi * P - kb;
  }
  return t;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Bytes the TMA part of a tile delivers.
template <int D>
__device__ __forceinline__ uint32_t kv_tile_tma_bytes(const PrefillParams& pp,
                                                      const PkaWorkItem& w, int kb) {
  constexpr int NB = D / 64;
  if (pp.a.kv_ragged) return (uint32_t)BN * 128 * NB;
  const int P = pp.a.page_size;
  const TileSplit t = split_tile(P, kb, min(kb + BN, w.kv_len));
  return (uint32_t)((t.p_hi - t.p_lo) * P) * 128 * NB;
}

// Issue the loads of one 128-key tile of K (or V) for kv head w.kv_head0:
// rows [kb, vend) of the window; rows past vend keep older finite data and
// are masked.  Lanes share the pages and rows of the window.
template <int D>
__device__ __forceinline__ void load_kv_tile(const PrefillParams& pp, const CUtensorMap* map,
                                             const uint16_t* pool, const PkaWorkItem& w, int kb,
                                             uint32_t dst, uint32_t bar, int lane) {
  constexpr int NB = D / 64;
  const AttnArgs& a = pp.a;
  if (a.kv_ragged) {
    if (lane == 0)
#pragma unroll
      for (int c = 0; c < NB; ++c)
        tc::tma_load_3d(dst + c * BLK, map, c * 64, w.kv_head0, w.kv_base + kb, bar);
    return;
  }
  const int P = a.page_size;
  const int Hk = a.num_kv_heads;
  const TileSplit t = split_tile(P, kb, min(kb + BN, w.kv_len));
  const bool nhd = a.layout == PKA_NHD;
  for (int pi = t.p_lo + lane; pi < t.p_hi; pi += 32) {
    const int page = a.kv_indices[w.kv_base + pi];
    const uint32_t d = dst + (uint32_t)(pi * P - kb) * 128;
#pragma unroll
    for (int c = 0; c < NB; ++c) {
      if (nhd)
        tc::tma_load_4d(d + c * BLK, map, c * 64, w.kv_head0, 0, page, bar);
      else
        tc::tma_load_4d(d + c * BLK, map, c * 64, 0, w.kv_head0, page, bar);
    }
  }
  // gathered rows: 16-byte chunks, swizzled by hand (chunk ^ (row & 7))
  constexpr int CH = D / 8;  // 16-byte chunks per row
  const int gathered = t.head_rows + (t.nrows - t.tail_start);
  for (int x = lane; x < gathered * CH; x += 32) {
    const int q = x / CH, ch = x - q * CH;
    const int r = q < t.head_rows ? q : t.tail_start + (q - t.head_rows);
    const int j = kb + r;
    const int pi = j / P;
    const int page = a.kv_indices[w.kv_base + pi];
    const int slot = j - pi * P;
    const int64_t off = (int64_t)page * a.page_stride +
                        (nhd ? ((int64_t)slot * Hk + w.kv_head0) * D
                             : ((int64_t)w.kv_head0 * P + slot) * D) +
                        ch * 8;
    const uint32_t d = dst + (ch / 8) * BLK + r * 128 + (((ch % 8) ^ (r & 7)) * 16);
    cp_async16(d, pool + off);
  }
}

// 128 consecutive mask bits starting at bit `start` (little-endian bit order);
// bits at or past `limit` read as 0 and are never fetched.
__device__ __forceinline__ void load_mask_bits(const uint8_t* mask, int64_t start, int64_t limit,
                                               uint32_t (&bits)[4]) {
  const int64_t byte0 = start >> 3;
  const int sh = (int)(start & 7);
  const int64_t last_byte = limit > start ? (limit - 1) >> 3 : byte0 - 1;
  uint32_t by[17];
#pragma unroll
  for (int b = 0; b < 17; ++b) by[b] = (byte0 + b <= last_byte) ? mask[byte0 + b] : 0u;
#pragma unroll
  for (int wd = 0; wd < 4; ++wd) {
    const uint64_t v = (uint64_t)by[4 * wd] | ((uint64_t)by[4 * wd + 1] << 8) |
                       ((uint64_t)by[4 * wd + 2] << 16) | ((uint64_t)by[4 * wd + 3] << 24) |
                       ((uint64_t)by[4 * wd + 4] << 32);
    bits[wd] = (uint32_t)(v >> sh);
  }
  // clear bits past the limit
  const int64_t keep = limit - start;
#pragma unroll
  for (int wd = 0; wd < 4; ++wd) {
    const int64_t lo = 32 * wd;
    if (keep <= lo) bits[wd] = 0;
    else if (keep < lo + 32) bits[wd] &= (1u << (keep - lo)) - 1u;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ Maps maps, const PrefillParams pp) {
  constexpr int NB = D / 64;
  const AttnArgs& a = pp.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;                              // NB blocks
  uint8_t* sK = sQ + NB * BLK;                     // STAGES x NB blocks
  uint8_t* sV = sK + STAGES * NB * BLK;            // STAGES x NB blocks
  uint8_t* sP = sV + STAGES * NB * BLK;            // 2 blocks (128 keys)
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i0 = a.cta_ptr[blockIdx.x], i1 = a.cta_ptr[blockIdx.x + 1];
  const int G = pp.group;

  // Zero the K/V stages once: rows of a partial tile that no TMA writes must
  // hold finite values (P is 0 there, and 0 * NaN would poison O).
  for (int x = threadIdx.x; x < 2 * STAGES * NB * (int)BLK / 16; x += kThreads)
    reinterpret_cast<uint4*>(sK)[x] = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars.q_full), 1);
    mbar_init(smem_u32(&bars.q_empty), 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 33);  // TMA expect_tx + 32 producer lanes
      mbar_init(smem_u32(&bars.v_full[s]), 33);
      mbar_init(smem_u32(&bars.kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars.s_full[0]), 1);
    mbar_init(smem_u32(&bars.s_full[1]), 1);
    mbar_init(smem_u32(&bars.p_full), BM);
    mbar_init(smem_u32(&bars.o_done), 1);
    mbar_init(smem_u32(&bars.o_free), BM);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  const uint32_t tS = tmem;            // two S buffers: columns [0,128) and [128,256)
  const uint32_t tO = tmem + 256;      // O: columns [256, 256 + D)

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tc::prefetch_tmap(&maps.q);
      tc::prefetch_tmap(&maps.kv_k);
      tc::prefetch_tmap(&maps.kv_v);
    }
    uint32_t kv_it = 0, q_uses = 0;
    for (int ii = i0; ii < i1 && !abort_flag; ++ii) {
      const PkaWorkItem w = a.items[ii];
      const int n = num_tiles(w);
      if (n == 0) continue;
      if (q_uses > 0 && !mbar_wait(smem_u32(&bars.q_empty), (q_uses - 1) & 1)) {
        fail(a, &abort_flag);
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(smem_u32(&bars.q_full), NB * BLK);
#pragma unroll
        for (int c = 0; c < NB; ++c)
          tc::tma_load_3d(smem_u32(sQ + c * BLK), &maps.q, c * 64, w.kv_head0 * G, w.q_row0,
                          smem_u32(&bars.q_full));
      }
      ++q_uses;
      for (int k = 0; k < n; ++k, ++kv_it) {
        const int s = kv_it % STAGES;
        if (kv_it >= STAGES &&
            !mbar_wait(smem_u32(&bars.kv_empty[s]), ((kv_it / STAGES) - 1) & 1)) {
          fail(a, &abort_flag);
          break;
        }
        const int kb = w.t0 + k * BN;
        const uint32_t bytes = kv_tile_tma_bytes<D>(pp, w, kb);
        if (lane == 0) {
          mbar_arrive_expect_tx(smem_u32(&bars.k_full[s]), bytes);
          mbar_arrive_expect_tx(smem_u32(&bars.v_full[s]), bytes);
        }
        __syncwarp();
        load_kv_tile<D>(pp, &maps.kv_k, a.k, w, kb, smem_u32(sK + s * NB * BLK),
                        smem_u32(&bars.k_full[s]), lane);
        load_kv_tile<D>(pp, &maps.kv_v, a.v, w, kb, smem_u32(sV + s * NB * BLK),
                        smem_u32(&bars.v_full[s]), lane);
        // Gathered rows are generic-proxy writes: wait for this lane's copies,
        // make them visible to the tensor cores, then arrive.
        asm volatile("cp.async.wait_all;" ::: "memory");
        tc::fence_proxy_async_smem();
        mbar_arrive(smem_u32(&bars.k_full[s]));
        mbar_arrive(smem_u32(&bars.v_full[s]));
      }
    }
    // Drain: the loads of the last stages must land before the CTA leaves.
    for (uint32_t k = kv_it > STAGES ? kv_it - STAGES : 0; k < kv_it; ++k) {
      const int s = k % STAGES;
      if (!mbar_wait(smem_u32(&bars.k_full[s]), (k / STAGES) & 1) ||
          !mbar_wait(smem_u32(&bars.v_full[s]), (k / STAGES) & 1))
        fail(a, &abort_flag);
    }
    if (q_uses > 0 && !mbar_wait(smem_u32(&bars.q_full), (q_uses - 1) & 1)) fail(a, &abort_flag);
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idO = tc::idesc_bf16_f32(BM, D, false, true);
      uint32_t kv_it = 0, gt = 0, q_uses = 0, o_uses = 0;
      auto pv = [&](uint32_t tile_kv_it, uint32_t tile_gt, bool first) -> bool {
        const int s = tile_kv_it % STAGES;
        if (!mbar_wait(smem_u32(&bars.p_full), tile_gt & 1)) return false;
        if (!mbar_wait(smem_u32(&bars.v_full[s]), (tile_kv_it / STAGES) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t vb = smem_u32(sV + s * NB * BLK);
        const uint32_t pb = smem_u32(sP);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t ad = tc::smem_desc_sw128(pb + (kk / 4) * BLK + (kk % 4) * 32, 16, 1024);
          const uint64_t bd = tc::smem_desc_sw128(vb + kk * 2048, BLK, 1024);
          tc::mma_bf16(tO, ad, bd, idO, (first && kk == 0) ? 0u : 1u);
        }
        tc::mma_commit(smem_u32(&bars.o_done));
        tc::mma_commit(smem_u32(&bars.kv_empty[s]));
        return true;
      };
      for (int ii = i0; ii < i1 && !abort_flag; ++ii) {
        const PkaWorkItem w = a.items[ii];
        const int n = num_tiles(w);
        if (n == 0) continue;
        if (!mbar_wait(smem_u32(&bars.q_full), q_uses & 1)) {
          fail(a, &abort_flag);
          break;
        }
        ++q_uses;
        tc::fence_after_sync();
        const uint32_t qb = smem_u32(sQ);
        bool ok = true;
        for (int k = 0; k < n && ok; ++k) {
          const uint32_t it = kv_it + k;
          const int s = it % STAGES;
          if (!mbar_wait(smem_u32(&bars.k_full[s]), (it / STAGES) & 1)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t kbase = smem_u32(sK + s * NB * BLK);
          const uint32_t dS = tS + ((gt + k) & 1) * BN;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ad = tc::smem_desc_sw128(qb + (kk / 4) * BLK + (kk % 4) * 32, 16, 1024);
            const uint64_t bd = tc::smem_desc_sw128(kbase + (kk / 4) * BLK + (kk % 4) * 32, 16, 1024);
            tc::mma_bf16(dS, ad, bd, idS, kk > 0 ? 1u : 0u);
          }
          tc::mma_commit(smem_u32(&bars.s_full[(gt + k) & 1]));
          if (k >= 1) {
            if (k == 1 && o_uses > 0 && !mbar_wait(smem_u32(&bars.o_free), (o_uses - 1) & 1)) {
              ok = false;
              break;
            }
            ok = pv(it - 1, gt + k - 1, k == 1);
          }
        }
        tc::mma_commit(smem_u32(&bars.q_empty));
        if (ok && n == 1 && o_uses > 0 && !mbar_wait(smem_u32(&bars.o_free), (o_uses - 1) & 1))
          ok = false;
        if (ok) ok = pv(kv_it + n - 1, gt + n - 1, n == 1);
        if (!ok) {
          fail(a, &abort_flag);
          break;
        }
        kv_it += n;
        gt += n;
        ++o_uses;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int row = threadIdx.x;             // 0..127 == TMEM lane
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int i_tok = row / G, g = row % G;
    uint32_t gt = 0;
    for (int ii = i0; ii < i1 && !abort_flag; ++ii) {
      const PkaWorkItem w = a.items[ii];
      const int n = num_tiles(w);
      const int i = w.q_local0 + i_tok;              // query index inside the request
      const int klim = w.kv_len - w.qo_len + i;      // causal: keys <= klim are visible
      const int64_t mrow = ((int64_t)w.mask_hi << 32 | (uint32_t)w.mask_lo) + (int64_t)i * w.kv_len;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int k = 0; k < n; ++k) {
        const uint32_t t = gt + k;
        if (!mbar_wait(smem_u32(&bars.s_full[t & 1]), (t >> 1) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        float x[BN];  // raw scores q.k (scaled below inside the exponent)
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tc::tmem_ld32(tS + (t & 1) * BN + lane_off + c * 32, r);
#pragma unroll
          for (int j = 0; j < 32; ++j) x[c * 32 + j] = __uint_as_float(r[j]);
        }
        tc::tmem_ld_wait();
        const int kb = w.t0 + k * BN;
        int vis_end = w.t1 - kb;  // columns >= vis_end are outside the key range
        if (a.mask_mode == PKA_MASK_CAUSAL) vis_end = min(vis_end, klim - kb + 1);
        uint32_t mbits[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
        if (a.mask_mode == PKA_MASK_CUSTOM)
          load_mask_bits(a.mask, mrow + kb, mrow + min(w.t1, w.kv_len), mbits);
        float mxa[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < BN; ++j) {
          const bool vis = j < vis_end && ((mbits[j >> 5] >> (j & 31)) & 1u);
          x[j] = vis ? x[j] : -INFINITY;
          mxa[j & 3] = fmaxf(mxa[j & 3], x[j]);
        }
        // row max in log2 units (scale > 0 keeps the order)
        const float mx = fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3])) * a.scale_log2;
        float alpha = 1.f;
        if (m == -INFINITY) {
          m = mx;
        } else if (mx > m + kRescaleThreshold) {
          alpha = exp2f(m - mx);
          m = mx;
        }
        const bool rescale = __any_sync(0xffffffffu, alpha != 1.f);
        float suma[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[BN / 2];
        if (m == -INFINITY) {
#pragma unroll
          for (int j = 0; j < BN / 2; ++j) pk[j] = 0u;
        } else {
          const float neg_m = -m;
#pragma unroll
          for (int j = 0; j < BN; j += 2) {
            const float p0 = exp2f(fmaf(x[j], a.scale_log2, neg_m));
            const float p1 = exp2f(fmaf(x[j + 1], a.scale_log2, neg_m));
            suma[(j >> 1) & 3] += p0 + p1;
            pk[j / 2] = float2_to_bf16x2(p0, p1);
          }
        }
        const float sum = (suma[0] + suma[1]) + (suma[2] + suma[3]);
        l = l * alpha + sum;
        // P and O may only change once the previous P V product has finished.
        if (k >= 1) {
          if (!mbar_wait(smem_u32(&bars.o_done), (t - 1) & 1)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          if (rescale) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              tc::tmem_ld32(tO + lane_off + c * 32, r);
              tc::tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
              tc::tmem_st32(tO + lane_off + c * 32, r);
            }
            tc::tmem_st_wait();
          }
        }
        // P row -> shared memory, 128-byte swizzled K-major layout
#pragma unroll
        for (int blk = 0; blk < 2; ++blk)
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            const uint32_t off = blk * BLK + row * 128 + ((ch ^ (row & 7)) * 16);
            *reinterpret_cast<uint4*>(sP + off) =
                make_uint4(pk[blk * 32 + ch * 4 + 0], pk[blk * 32 + ch * 4 + 1],
                           pk[blk * 32 + ch * 4 + 2], pk[blk * 32 + ch * 4 + 3]);
          }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        mbar_arrive(smem_u32(&bars.p_full));
      }
      if (!ok) {
        fail(a, &abort_flag);
        break;
      }
      // ---------------- epilogue
      float o[D];
#pragma unroll
      for (int j = 0; j < D; ++j) o[j] = 0.f;
      if (n > 0) {
        if (!mbar_wait(smem_u32(&bars.o_done), (gt + n - 1) & 1)) {
          fail(a, &abort_flag);
          break;
        }
        tc::fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tc::tmem_ld32(tO + lane_off + c * 32, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) o[c * 32 + j] = __uint_as_float(r[j]);
        }
        tc::fence_before_sync();
        mbar_arrive(smem_u32(&bars.o_free));
      }
      gt += n;
      if (i_tok >= w.q_count) continue;
      const bool any = l > 0.f;
      const float inv = any ? 1.f / l : 0.f;
      const float lse_v = any ? m + log2f(l) : -INFINITY;
      const int head = w.kv_head0 * G + g;
      if (w.out_rec < 0) {
        uint16_t* dst = a.o + ((int64_t)(w.q_row0 + i_tok) * a.num_qo_heads + head) * D;
#pragma unroll
        for (int j = 0; j < D; j += 8) {
          uint4 v;
          v.x = float2_to_bf16x2(o[j] * inv, o[j + 1] * inv);
          v.y = float2_to_bf16x2(o[j + 2] * inv, o[j + 3] * inv);
          v.z = float2_to_bf16x2(o[j + 4] * inv, o[j + 5] * inv);
          v.w = float2_to_bf16x2(o[j + 6] * inv, o[j + 7] * inv);
          *reinterpret_cast<uint4*>(dst + j) = v;
        }
        if (a.lse) a.lse[(int64_t)(w.q_row0 + i_tok) * a.num_qo_heads + head] = lse_v;
      } else {
        const int rec = w.out_rec + i_tok * G + g;
        float* dst = a.part_o + (int64_t)rec * D;
#pragma unroll
        for (int j = 0; j < D; j += 4)
          *reinterpret_cast<float4*>(dst + j) =
              make_float4(o[j] * inv, o[j + 1] * inv, o[j + 2] * inv, o[j + 3] * inv);
        a.part_lse[rec] = lse_v;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch
// ---------------------------------------------------------------------------
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

bool encode(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
            const uint64_t* strides_bytes, const uint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, s, b, e,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_t(const PrefillParams& pp, int num_ctas, int nnz_q, int64_t total_kv,
                     cudaStream_t stream) {
  const AttnArgs& a = pp.a;
  const int G = pp.group;
  const uint64_t Hq = a.num_qo_heads, Hk = a.num_kv_heads;
  Maps maps;
  {
    const uint64_t dims[3] = {(uint64_t)D, Hq, (uint64_t)(nnz_q > 0 ? nnz_q : 1)};
    const uint64_t str[2] = {(uint64_t)D * 2, Hq * D * 2};
    const uint32_t box[3] = {64, (uint32_t)G, (uint32_t)(BM / G)};
    if (!encode(&maps.q, a.q, 3, dims, str, box)) return cudaErrorInvalidValue;
  }
  if (a.kv_ragged) {
    const uint64_t dims[3] = {(uint64_t)D, Hk, (uint64_t)(total_kv > 0 ? total_kv : 1)};
    const uint64_t str[2] = {(uint64_t)D * 2, Hk * D * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)BN};
    if (!encode(&maps.kv_k, a.k, 3, dims, str, box) || !encode(&maps.kv_v, a.v, 3, dims, str, box))
      return cudaErrorInvalidValue;
  } else {
    // One box = one whole page of one kv head.  Pages of other sizes, and
    // partial pages, are gathered with cp.async and never use the map.
    const uint64_t P = a.page_size;
    const uint32_t pb = (P % 8 == 0 && P <= (uint64_t)BN) ? (uint32_t)P : 1u;
    const uint64_t pages = (uint64_t)1 << 31;  // page ids come from kv_indices
    uint64_t dims[4], str[3];
    uint32_t box[4];
    if (a.layout == PKA_NHD) {
      dims[0] = D; dims[1] = Hk; dims[2] = P; dims[3] = pages;
      str[0] = (uint64_t)D * 2; str[1] = Hk * D * 2; str[2] = (uint64_t)a.page_stride * 2;
      box[0] = 64; box[1] = 1; box[2] = pb; box[3] = 1;
    } else {
      dims[0] = D; dims[1] = P; dims[2] = Hk; dims[3] = pages;
      str[0] = (uint64_t)D * 2; str[1] = P * D * 2; str[2] = (uint64_t)a.page_stride * 2;
      box[0] = 64; box[1] = pb; box[2] = 1; box[3] = 1;
    }
    if (!encode(&maps.kv_k, a.k, 4, dims, str, box) || !encode(&maps.kv_v, a.v, 4, dims, str, box))
      return cudaErrorInvalidValue;
  }
  constexpr int NB = D / 64;
  // At least 120 KiB, so that one CTA (and its 512 TMEM columns) owns each SM.
  size_t smem = 1024 + (size_t)(NB + 2 * STAGES * NB + 2) * BLK;
  if (smem < 120 * 1024) smem = 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  prefill_kernel<D><<<num_ctas, kThreads, smem, stream>>>(maps, pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const AttnArgs& a0, int num_ctas, int head_dim, int group,
                           int nnz_q, int64_t total_kv, cudaStream_t stream) {
  PrefillParams pp;
  pp.a = a0;
  pp.a.err = device_error_word();
  pp.group = group;
  if (head_dim == 128) return launch_t<128>(pp, num_ctas, nnz_q, total_kv, stream);
  return launch_t<64>(pp, num_ctas, nnz_q, total_kv, stream);
}

}  // namespace pka
