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
// (bf16, in tensor memory) -> O += P V (tcgen05, fp32 in TMEM).  The
// epilogue writes bf16 O and the base-2 LSE, or a normalised fp32 partial
// state that the merge kernel combines ("A worked split-KV example").
//
// Warp roles (352 threads): warpgroups 0 and 1 run the softmax and epilogue
// of two 128-row query tiles of the same (request, kv head) (thread = row =
// TMEM lane); warp 8 loads Q and the K ring, warp 10 the V ring (TMA page
// boxes and gather4 rows, cp.async for the rest), warp 9 allocates TMEM and
// issues the MMAs (the whole warp runs the issue loop; one elected lane
// issues).  Both query tiles share each K/V tile and the tensor core
// alternates between them, so one tile's MMAs overlap the other tile's
// softmax.  P stays in tensor memory (it overwrites the first half of its S
// tile) and feeds the P V product as the A operand.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "pka_internal.h"
#include "tc_device.cuh"

namespace pka {
namespace {

constexpr int BM = kPrefillTileRows;  // 128 packed rows
constexpr int BN = kPrefillTileKeys;  // 128 keys
// K tiles are released as soon as both QK^T products have read them, V tiles
// only after both P V products, so the K ring runs deeper than the V ring.
template <int D> struct Ring {
  static constexpr int K = D == 128 ? 3 : 4;
  static constexpr int V = D == 128 ? 2 : 4;
};
constexpr uint32_t BLK = 16384;       // one [128 rows x 128 B] swizzled block
// softmax warpgroups 0-1, Q+K producer warp 8, MMA warp 9, V producer warp 10
constexpr int kThreads = 352;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

struct Maps {
  CUtensorMap q;     // 3-D {D, Hq, nnz_q}, box {64, g, 128/g}
  CUtensorMap kv_k;  // paged: 4-D, box = one whole page; ragged: 3-D, box 128 rows
  CUtensorMap kv_v;
  CUtensorMap row_k;  // paged: the pool as 2-D rows of D elements, box {64, 1} (row gathers)
  CUtensorMap row_v;
};

struct PrefillParams {
  AttnArgs a;
  int group;
  int gather;              // 1: rows outside whole-page boxes come by TMA gather4
  int64_t rows_per_page;   // page_stride / D: rows of the 2-D view per page
};

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];  // per query tile
};

// 2^x on the special-function unit (inputs here are <= 8; results below the
// smallest normal flush to 0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

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
// Returns whether this lane issued cp.async copies (generic-proxy writes the
// caller has to wait for and fence before it arrives).
template <int D>
__device__ __forceinline__ bool load_kv_tile(const PrefillParams& pp, const CUtensorMap* map,
                                             const CUtensorMap& maps_row_k,
                                             const CUtensorMap& maps_row_v, const uint16_t* pool,
                                             const PkaWorkItem& w, int kb, uint32_t dst,
                                             uint32_t bar, int lane) {
  constexpr int NB = D / 64;
  const AttnArgs& a = pp.a;
  if (a.kv_ragged) {
    if (lane == 0)
#pragma unroll
      for (int c = 0; c < NB; ++c)
        tc::tma_load_3d(dst + c * BLK, map, c * 64, w.kv_head0, w.kv_base + kb, bar);
    return false;
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
  // Rows outside whole-page boxes.  With the 2-D row maps: one TMA gather4
  // per four rows and 64-column block (each lane one group, its own bytes
  // added to the barrier's count); a short last group repeats its last row
  // (rows past the window hold finite data and are masked).  Without them, or
  // for a group whose row index exceeds the 2-D map, 16-byte cp.async chunks
  // swizzled by hand (chunk ^ (row & 7)).
  constexpr int CH = D / 8;  // 16-byte chunks per row
  bool copied = false;
  auto row_addr = [&](int r, int64_t& off, int64_t& row) {
    const int j = kb + r;
    const int pi = j / P;
    const int page = a.kv_indices[w.kv_base + pi];
    const int slot = j - pi * P;
    const int64_t in_page = nhd ? (int64_t)slot * Hk + w.kv_head0 : (int64_t)w.kv_head0 * P + slot;
    off = (int64_t)page * a.page_stride + in_page * D;
    row = (int64_t)page * pp.rows_per_page + in_page;
  };
  if (pp.gather) {
    const int gh = (t.head_rows + 3) / 4, gt = (t.nrows - t.tail_start + 3) / 4;
    const CUtensorMap* rmap = pool == a.k ? &maps_row_k : &maps_row_v;
    for (int gi = lane; gi < gh + gt; gi += 32) {
      const int r0 = gi < gh ? 4 * gi : t.tail_start + 4 * (gi - gh);
      const int rend = gi < gh ? t.head_rows : t.nrows;
      int64_t off[4], row[4];
      bool fits = true;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        row_addr(min(r0 + q, rend - 1), off[q], row[q]);
        fits = fits && row[q] < ((int64_t)1 << 31);
      }
      if (fits) {
        tc::mbar_expect_tx(bar, (uint32_t)(4 * 128 * NB));
#pragma unroll
        for (int c = 0; c < NB; ++c)
          tc::tma_gather4(dst + c * BLK + r0 * 128, rmap, c * 64, (int)row[0], (int)row[1],
                          (int)row[2], (int)row[3], bar);
      } else {
        for (int q = 0; q < 4 && r0 + q < rend; ++q)
          for (int ch = 0; ch < CH; ++ch) {
            const int r = r0 + q;
            cp_async16(dst + (ch / 8) * BLK + r * 128 + (((ch % 8) ^ (r & 7)) * 16),
                       pool + off[q] + ch * 8);
          }
        copied = true;
      }
    }
    return copied;
  }
  const int gathered = t.head_rows + (t.nrows - t.tail_start);
  for (int x = lane; x < gathered * CH; x += 32) {
    const int q = x / CH, ch = x - q * CH;
    const int r = q < t.head_rows ? q : t.tail_start + (q - t.head_rows);
    int64_t off, row;
    row_addr(r, off, row);
    const uint32_t d = dst + (ch / 8) * BLK + r * 128 + (((ch % 8) ^ (r & 7)) * 16);
    cp_async16(d, pool + off + ch * 8);
    copied = true;
  }
  return copied;
}

// 128 consecutive mask bits starting at bit `start` (little-endian bit order);
// bits at or past `limit` read as 0.  Five aligned 32-bit loads and funnel
// shifts when the mask is 4-byte aligned and the words lie before the limit,
// single bytes otherwise (near the end of the mask).
__device__ __forceinline__ void load_mask_bits(const uint8_t* mask, int64_t start, int64_t limit,
                                               uint32_t (&bits)[4]) {
  const int64_t last_byte = limit > start ? (limit - 1) >> 3 : (start >> 3) - 1;
  const int64_t ab = (start >> 3) & ~int64_t(3);  // aligned byte of the first word
  const int p = (int)(start - ab * 8);            // 0..31
  if ((reinterpret_cast<uintptr_t>(mask) & 3) == 0 && ab + 20 <= last_byte + 1) {
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(mask + ab);
    uint32_t wv[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) wv[i] = __ldg(wp + i);
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) bits[wd] = __funnelshift_r(wv[wd], wv[wd + 1], p);
  } else {
    const int64_t byte0 = start >> 3;
    const int sh = (int)(start & 7);
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

// 32-byte global store (sm_100 family); the address must be 32-byte aligned.
// Each thread of the epilogue writes its own row, so a warp's store touches 32
// rows: 32-byte pieces make every piece a whole sector and halve the count.
__device__ __forceinline__ void st_global_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t a4, uint32_t a5, uint32_t a6,
                                             uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0),
               "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ Maps maps, const PrefillParams pp) {
  constexpr int NB = D / 64;
  const AttnArgs& a = pp.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  constexpr int KS = Ring<D>::K, VS = Ring<D>::V;
  uint8_t* sQ = smem;                // 2 tiles x NB blocks
  uint8_t* sK = sQ + 2 * NB * BLK;   // KS x NB blocks
  uint8_t* sV = sK + KS * NB * BLK;  // VS x NB blocks
  __shared__ Bars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i0 = a.cta_ptr[blockIdx.x], i1 = a.cta_ptr[blockIdx.x + 1];
  if (i0 >= i1) return;  // an empty CTA of a fixed (graph mode) grid: no TMEM, no barriers
  const int G = pp.group;
  const int TQ = BM / G;  // query tokens of one 128-row tile

  // Zero the K/V stages once: rows of a partial tile that no load writes must
  // hold finite values (P is 0 there, and 0 * NaN would poison O).
  for (int x = threadIdx.x; x < (KS + VS) * NB * (int)BLK / 16; x += kThreads)
    reinterpret_cast<uint4*>(sK)[x] = make_uint4(0, 0, 0, 0);
  tc::fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars.q_full), 1);
    mbar_init(smem_u32(&bars.q_empty), 1);
    for (int s = 0; s < KS; ++s) {
      mbar_init(smem_u32(&bars.k_full[s]), 33);  // TMA expect_tx + 32 producer lanes
      mbar_init(smem_u32(&bars.k_empty[s]), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(smem_u32(&bars.v_full[s]), 33);
      mbar_init(smem_u32(&bars.v_empty[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&bars.s_full[x]), 1);
      mbar_init(smem_u32(&bars.p_full[x]), BM);
      mbar_init(smem_u32(&bars.o_done[x]), 1);
      mbar_init(smem_u32(&bars.o_free[x]), BM);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tc::tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base_sh;
  // TMEM columns: S of tile x at [128x, 128x + 128) (P, bf16, reuses its first
  // 64 columns), O of tile x at [256 + 128x, 256 + 128x + D).

  if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ producers
    // warp 8: Q tiles and the K ring; warp 10: the V ring.
    const bool kq = warp == 8;
    const int ns = kq ? KS : VS;
    uint64_t* full = kq ? bars.k_full : bars.v_full;
    uint64_t* empty = kq ? bars.k_empty : bars.v_empty;
    uint8_t* ring = kq ? sK : sV;
    const CUtensorMap* map = kq ? &maps.kv_k : &maps.kv_v;
    const uint16_t* pool = kq ? a.k : a.v;
    if (lane == 0) {
      if (kq) tc::prefetch_tmap(&maps.q);
      tc::prefetch_tmap(map);
    }
    uint32_t it = 0, q_uses = 0;
    for (int ii = i0; ii < i1 && !warp_any(&abort_flag); ++ii) {
      const PkaWorkItem w = a.items[ii];
      const int n = num_tiles(w);
      if (n == 0) continue;
      if (kq) {
        const bool two = w.q_count > TQ;
        if (q_uses > 0 && !mbar_wait_warp(smem_u32(&bars.q_empty), (q_uses - 1) & 1)) {
          fail(a, &abort_flag);
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(smem_u32(&bars.q_full), (two ? 2 : 1) * NB * BLK);
          for (int x = 0; x < (two ? 2 : 1); ++x)
#pragma unroll
            for (int c = 0; c < NB; ++c)
              tc::tma_load_3d(smem_u32(sQ + (x * NB + c) * BLK), &maps.q, c * 64, w.kv_head0 * G,
                              w.q_row0 + x * TQ, smem_u32(&bars.q_full));
        }
        ++q_uses;
      }
      for (int k = 0; k < n; ++k, ++it) {
        const int s = it % ns;
        if (it >= (uint32_t)ns && !mbar_wait_warp(smem_u32(&empty[s]), ((it / ns) - 1) & 1)) {
          fail(a, &abort_flag);
          break;
        }
        const int kb = w.t0 + k * BN;
        const uint32_t bytes = kv_tile_tma_bytes<D>(pp, w, kb);
        if (lane == 0) mbar_arrive_expect_tx(smem_u32(&full[s]), bytes);
        __syncwarp();
        const bool copied =
            load_kv_tile<D>(pp, map, maps.row_k, maps.row_v, pool, w, kb,
                            smem_u32(ring + s * NB * BLK), smem_u32(&full[s]), lane);
        // Rows copied with cp.async are generic-proxy writes: wait for this
        // lane's copies and make them visible to the tensor cores before the
        // arrival.  TMA rows complete on the barrier by themselves.
        if (copied) {
          asm volatile("cp.async.wait_all;" ::: "memory");
          tc::fence_proxy_async_smem();
        }
        mbar_arrive(smem_u32(&full[s]));
      }
    }
    // Drain: the loads of the last stages must land before the CTA leaves.
    for (uint32_t k = it > (uint32_t)ns ? it - ns : 0; k < it; ++k)
      if (!mbar_wait_warp(smem_u32(&full[k % ns]), (k / ns) & 1)) fail(a, &abort_flag);
    if (kq && q_uses > 0 && !mbar_wait_warp(smem_u32(&bars.q_full), (q_uses - 1) & 1))
      fail(a, &abort_flag);
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // Order per key tile k (two query tiles A and B):
    //   PV_A(k), S_A(k+1), PV_B(k), S_B(k+1)
    // so that the tensor core works on one tile while the other tile's
    // softmax runs.  MMAs of one thread execute in issue order, so S_x(k+1)
    // may overwrite the P_x(k) that PV_x(k) reads.
    // The whole warp runs the loop and every value in it is warp-uniform;
    // elect.sync inside each MMA and commit picks the one issuing lane.  (The
    // same loop run by lane 0 alone under a branch issued the MMAs about 20%
    // slower on the append-prefill workload.)
    {
      constexpr uint32_t idS = tc::idesc_bf16_f32(BM, BN, false, false);
      constexpr uint32_t idO = tc::idesc_bf16_f32(BM, D, false, true);
      uint32_t kv_it = 0, q_uses = 0;
      uint32_t uses0 = 0, uses1 = 0, o_uses0 = 0, o_uses1 = 0;  // per query tile
      const bool custom = a.mask_mode == PKA_MASK_CUSTOM;
      bool ok = true;
      // Descriptor bases are built once; each MMA only adds the (constant)
      // start-address offset of its 16-wide K slice, in 16-byte units.
      const uint64_t dq0 = tc::smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint64_t dk0 = tc::smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint64_t dv0 = tc::smem_desc_sw128(smem_u32(sV), BLK, 1024);
      auto issue_s = [&](int x, uint32_t it) {
        const uint64_t ad = dq0 + (uint64_t)((x * NB * BLK) >> 4);
        const uint64_t bd = dk0 + (uint64_t)(((it % KS) * NB * BLK) >> 4);
        const uint32_t d = tmem + x * 128;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t off = (uint64_t)(((kk / 4) * BLK + (kk % 4) * 32) >> 4);
          tc::mma_bf16_elect(d, ad + off, bd + off, idS, kk > 0 ? 1u : 0u);
        }
        tc::mma_commit_elect(smem_u32(&bars.s_full[x]));
      };
      auto issue_pv = [&](int x, uint32_t it, bool first) {
        const uint64_t bd = dv0 + (uint64_t)(((it % VS) * NB * BLK) >> 4);
        const uint32_t d = tmem + 256 + x * 128, pa = tmem + x * 128;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          tc::mma_bf16_ts_elect(d, pa + kk * 8, bd + (uint64_t)((kk * 2048) >> 4), idO,
                                (first && kk == 0) ? 0u : 1u);
        tc::mma_commit_elect(smem_u32(&bars.o_done[x]));
      };
      for (int ii = i0; ii < i1 && ok && !warp_any(&abort_flag); ++ii) {
        const PkaWorkItem w = a.items[ii];
        const int n = num_tiles(w);
        if (n == 0) continue;
        const int nx = w.q_count > TQ ? 2 : 1;
        ok = mbar_wait_warp(smem_u32(&bars.q_full), q_uses & 1);
        ++q_uses;
        if (ok) ok = mbar_wait_warp(smem_u32(&bars.k_full[kv_it % KS]), (kv_it / KS) & 1);
        if (!ok) break;
        tc::fence_after_sync();
        for (int x = 0; x < nx; ++x) issue_s(x, kv_it);
        tc::mma_commit_elect(smem_u32(&bars.k_empty[kv_it % KS]));
        for (int k = 0; k < n && ok; ++k) {
          const uint32_t it = kv_it + k;
          for (int x = 0; x < nx && ok; ++x) {
            const uint32_t ux = x ? uses1 : uses0, ox = x ? o_uses1 : o_uses0;
            // With a custom mask the softmax is the longer step: the V and K
            // stages are awaited while the warp waits for P anyway, so that
            // only P's wait stands between the softmax and the P V product
            // (+4% on the ragged custom-mask workload; -1.5% when taken for
            // causal batches, whose next K stage is sometimes still loading).
            const bool kv_first = custom && x == 0;
            if (kv_first) {
              if (k == 0 && ox > 0) ok = mbar_wait_warp(smem_u32(&bars.o_free[x]), (ox - 1) & 1);
              if (ok) ok = mbar_wait_warp(smem_u32(&bars.v_full[it % VS]), (it / VS) & 1);
              if (ok && k + 1 < n)
                ok = mbar_wait_warp(smem_u32(&bars.k_full[(it + 1) % KS]), ((it + 1) / KS) & 1);
              if (ok) ok = mbar_wait_warp(smem_u32(&bars.p_full[x]), (ux + k) & 1);
            } else {
              ok = mbar_wait_warp(smem_u32(&bars.p_full[x]), (ux + k) & 1);
              if (ok && k == 0 && ox > 0)
                ok = mbar_wait_warp(smem_u32(&bars.o_free[x]), (ox - 1) & 1);
              if (ok && x == 0) ok = mbar_wait_warp(smem_u32(&bars.v_full[it % VS]), (it / VS) & 1);
            }
            if (!ok) break;
            tc::fence_after_sync();
            issue_pv(x, it, k == 0);
            if (k + 1 < n) {
              if (x == 0 && !kv_first) {
                ok = mbar_wait_warp(smem_u32(&bars.k_full[(it + 1) % KS]), ((it + 1) / KS) & 1);
                if (!ok) break;
                tc::fence_after_sync();
              }
              issue_s(x, it + 1);
              if (x == nx - 1) tc::mma_commit_elect(smem_u32(&bars.k_empty[(it + 1) % KS]));
            }
          }
          tc::mma_commit_elect(smem_u32(&bars.v_empty[it % VS]));
        }
        tc::mma_commit_elect(smem_u32(&bars.q_empty));
        uses0 += n;
        o_uses0 += 1;
        if (nx == 2) {
          uses1 += n;
          o_uses1 += 1;
        }
        kv_it += n;
      }
      if (!ok) fail(a, &abort_flag);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int x = warp >> 2;                 // query tile of this warpgroup
    const int row = threadIdx.x & (BM - 1);  // TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + x * 128 + lane_off;
    const uint32_t tO = tmem + 256 + x * 128 + lane_off;
    const int i_tok = x * TQ + row / G, g = row % G;
    const float sc = a.scale_log2;
    uint32_t uses = 0;
    for (int ii = i0; ii < i1 && !warp_any(&abort_flag); ++ii) {
      const PkaWorkItem w = a.items[ii];
      if (x == 1 && w.q_count <= TQ) continue;  // no second tile in this item
      const int n = num_tiles(w);
      const int i = w.q_local0 + i_tok;              // query index inside the request
      const int klim = w.kv_len - w.qo_len + i;      // causal: keys <= klim are visible
      const int klim_first = w.kv_len - w.qo_len + w.q_local0 + x * TQ;
      const int64_t mrow = ((int64_t)w.mask_hi << 32 | (uint32_t)w.mask_lo) + (int64_t)i * w.kv_len;
      const int mm = (w.flags & PKA_ITEM_ALL_VISIBLE) ? (int)PKA_MASK_NONE : a.mask_mode;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int k = 0; k < n; ++k) {
        const int kb = w.t0 + k * BN;
        // Custom-mask words are read before the wait on S, so that their
        // global-memory latency overlaps the tile's MMAs.
        uint32_t mbits[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
        if (mm == PKA_MASK_CUSTOM)
          load_mask_bits(a.mask, mrow + kb, mrow + min(w.t1, w.kv_len), mbits);
        if (!mbar_wait_warp(smem_u32(&bars.s_full[x]), (uses + k) & 1)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        // Only tiles that reach past the key range, the causal diagonal of the
        // warpgroup's first row, or a custom mask with a cleared bit in this
        // row need per-element masking.
        const bool need_mask =
            (kb + BN > w.t1) ||
            (mm == PKA_MASK_CUSTOM && (mbits[0] & mbits[1] & mbits[2] & mbits[3]) != 0xffffffffu) ||
            (mm == PKA_MASK_CAUSAL && kb + BN - 1 > klim_first);
        int vis_end = w.t1 - kb;
        if (mm == PKA_MASK_CAUSAL) vis_end = min(vis_end, klim - kb + 1);
        // The whole S row in one round trip (four 32-column loads, one wait):
        // under tensor-core traffic a TMEM load takes hundreds of cycles, so
        // one exposed latency per tile instead of one per chunk.
        uint32_t r[BN / 32][32];
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) tc::tmem_ld32(tS + c * 32, r[c]);
        tc::tmem_ld_wait();
        if (need_mask) {
          // fold the end of the visible range into the bits, then one bit
          // test per score
#pragma unroll
          for (int c = 0; c < BN / 32; ++c) {
            const int rem = vis_end - 32 * c;
            if (rem <= 0) mbits[c] = 0u;
            else if (rem < 32) mbits[c] &= (1u << rem) - 1u;
          }
#pragma unroll
          for (int c = 0; c < BN / 32; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (!(mbits[c] & (1u << j))) r[c][j] = __float_as_uint(-INFINITY);
        }
        float mxa[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < BN / 32; ++c)
#pragma unroll
          for (int j = 0; j < 32; j += 2)
            mxa[(j >> 1) & 3] =
                max3(mxa[(j >> 1) & 3], __uint_as_float(r[c][j]), __uint_as_float(r[c][j + 1]));
        const float mx = fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3])) * sc;
        float alpha = 1.f;
        if (m == -INFINITY) {
          m = mx;
        } else if (mx > m + kRescaleThreshold) {
          alpha = exp2f(m - mx);
          m = mx;
        }
        // probabilities (masked scores are -inf and give 0) -> P, bf16, packed
        // in place over the consumed scores and stored over the first 64
        // columns of S
        // With m = -inf every score of the row so far is -inf (masked), and
        // -inf * scale + 0 = -inf gives p = ex2(-inf) = 0 with no select (the
        // scale is positive).
        float2 sum2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        const bool none = m == -INFINITY;
        const float neg_m = none ? 0.f : -m;
        const float2 sc2 = make_float2(sc, sc), negm2 = make_float2(neg_m, neg_m);
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 t2 = __ffma2_rn(
                make_float2(__uint_as_float(r[c][j]), __uint_as_float(r[c][j + 1])), sc2, negm2);
            const float p0 = ex2(t2.x);
            const float p1 = ex2(t2.y);
            sum2[(j >> 1) & 1] = __fadd2_rn(sum2[(j >> 1) & 1], make_float2(p0, p1));
            r[c][j / 2] = float2_to_bf16x2(p0, p1);
          }
          tc::tmem_st16(tS + c * 16, *reinterpret_cast<const uint32_t(*)[16]>(&r[c][0]));
        }
        l = l * alpha + ((sum2[0].x + sum2[0].y) + (sum2[1].x + sum2[1].y));
        // O of the earlier key tiles is final here: S_x(k) was issued after
        // PV_x(k-1), and MMAs complete in order.
        if (k >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tc::tmem_ld32(tO + c * 32, r);
            tc::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__uint_as_float(r[j]) * alpha);
            tc::tmem_st32(tO + c * 32, r);
          }
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        mbar_arrive(smem_u32(&bars.p_full[x]));
      }
      if (!ok) {
        fail(a, &abort_flag);
        break;
      }
      // ---------------- epilogue
      const bool store = i_tok < w.q_count;
      const bool any = l > 0.f;
      const float inv = any ? a.v_scale / l : 0.f;  // V's scale (1 for bf16 K/V)
      const int head = w.kv_head0 * G + g;
      uint16_t* odst = a.o + ((int64_t)(w.q_row0 + i_tok) * a.num_qo_heads + head) * D;
      const int rec = w.out_rec + i_tok * G + g;
      float* pdst = a.part_o + (int64_t)rec * D;
      if (n > 0) {
        if (!mbar_wait_warp(smem_u32(&bars.o_done[x]), (uses + n - 1) & 1)) {
          fail(a, &abort_flag);
          break;
        }
        tc::fence_after_sync();
        // All of O in one round trip; O's columns are free for the next
        // item's PV as soon as the loads complete, before any global store.
        uint32_t r[D / 32][32];
#pragma unroll
        for (int c = 0; c < D / 32; ++c) tc::tmem_ld32(tO + c * 32, r[c]);
        tc::tmem_ld_wait();
        tc::fence_before_sync();
        mbar_arrive(smem_u32(&bars.o_free[x]));
        const bool v8 =
            ((reinterpret_cast<uintptr_t>(a.o) | reinterpret_cast<uintptr_t>(a.part_o)) & 31) == 0;
        if (store && v8) {
          auto cv = [&](int c, int j) {
            return float2_to_bf16x2(__uint_as_float(r[c][j]) * inv,
                                    __uint_as_float(r[c][j + 1]) * inv);
          };
          auto fv = [&](int c, int j) { return __float_as_uint(__uint_as_float(r[c][j]) * inv); };
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            if (w.out_rec < 0) {
#pragma unroll
              for (int j = 0; j < 32; j += 16)
                st_global_v8(odst + c * 32 + j, cv(c, j), cv(c, j + 2), cv(c, j + 4),
                             cv(c, j + 6), cv(c, j + 8), cv(c, j + 10), cv(c, j + 12),
                             cv(c, j + 14));
            } else {
#pragma unroll
              for (int j = 0; j < 32; j += 8)
                st_global_v8(pdst + c * 32 + j, fv(c, j), fv(c, j + 1), fv(c, j + 2),
                             fv(c, j + 3), fv(c, j + 4), fv(c, j + 5), fv(c, j + 6),
                             fv(c, j + 7));
            }
          }
        } else if (store) {  // 16-byte aligned outputs
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            if (w.out_rec < 0) {
#pragma unroll
              for (int j = 0; j < 32; j += 8) {
                uint4 v;
                v.x = float2_to_bf16x2(__uint_as_float(r[c][j]) * inv,
                                       __uint_as_float(r[c][j + 1]) * inv);
                v.y = float2_to_bf16x2(__uint_as_float(r[c][j + 2]) * inv,
                                       __uint_as_float(r[c][j + 3]) * inv);
                v.z = float2_to_bf16x2(__uint_as_float(r[c][j + 4]) * inv,
                                       __uint_as_float(r[c][j + 5]) * inv);
                v.w = float2_to_bf16x2(__uint_as_float(r[c][j + 6]) * inv,
                                       __uint_as_float(r[c][j + 7]) * inv);
                *reinterpret_cast<uint4*>(odst + c * 32 + j) = v;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4*>(pdst + c * 32 + j) = make_float4(
                    __uint_as_float(r[c][j]) * inv, __uint_as_float(r[c][j + 1]) * inv,
                    __uint_as_float(r[c][j + 2]) * inv, __uint_as_float(r[c][j + 3]) * inv);
            }
          }
        }
      } else if (store) {
        // empty key range: zero output
        for (int j = 0; j < D; j += 8) {
          if (w.out_rec < 0)
            *reinterpret_cast<uint4*>(odst + j) = make_uint4(0, 0, 0, 0);
          else {
            *reinterpret_cast<float4*>(pdst + j) = make_float4(0.f, 0.f, 0.f, 0.f);
            *reinterpret_cast<float4*>(pdst + j + 4) = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
      uses += n;
      if (!store) continue;
      const float lse_v = any ? m + log2f(l) : -INFINITY;
      if (w.out_rec < 0) {
        if (a.lse) a.lse[(int64_t)(w.q_row0 + i_tok) * a.num_qo_heads + head] = lse_v;
      } else {
        a.part_lse[rec] = lse_v;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 9) {
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

// Encode the launch's tensor maps; returns whether the row maps for gather4
// were made (0 / 1), or -1 on failure.
template <int D>
int encode_maps(Maps& maps, const AttnArgs& a, int G, int nnz_q, int64_t total_kv) {
  int pp_gather = 0;
  const uint64_t Hq = a.num_qo_heads, Hk = a.num_kv_heads;
  std::memset(&maps, 0, sizeof(maps));
  {
    const uint64_t dims[3] = {(uint64_t)D, Hq, (uint64_t)(nnz_q > 0 ? nnz_q : 1)};
    const uint64_t str[2] = {(uint64_t)D * 2, Hq * D * 2};
    const uint32_t box[3] = {64, (uint32_t)G, (uint32_t)(BM / G)};
    if (!encode(&maps.q, a.q, 3, dims, str, box)) return -1;
  }
  if (a.kv_ragged) {
    const uint64_t dims[3] = {(uint64_t)D, Hk, (uint64_t)(total_kv > 0 ? total_kv : 1)};
    const uint64_t str[2] = {(uint64_t)D * 2, Hk * D * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)BN};
    if (!encode(&maps.kv_k, a.k, 3, dims, str, box) || !encode(&maps.kv_v, a.v, 3, dims, str, box))
      return -1;
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
      return -1;
    // The pool as rows of D elements (one kv head of one slot), for gather4:
    // row = page * (page_stride / D) + the slot's and head's row in the page.
    if (a.page_stride % D == 0) {
      const uint64_t rdims[2] = {(uint64_t)D, (uint64_t)1 << 31};
      const uint64_t rstr[1] = {(uint64_t)D * 2};
      const uint32_t rbox[2] = {64, 1};
      if (!encode(&maps.row_k, a.k, 2, rdims, rstr, rbox) ||
          !encode(&maps.row_v, a.v, 2, rdims, rstr, rbox))
        return -1;
      pp_gather = 1;
    }
  }
  return pp_gather;
}

template <int D>
cudaError_t launch_t(PrefillParams pp, int num_ctas, int nnz_q, int64_t total_kv,
                     MapCache* cache, cudaStream_t stream) {
  const AttnArgs& a = pp.a;
  static_assert(sizeof(Maps) <= sizeof(MapCache::maps), "map cache too small");
  Maps maps;
  // the maps describe Q and the K/V pools: encode them again only when one of
  // the buffers, its stride or its declared rows differ from the cached ones
  const uint64_t key[MapCache::kKeyWords] = {
      reinterpret_cast<uintptr_t>(a.q), reinterpret_cast<uintptr_t>(a.k),
      reinterpret_cast<uintptr_t>(a.v), (uint64_t)a.page_stride, (uint64_t)a.page_size,
      (uint64_t)a.layout, (uint64_t)a.kv_ragged, (uint64_t)a.num_qo_heads,
      (uint64_t)a.num_kv_heads, (uint64_t)pp.group, (uint64_t)nnz_q, (uint64_t)total_kv,
      (uint64_t)D, 0, 0, 0};
  int pp_gather;
  if (cache && cache->hit(key)) {
    std::memcpy(&maps, cache->maps, sizeof(maps));
    pp_gather = cache->aux;
  } else {
    pp_gather = encode_maps<D>(maps, a, pp.group, nnz_q, total_kv);
    if (pp_gather < 0) return cudaErrorInvalidValue;
    if (cache) cache->store(key, &maps, sizeof(maps), pp_gather);
  }
  constexpr int NB = D / 64;
  // At least 120 KiB, so that one CTA (and its 512 TMEM columns) owns each SM.
  size_t smem = 1024 + (size_t)(2 + Ring<D>::K + Ring<D>::V) * NB * BLK;
  if (smem < 120 * 1024) smem = 120 * 1024;
  cudaError_t e = ensure_dynamic_smem<prefill_kernel<D>>((int)smem);
  if (e != cudaSuccess) return e;
  pp.gather = pp_gather;
  pp.rows_per_page = pp_gather ? a.page_stride / D : 0;
  prefill_kernel<D><<<num_ctas, kThreads, smem, stream>>>(maps, pp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const AttnArgs& a0, int num_ctas, int head_dim, int group,
                           int nnz_q, int64_t total_kv, MapCache* cache, cudaStream_t stream) {
  PrefillParams pp;
  pp.a = a0;
  pp.a.err = device_error_word();
  pp.group = group;
  if (head_dim == 128) return launch_t<128>(pp, num_ctas, nnz_q, total_kv, cache, stream);
  return launch_t<64>(pp, num_ctas, nnz_q, total_kv, cache, stream);
}

}  // namespace pka
