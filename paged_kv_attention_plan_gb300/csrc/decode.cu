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
// state.  The pieces of a split request count themselves in a join counter
// of the plan image, and the last one merges the pieces' states ("A worked
// split-KV example") and writes O and the LSE, so no separate merge launch
// follows the decode kernel.  Every piece writes its partial state.  A
// consumer warp that finds (from a read of the counter during its last tile)
// that every other piece has finished then merges all the pieces' states.
// Otherwise, for a CTA's last item it counts the piece in itself and merges
// if that completes the count (each warp its own kv head, in parallel);
// earlier split pieces go to the CTA's join warp, which makes their states
// visible GPU-wide and counts them in while the consumers go on with the next
// item.
//
// e4m3 K/V (8-bit codes with one scale per pool) stages half the bytes per
// key.  K fragments come straight from shared memory: one 32-bit load holds
// four consecutive dims of a key, converted to f16 pairs; the dims of each
// 16-wide k-block are taken in the order 0-3 | 4-7 | ... instead of the MMA's
// 0,1,8,9 | 2,3,10,11 | ..., and Q's fragments follow the same order, so the
// dot products are unchanged.  Each warp converts its kv head's V rows to f16
// in a scratch tile read with ldmatrix.trans.  These MMAs run in f16 (e4m3
// values are exact in f16; Q rounds to f16 once, P is in [0, 1]).  K's scale
// is folded into the softmax scale and V's scale into the output.
//
// Pages of 8 or a multiple of 16 slots (not ragged K/V, and e4m3 only with
// D = 128) take a boxed staging layout instead: per 16-key tile, one TMA box
// per 128-byte column block (64 bf16 dims or 128 e4m3 dims) and per K/V
// brings the keys of all the CTA's kv heads, with the 128-byte swizzle
// (16-byte chunk c of row r stored at chunk c ^ (r & 7)); the fragment
// addresses follow the swizzle.  A few large copies per tile replace one
// copy per key row.  An HND box is [heads][slots]: a head's consecutive keys
// are consecutive rows.  An NHD box is [slots][heads]; its head count is
// rounded up to an odd number (the extra head lies past the pool's last head
// and is zero-filled, or belongs to the next head block), so that a head's
// 8 consecutive keys fall in 8 different swizzle phases.
//
// In either layout the rows of a tile past its last key hold whatever the
// stage held before (or, boxed, the rest of the request's last page): their
// scores are replaced by -inf and their V values by zeros in registers
// before the P V product, so shared memory is never cleared.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "pka_internal.h"
#include "tc_device.cuh"

namespace pka {
namespace {

constexpr int TS = kDecodeTileTokens;  // keys per stage = one m16 MMA block
constexpr int kMaxStages = 4;
constexpr int kMaxStagesF8 = 6;
constexpr int kJoinRing = 4;  // split pieces in flight between the consumers and the join warp
// Dynamic shared memory for stages (and the e4m3 V scratch): 227 KiB less
// the 1 KiB alignment pad, the barriers and the static variables.
constexpr int kStageBudget = 227 * 1024 - 2048;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

struct Bars {
  uint64_t* base;
  int stages;
  __device__ uint32_t full(int s) const { return smem_u32(base + s); }
  __device__ uint32_t empty(int s) const { return smem_u32(base + stages + s); }
};

// Bytes of one key row in a stage: the CTA's kv heads, plus 16 bytes of pad
// (ES bytes per element: 2 for bf16, 1 for e4m3).
__host__ __device__ constexpr int row_bytes(int hpc, int D, int ES = 2) {
  return hpc * D * ES + 16;
}
// e4m3 path: a warp's f16 V scratch, [16 keys][D + 8] halves (padded rows).
__host__ __device__ constexpr int vs_row_bytes(int D) { return (D + 8) * 2; }

struct DecodeMaps {
  // boxed staging: NHD pool {D, Hk, P, pages}, box {cols, odd heads, R, 1};
  // HND pool {D, P, Hk, pages}, box {cols, R, heads, 1}; R = min(P, 16)
  CUtensorMap k;
  CUtensorMap v;
};

// Tiles start at multiples of 16 keys inside a request (the planner cuts
// there), so with P = 8 or P a multiple of 16 every box of min(P, 16) slots
// stays inside one page.
__host__ __device__ inline bool use_boxes(int P, int ragged, int D, int ES) {
  return !ragged && (P == 8 || P % 16 == 0) && D * ES >= 128;
}

// Heads per box: the CTA's heads; an NHD box rounds them up to an odd count.
__host__ __device__ inline int box_heads(int layout, int hpc) {
  return layout == PKA_NHD ? (hpc | 1) : hpc;
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

// The same product with f16 operands (e4m3 K/V).
__device__ __forceinline__ void mma16816_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two e4m3 codes (low byte first) -> two f16 (low half first); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes) {
  uint32_t r;
  asm("{\n .reg .b16 c;\n cvt.u16.u32 c, %1;\n cvt.rn.f16x2.e4m3x2 %0, c;\n}"
      : "=r"(r)
      : "r"(codes));
  return r;
}

// Round two floats to f16 and pack them (low = a).
__device__ __forceinline__ uint32_t float2_to_f16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint32_t transpose8x8(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// n-way merge of the pieces of one split (request, kv head) for its G qo
// heads, all read from the float workspace ("Deep Dive - FlashInfer", "Core
// mechanism" and "A worked split-KV example"): with b_k the pieces' base-2
// statistics, m = max b_k and s = sum 2^(b_k - m), o = sum (2^(b_k - m) / s)
// o_k and lse = m + log2 s; pieces with b_k = -inf carry no weight, and if
// all are empty o = 0 and lse = -inf.  Every lane owns D / 32 dims of every
// head and folds the (piece, head) pairs in one at a time (a running max with
// rescaling), so all lanes hold the same statistics and nothing is exchanged.
// The states come from other SMs and are read through L2 (.cg), 16 pairs
// per round, all loads of a round issued before any is used.
template <int D, int G>
__device__ __noinline__ void join_merge_g(const AttnArgs& a, const PkaDecodeJoin j, int row,
                                          int head0, int lane) {
  constexpr int PER = D / 32;
  constexpr int CH = G == 8 ? 8 : 12;  // pairs per round; a multiple of G (pair q is head q % G)
  const int pairs = j.nslots * G;
  float m[G], s[G], acc[G][PER];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    s[h] = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[h][e] = 0.f;
  }
  for (int p0 = 0; p0 < pairs; p0 += CH) {
    float b[CH], x[CH][PER];
#pragma unroll
    for (int q = 0; q < CH; ++q) {
      const int p = p0 + q;
      const bool ok = p < pairs;
      const int64_t rec = j.rec_first + (int64_t)(p / G) * j.rec_stride + q % G;
      b[q] = ok ? __ldcg(a.part_lse + rec) : -INFINITY;
      const float* src = a.part_o + (ok ? rec : 0) * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = ok ? __ldcg(reinterpret_cast<const float4*>(src))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        x[q][0] = v.x;
        x[q][1] = v.y;
        x[q][2] = v.z;
        x[q][3] = v.w;
      } else {
        const float2 v = ok ? __ldcg(reinterpret_cast<const float2*>(src)) : make_float2(0.f, 0.f);
        x[q][0] = v.x;
        x[q][1] = v.y;
      }
    }
#pragma unroll
    for (int q = 0; q < CH; ++q) {
      const int h = q % G;
      if (b[q] == -INFINITY) continue;
      if (b[q] > m[h]) {
        const float sc = exp2f(m[h] - b[q]);  // 0 while m is -inf
        s[h] = s[h] * sc + 1.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[h][e] = acc[h][e] * sc + x[q][e];
        m[h] = b[q];
      } else {
        const float wq = exp2f(b[q] - m[h]);
        s[h] += wq;
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[h][e] += wq * x[q][e];
      }
    }
  }
  const int Hq = a.num_qo_heads;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const bool any = s[h] > 0.f;
    const float inv = any ? 1.f / s[h] : 0.f;
    const int64_t oi = (int64_t)row * Hq + head0 + h;
    uint16_t* dst = a.o + oi * D + lane * PER;
    if constexpr (PER == 4) {
      uint2 pk;
      pk.x = float2_to_bf16x2(acc[h][0] * inv, acc[h][1] * inv);
      pk.y = float2_to_bf16x2(acc[h][2] * inv, acc[h][3] * inv);
      *reinterpret_cast<uint2*>(dst) = pk;
    } else {
      *reinterpret_cast<uint32_t*>(dst) = float2_to_bf16x2(acc[h][0] * inv, acc[h][1] * inv);
    }
    if (lane == 0 && a.lse) a.lse[oi] = any ? m[h] + log2f(s[h]) : -INFINITY;
  }
}

template <int D>
__device__ __forceinline__ void join_merge(const AttnArgs& a, const PkaDecodeJoin& j, int row,
                                           int head0, int G, int lane) {
  switch (G) {
    case 1: join_merge_g<D, 1>(a, j, row, head0, lane); break;
    case 2: join_merge_g<D, 2>(a, j, row, head0, lane); break;
    case 4: join_merge_g<D, 4>(a, j, row, head0, lane); break;
    default: join_merge_g<D, 8>(a, j, row, head0, lane); break;
  }
}

// Issue the bulk copies of keys [a0, a0 + n) of item w (K and V) into a stage
// (ES bytes per element).
// `page` is the page id of key a0 + (lane & 15), loaded ahead by the caller
// (unused for ragged K/V and for head-major pages).
template <int D, int ES>
__device__ __forceinline__ void issue_tile_copies(const AttnArgs& a, const PkaWorkItem& w,
                                                  int a0, int n, int hpc, uint32_t dK,
                                                  uint32_t dV, uint32_t bar, int lane, int page) {
  const int Hk = a.num_kv_heads;
  const int P = a.page_size;
  const int RS = row_bytes(hpc, D, ES);
  const uint8_t* kp = reinterpret_cast<const uint8_t*>(a.k);
  const uint8_t* vp = reinterpret_cast<const uint8_t*>(a.v);
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
      off = (int64_t)page * a.page_stride + (int64_t)(j % P) * row;
    }
    off += (int64_t)w.kv_head0 * D;
    if (lane < 16)
      bulk_g2s(dK + t * RS, kp + off * ES, (uint32_t)(hpc * D * ES), bar);
    else
      bulk_g2s(dV + t * RS, vp + off * ES, (uint32_t)(hpc * D * ES), bar);
    return;
  }
  // HND page [Hk, P, D]: one copy per (key, kv head, K or V)
  for (int x = lane; x < n * hpc * 2; x += 32) {
    const int kv = x & 1, h = (x >> 1) % hpc, t = (x >> 1) / hpc;
    const int j = a0 + t;
    const int page = a.kv_indices[w.kv_base + j / P];
    const int64_t off =
        (int64_t)page * a.page_stride + ((int64_t)(w.kv_head0 + h) * P + (j % P)) * D;
    const uint32_t d = (kv ? dV : dK) + t * RS + h * D * ES;
    bulk_g2s(d, (kv ? vp : kp) + off * ES, (uint32_t)(D * ES), bar);
  }
}

// Boxed staging of keys [a0, a0 + n) (a0 is a multiple of 16): boxes of
// R = min(P, 16) slots that hold at least one key of the tile, for every
// 128-byte column block, K and V.  Issued by one lane; returns the bytes.
template <int D, int ES>
__device__ __forceinline__ uint32_t issue_tile_boxes(const AttnArgs& a, const DecodeMaps& maps,
                                                     const PkaWorkItem& w, int a0, int n, int hb,
                                                     uint32_t dK, uint32_t dV, uint32_t bar) {
  constexpr int CW = 128 / ES;          // columns of one block
  constexpr int NBc = D / CW;           // blocks per row
  const int P = a.page_size;
  const int R = P < TS ? P : TS;
  const uint32_t blk = (uint32_t)(TS * hb * 128);   // one block of a stage
  const uint32_t box = (uint32_t)(R * hb * 128);    // one box
  const int nbox = (n + R - 1) / R;
  const bool nhd = a.layout == PKA_NHD;
  for (int b = 0; b < nbox; ++b) {
    const int j = a0 + b * R;
    const int page = a.kv_indices[w.kv_base + j / P];
    const int slot = j % P;
#pragma unroll
    for (int c = 0; c < NBc; ++c) {
      const uint32_t off = c * blk + b * box;
      if (nhd) {
        tc::tma_load_4d(dK + off, &maps.k, c * CW, w.kv_head0, slot, page, bar);
        tc::tma_load_4d(dV + off, &maps.v, c * CW, w.kv_head0, slot, page, bar);
      } else {
        tc::tma_load_4d(dK + off, &maps.k, c * CW, slot, w.kv_head0, page, bar);
        tc::tma_load_4d(dV + off, &maps.v, c * CW, slot, w.kv_head0, page, bar);
      }
    }
  }
  return (uint32_t)nbox * NBc * 2 * box;
}

// Warps: consumers 0 .. hpc - 1 (one per kv head), producer hpc, join warp hpc + 1.
// F8: the K/V pools hold e4m3 codes.
template <int D, bool F8>
__global__ void __launch_bounds__(320, 1)
    decode_kernel(const __grid_constant__ DecodeMaps maps, const AttnArgs a, const int stages,
                  const int hb) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ volatile int abort_flag;
  // Handoff of split pieces to the join warp: per slot, one arrival per
  // consumer warp (jfull) and a release by the join warp (jempty); jneed[s][hl]
  // says whether kv head hl's partial state still has to be counted in.
  __shared__ uint64_t jfull[kJoinRing], jempty[kJoinRing];
  __shared__ int jneed[kJoinRing][8];
  constexpr int KS = D / 16;  // k-steps of the QK^T product
  constexpr int MT = D / 16;  // 16-dim blocks of the P V product
  const int hpc = a.heads_per_cta;
  const int G = a.num_qo_heads / a.num_kv_heads;
  const int n_cons = hpc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int ES = F8 ? 1 : 2;  // bytes per K/V element
  // hb > 0: boxed staging (hb heads per box row group, D * ES / 128 blocks of
  // [16 keys x hb heads] 128-byte rows); hb == 0: one padded row per key
  const bool boxed = hb > 0;
  const int RS = row_bytes(hpc, D, ES);
  const int stage_bytes = boxed ? (D * ES / 128) * TS * hb * 128 : TS * RS;
  uint8_t* sK = smem;
  uint8_t* sV = smem + stages * stage_bytes;
  uint8_t* sVc = smem + 2 * stages * stage_bytes;  // e4m3: per-warp f16 V scratch
  const int scratch_bytes = F8 ? hpc * TS * vs_row_bytes(D) : 0;
  const Bars bars{reinterpret_cast<uint64_t*>(smem + 2 * stages * stage_bytes + scratch_bytes),
                  stages};

  const int i0 = a.cta_ptr[blockIdx.x], i1 = a.cta_ptr[blockIdx.x + 1];
  if (i0 >= i1) return;  // an empty CTA of a fixed (graph mode) grid
  // Rows of a tile past its last key are never zeroed in shared memory: their
  // scores are replaced by -inf and their V values by zeros in registers.
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(bars.full(s), 33);  // expect_tx by lane 0 + the 32 producer lanes
      mbar_init(bars.empty(s), n_cons);
    }
    for (int s = 0; s < kJoinRing; ++s) {
      mbar_init(smem_u32(&jfull[s]), n_cons);
      mbar_init(smem_u32(&jempty[s]), 1);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == n_cons) {
    // ---------------- producer warp ----------------
    // Row copies of paged K/V: the page ids of a tile are loaded one tile
    // ahead (lanes t and t + 16 hold the page of key t), so their latency
    // overlaps the wait for a free stage instead of delaying the copies.  With
    // one-token pages every key has its own id.  (Boxed staging needs one or
    // two ids a tile and loads them as it issues: loading them ahead measured
    // slower there.)
    const int P = a.page_size;
    const bool ahead = !boxed && !a.kv_ragged && !(a.layout == PKA_HND && P > 1);
    auto tile_page = [&](const PkaWorkItem& w, int a0) -> int {
      const int j = a0 + (lane & 15);
      return j < w.t1 ? a.kv_indices[w.kv_base + j / P] : 0;
    };
    uint32_t it = 0;
    for (int ii = i0; ii < i1 && !warp_any(&abort_flag); ++ii) {
      const PkaWorkItem w = a.items[ii];
      int page = ahead ? tile_page(w, w.t0) : 0;
      for (int a0 = w.t0; a0 < w.t1; a0 += TS, ++it) {
        const int s = it % stages;
        const int next_page = ahead && a0 + TS < w.t1 ? tile_page(w, a0 + TS) : 0;
        if (!mbar_wait_warp(bars.empty(s), ((it / stages) & 1) ^ 1)) {
          record_timeout(a.err, &abort_flag);
          break;
        }
        const int n = min(TS, w.t1 - a0);
        if (boxed) {
          if (lane == 0) {
            const int R = a.page_size < TS ? a.page_size : TS;
            mbar_arrive_expect_tx(bars.full(s), (uint32_t)(((n + R - 1) / R) * (D * ES / 128) *
                                                           2 * R * hb * 128));
            issue_tile_boxes<D, ES>(a, maps, w, a0, n, hb, smem_u32(sK + s * stage_bytes),
                                    smem_u32(sV + s * stage_bytes), bars.full(s));
          }
          __syncwarp();
        } else {
          if (lane == 0) mbar_arrive_expect_tx(bars.full(s), (uint32_t)(2 * n * hpc * D * ES));
          __syncwarp();
          issue_tile_copies<D, ES>(a, w, a0, n, hpc, smem_u32(sK + s * stage_bytes),
                                   smem_u32(sV + s * stage_bytes), bars.full(s), lane, page);
        }
        mbar_arrive(bars.full(s));
        page = next_page;
      }
    }
    // Drain: every issued tile's copies must land before the CTA leaves.
    const uint32_t first = it > (uint32_t)stages ? it - stages : 0;
    for (uint32_t k = first; k < it; ++k)
      if (!mbar_wait_warp(bars.full(k % stages), (k / stages) & 1)) record_timeout(a.err, &abort_flag);
    return;
  }
  if (warp == n_cons + 1) {
    // ---------------- join warp ----------------
    // Takes the split pieces before the CTA's last item, in the consumers'
    // order.  For every kv head whose consumer wrote a partial state: fence
    // (the consumers' stores reach it through the CTA-scope barrier, the fence
    // makes them visible GPU-wide), count the piece in, and if that completes
    // the count merge all pieces (rare: such a piece is normally the first
    // item of its CTA, and its unit's other pieces end later).
    uint32_t jc = 0;
    for (int ii = i0; ii < i1 - 1 && !warp_any(&abort_flag); ++ii) {
      const PkaWorkItem w = a.items[ii];
      if (w.join < 0 || !a.joins) continue;
      const int s = jc % kJoinRing;
      if (!mbar_wait_warp(smem_u32(&jfull[s]), (jc / kJoinRing) & 1)) {
        record_timeout(a.err, &abort_flag);
        break;
      }
      const int need = lane < n_cons ? jneed[s][lane] : 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&jempty[s]));
      ++jc;
      if (!__ballot_sync(0xffffffffu, need)) continue;
      __threadfence();
      int last = 0;
      if (need) {
        PkaDecodeJoin* jp = a.joins + w.join + lane;
        last = atomicAdd(&jp->arrived, 1) == jp->nslots - 1;
      }
      uint32_t lm = __ballot_sync(0xffffffffu, last);
      if (lm) __threadfence();
      while (lm) {
        const int hq = __ffs(lm) - 1;
        lm &= lm - 1;
        PkaDecodeJoin* jq = a.joins + w.join + hq;
        join_merge<D>(a, *jq, w.q_row0, (w.kv_head0 + hq) * G, G, lane);
        __syncwarp();
        if (lane == 0) jq->arrived = 0;  // every piece has arrived: re-arm for the next run
      }
    }
    return;
  }
  if (warp > n_cons + 1) return;

  // ---------------- consumer warps: warp hl serves kv head kv_head0 + hl ----------------
  const int hl = warp;
  const int qd = lane & 3;    // thread in quad: heads 2qd, 2qd + 1 of S^T
  const int grp = lane >> 2;  // group: key row of S^T; head of the Q^T / P^T fragments
  const int Hq = a.num_qo_heads;
  // ldmatrix row addresses (bytes inside a stage) of this lane
  const int mi = lane >> 3, mr = lane & 7;
  const uint32_t k_lane = (uint32_t)((mr + 8 * (mi & 1)) * RS + hl * D * 2 + 16 * (mi >> 1));
  const uint32_t v_lane = (uint32_t)((mr + 8 * (mi >> 1)) * RS + hl * D * 2 + 16 * (mi & 1));
  // boxed staging: row of key t of kv head hl in a block, and the address of
  // 16-byte chunk c of a row (blocks of 8 chunks, 128-byte swizzle)
  const int R = a.page_size < TS ? a.page_size : TS;
  const bool nhd = a.layout == PKA_NHD;
  const uint32_t blk = (uint32_t)(TS * hb * 128);
  auto box_row = [&](int t) -> int {
    return nhd ? (t / R) * R * hb + (t % R) * hb + hl : (t / R) * R * hb + hl * R + (t % R);
  };
  auto box_addr = [&](int row, int c) -> uint32_t {
    return (uint32_t)((c >> 3) * blk + row * 128 + (((c & 7) ^ (row & 7)) << 4));
  };
  const int k_key = mr + 8 * (mi & 1), v_key = mr + 8 * (mi >> 1);
  const int k_row = boxed ? box_row(k_key) : 0, v_row = boxed ? box_row(v_key) : 0;
  const uint32_t sK0 = smem_u32(sK), sV0 = smem_u32(sV);
  const float sc = a.scale_log2;
  uint32_t it = 0, jc = 0;
  for (int ii = i0; ii < i1 && !warp_any(&abort_flag); ++ii) {
    const PkaWorkItem w = a.items[ii];
    const int head_base = (w.kv_head0 + hl) * G;  // first qo head of this kv head
    // split piece: the join's fixed fields now, the counter during the last tile
    PkaDecodeJoin* jp = (w.join >= 0 && a.joins) ? a.joins + w.join + hl : nullptr;
    PkaDecodeJoin jv{};
    if (jp) jv = *jp;
    int hint = -1;
    // Q^T fragments (k = dims, n = heads): head grp, dims 16ks + 2qd (+1, +8, +9);
    // e4m3 K/V: dims 16ks + 4qd (+1 | +2, +3) in f16 (the k order of the K
    // fragments read from e4m3 rows)
    uint32_t qf[KS][2];
    {
      const bool real = grp < G;
      const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
          a.q + ((int64_t)w.q_row0 * Hq + head_base + (real ? grp : 0)) * D);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        if constexpr (F8) {
          const uint2 q4 = real ? *reinterpret_cast<const uint2*>(qrow + 8 * ks + 2 * qd)
                                : make_uint2(0u, 0u);
          const float2 f0 = bf16x2_to_float2(q4.x), f1 = bf16x2_to_float2(q4.y);
          qf[ks][0] = float2_to_f16x2(f0.x, f0.y);
          qf[ks][1] = float2_to_f16x2(f1.x, f1.y);
        } else {
          qf[ks][0] = real ? qrow[8 * ks + qd] : 0u;
          qf[ks][1] = real ? qrow[8 * ks + 4 + qd] : 0u;
        }
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
      if (jp && a0 + TS >= w.t1 && lane == 0)
        hint = *reinterpret_cast<volatile int32_t*>(&jp->arrived);
      if (!mbar_wait_warp(bars.full(s), (it / stages) & 1)) {
        record_timeout(a.err, &abort_flag);
        break;
      }
      const int n = min(TS, w.t1 - a0);
      const uint32_t kb = sK0 + s * stage_bytes, vb = sV0 + s * stage_bytes;
      // S^T = K . Q^T
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (F8) {
        // keys grp and grp + 8, dims 16ks + 4qd .. + 3 of each: one word each
        // (chunk ks of the key's 128-byte row)
        const int r0 = boxed ? box_row(grp) : 0, r1 = boxed ? box_row(grp + 8) : 0;
        const uint32_t k0 = kb + (uint32_t)(grp * RS + hl * D + 4 * qd);
        const uint32_t k1 = k0 + 8 * RS;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t w0 =
              ld_shared_u32(boxed ? kb + box_addr(r0, ks) + 4 * qd : k0 + 16 * ks);
          const uint32_t w1 =
              ld_shared_u32(boxed ? kb + box_addr(r1, ks) + 4 * qd : k1 + 16 * ks);
          uint32_t af[4];
          af[0] = e4m3x2_to_f16x2(w0 & 0xffffu);
          af[1] = e4m3x2_to_f16x2(w1 & 0xffffu);
          af[2] = e4m3x2_to_f16x2(w0 >> 16);
          af[3] = e4m3x2_to_f16x2(w1 >> 16);
          mma16816_f16(sacc, af, qf[ks][0], qf[ks][1]);
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t af[4];
          ldsm_x4(kb + (boxed ? box_addr(k_row, 2 * ks + (mi >> 1)) : k_lane + 32 * ks), af);
          mma16816(sacc, af, qf[ks][0], qf[ks][1]);
        }
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
      if constexpr (F8) {
        const uint32_t pb0 = transpose8x8(float2_to_f16x2(p00, p01));
        const uint32_t pb1 = transpose8x8(float2_to_f16x2(p10, p11));
        // V rows of this kv head, e4m3 -> f16, into the warp's scratch (two
        // lanes per key, D / 2 codes each), then O^T += V^T . P^T from it
        const uint32_t vs = smem_u32(sVc) + (uint32_t)(hl * TS * vs_row_bytes(D));
        {
          // keys past the tile (n < 16) may hold anything: they become zeros.
          // Lane = key + 16 * half: each group of 8 lanes stores 8 different
          // keys' rows, whose starts fall in 8 different bank groups.
          constexpr int PL = D / 2;  // codes per lane
          const int key = lane & 15, half = lane >> 4;
          const int vrow = boxed ? box_row(key) : 0;
          const uint32_t src = vb + (uint32_t)(key * RS + hl * D + half * PL);
          const uint32_t dst = vs + (uint32_t)(key * vs_row_bytes(D) + half * PL * 2);
#pragma unroll
          for (int x = 0; x < PL / 16; ++x) {
            uint4 c = ld_shared_v4(boxed ? vb + box_addr(vrow, half * (PL / 16) + x)
                                         : src + 16 * x);
            if (key >= n) c = make_uint4(0u, 0u, 0u, 0u);
            st_shared_v4(dst + 32 * x,
                         make_uint4(e4m3x2_to_f16x2(c.x & 0xffffu), e4m3x2_to_f16x2(c.x >> 16),
                                    e4m3x2_to_f16x2(c.y & 0xffffu), e4m3x2_to_f16x2(c.y >> 16)));
            st_shared_v4(dst + 32 * x + 16,
                         make_uint4(e4m3x2_to_f16x2(c.z & 0xffffu), e4m3x2_to_f16x2(c.z >> 16),
                                    e4m3x2_to_f16x2(c.w & 0xffffu), e4m3x2_to_f16x2(c.w >> 16)));
          }
        }
        __syncwarp();
        const uint32_t vl = vs + (uint32_t)((mr + 8 * (mi >> 1)) * vs_row_bytes(D) + 16 * (mi & 1));
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t af[4];
          ldsm_x4_t(vl + 32 * mt, af);
          mma16816_f16(acc[mt], af, pb0, pb1);
        }
      } else {
        const uint32_t pb0 = transpose8x8(float2_to_bf16x2(p00, p01));
        const uint32_t pb1 = transpose8x8(float2_to_bf16x2(p10, p11));
        // O^T += V^T . P^T.  Keys past the tile (n < 16) may hold anything in
        // the boxed layout: their V values become zeros (lane holds keys 2qd,
        // 2qd + 1 in af[0], af[1] and keys 8 + 2qd, 9 + 2qd in af[2], af[3]).
        const uint32_t vm0 = (2 * qd < n ? 0xffffu : 0u) | (2 * qd + 1 < n ? 0xffff0000u : 0u);
        const uint32_t vm1 =
            (2 * qd + 8 < n ? 0xffffu : 0u) | (2 * qd + 9 < n ? 0xffff0000u : 0u);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t af[4];
          ldsm_x4_t(vb + (boxed ? box_addr(v_row, 2 * mt + (mi & 1)) : v_lane + 32 * mt), af);
          af[0] &= vm0;
          af[1] &= vm0;
          af[2] &= vm1;
          af[3] &= vm1;
          mma16816(acc[mt], af, pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.empty(s));
    }
    if (warp_any(&abort_flag)) break;

    // Sum the exp shares over the 8 key groups; normalise and write.
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    // Write O and the LSE, or this piece's partial state.  A split piece
    // whose counter read (issued during the last tile) shows every other
    // piece finished then merges all of them at once.
    const bool merge_now = jp && __shfl_sync(0xffffffffu, hint, 0) == jv.nslots - 1;
    {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 2 * qd + hh;  // head of this lane's accumulator columns
        if (h >= G) continue;
        const float l = hh ? l1 : l0, m = hh ? m1 : m0;
        const bool any = l > 0.f;
        const float inv = any ? a.v_scale / l : 0.f;  // V's scale (1 for bf16 K/V)
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
    bool do_merge = merge_now;
    if (jp && !merge_now && ii + 1 == i1) {
      // the CTA's last item: count the piece in here; the fence makes this
      // lane's partial state visible GPU-wide before the arrival
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = atomicAdd(&jp->arrived, 1) == jv.nslots - 1;
      do_merge = __shfl_sync(0xffffffffu, last, 0) != 0;
    }
    if (do_merge) {
      // this warp's own state was just written (the warp barrier orders it
      // for the other lanes); the fence, after the counter read or the
      // arrival, orders the other pieces' states before the reads
      __syncwarp();
      __threadfence();
      join_merge<D>(a, jv, w.q_row0, head_base, G, lane);
      __syncwarp();
      if (lane == 0) jp->arrived = 0;  // every piece is done: re-arm for the next run
    }
    if (jp && ii + 1 < i1) {
      // hand the piece to the join warp (kv head hl still to count in or not)
      __syncwarp();
      if (lane == 0) {
        const int js = jc % kJoinRing;
        if (jc >= (uint32_t)kJoinRing &&
            !mbar_wait(smem_u32(&jempty[js]), ((jc / kJoinRing) - 1) & 1)) {
          record_timeout(a.err, &abort_flag);
        } else {
          jneed[js][hl] = merge_now ? 0 : 1;
          mbar_arrive(smem_u32(&jfull[js]));
        }
      }
      ++jc;
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

// Boxed staging maps: NHD pool {D, Hk, P, pages} with box {128 B of columns,
// hb heads, R slots, 1}; HND pool {D, P, Hk, pages} with box {128 B, R slots,
// hb heads, 1}; R = min(P, 16); 128-byte swizzle.  Page ids come from
// kv_indices, so the page dimension is declared as large as TMA allows.
bool encode_box(CUtensorMap* m, const void* base, const AttnArgs& a, int D, int ES, int hb) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t P = a.page_size, Hk = a.num_kv_heads, E = ES;
  const cuuint32_t R = (cuuint32_t)(P < (cuuint64_t)TS ? P : TS), CW = 128 / ES;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4];
  if (a.layout == PKA_NHD) {
    dims[0] = D; dims[1] = Hk; dims[2] = P; dims[3] = (cuuint64_t)1 << 31;
    strides[0] = D * E; strides[1] = Hk * D * E; strides[2] = (cuuint64_t)a.page_stride * E;
    box[0] = CW; box[1] = (cuuint32_t)hb; box[2] = R; box[3] = 1;
  } else {
    dims[0] = D; dims[1] = P; dims[2] = Hk; dims[3] = (cuuint64_t)1 << 31;
    strides[0] = D * E; strides[1] = P * D * E; strides[2] = (cuuint64_t)a.page_stride * E;
    box[0] = CW; box[1] = R; box[2] = (cuuint32_t)hb; box[3] = 1;
  }
  cuuint32_t es[4] = {1, 1, 1, 1};
  return fn(m, ES == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
            const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool F8>
cudaError_t launch_t(const AttnArgs& a, int num_ctas, MapCache* cache, cudaStream_t stream) {
  constexpr int ES = F8 ? 1 : 2;
  const int hpc = a.heads_per_cta;
  static_assert(sizeof(DecodeMaps) <= sizeof(MapCache::maps), "map cache too small");
  DecodeMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  int hb = use_boxes(a.page_size, a.kv_ragged, D, ES) ? box_heads(a.layout, hpc) : 0;
  if (hb) {
    // the boxed maps describe the pools: encode them again only when the
    // pools, their layout or the head block differ from the cached ones
    const uint64_t key[MapCache::kKeyWords] = {
        reinterpret_cast<uintptr_t>(a.k), reinterpret_cast<uintptr_t>(a.v),
        (uint64_t)a.page_stride, (uint64_t)a.page_size, (uint64_t)a.layout,
        (uint64_t)a.num_kv_heads, (uint64_t)D, (uint64_t)ES, (uint64_t)hb, 0, 0, 0, 0, 0, 0, 0};
    if (cache && cache->hit(key)) {
      std::memcpy(&maps, cache->maps, sizeof(maps));
      hb = cache->aux;
    } else {
      if (!encode_box(&maps.k, a.k, a, D, ES, hb) || !encode_box(&maps.v, a.v, a, D, ES, hb))
        hb = 0;  // fall back to one bulk copy per key row
      if (cache) cache->store(key, &maps, sizeof(maps), hb);
    }
  }
  const int stage_bytes = 2 * (hb ? (D * ES / 128) * TS * hb * 128 : TS * row_bytes(hpc, D, ES));
  const int scratch = F8 ? hpc * TS * vs_row_bytes(D) : 0;
  int stages = (kStageBudget - scratch) / stage_bytes;
  if (stages > (F8 ? kMaxStagesF8 : kMaxStages)) stages = F8 ? kMaxStagesF8 : kMaxStages;
  if (stages < 2) return cudaErrorInvalidConfiguration;
  // the swizzled blocks need 1024-byte alignment: pad the dynamic allocation
  const size_t smem =
      1024 + (size_t)stages * stage_bytes + scratch + 2 * stages * sizeof(uint64_t);
  cudaError_t e = ensure_dynamic_smem<decode_kernel<D, F8>>((int)smem);
  if (e != cudaSuccess) return e;
  decode_kernel<D, F8><<<num_ctas, 32 * (hpc + 2), smem, stream>>>(maps, a, stages, hb);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const AttnArgs& a0, int num_ctas, int head_dim, int group,
                          MapCache* cache, cudaStream_t stream) {
  AttnArgs a = a0;
  a.err = device_error_word();
  (void)group;
  if (a.kv_fp8)
    return head_dim == 128 ? launch_t<128, true>(a, num_ctas, cache, stream)
                           : launch_t<64, true>(a, num_ctas, cache, stream);
  return head_dim == 128 ? launch_t<128, false>(a, num_ctas, cache, stream)
                         : launch_t<64, false>(a, num_ctas, cache, stream);
}

}  // namespace pka
