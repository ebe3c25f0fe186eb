// Stage 1 for GQA: one block per work item (request b, KV head, split s).
// The block streams the split's K and V rows through shared memory and
// leaves, for each of the group's query heads, the normalised P.V partial and
// its log2-sum-exp2 (scores are pre-multiplied by log2 e).
//
// Warp layout. W = gqa_warps(D) warps; warp w takes the 16-token blocks w,
// w + W, w + 2W, ... of the item and owns gqa_stages_per_warp(D) stages. Each
// warp issues the copies of its own next blocks as soon as it has finished
// with a stage, so its copies are in flight while it computes: the aiter pull
// 4758 page's two-blocks-in-flight idea (Technical Details 1: retire only the
// page-number load early, wait for a KV copy only where its data is read)
// carried to several warps, because one warp's copies are issued one after
// another. Page ids are read ahead of use in a per-warp register window. A
// stage is only ever filled and read by its own warp, in order, so a wait on
// a phase parity cannot be confused with an older phase. Every warp runs its
// own online softmax; a fixed-order merge of the warps ends the item.
//
// K/V movement (template TILES):
//   * TILES: each 16-token block is one page-aligned run of 16 rows, moved as
//     two TMA tensor copies (K tile, V tile) through a 3D tensor map
//     {64 columns, pool rows, D/64 column blocks} with a {64, 16, D/64} box
//     and 128-byte swizzle: element (row r, column d) of a tile sits at
//     (d/64)*2048 + r*128 + (((d%64)/8) ^ (r%8))*16 + (d%8)*2, so 8
//     consecutive rows of one 16-byte column chunk hit 8 distinct bank groups.
//   * !TILES (any page size, any split boundary): one bulk copy per K or V
//     row into rows padded to D*2 + 16 bytes, the bank-conflict-free pitch of
//     the rocm-libraries pull 10102 page (Motivation: pad the row pitch so a
//     wave's reads spread over all banks), redone for 32 banks x 4 bytes.
//
// This header holds what both consumers share (stage1_gqa_fma.cu,
// stage1_gqa_mma.cu): shared-memory layout, the per-warp copy pipeline and
// the cross-warp merge.
#pragma once

#include "device.cuh"
#include "kernels.h"

namespace pkvd {
namespace gqa {


constexpr unsigned kFull = 0xffffffffu;
constexpr int BLK = kGqaBlockTokens;

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// ------------------------------------------------------------ smem layout

// Byte offset, inside a K or V tile, of the 16-byte column chunk cc of row r.
template <int D, bool TILES>
__device__ __forceinline__ int chunk_off(int r, int cc) {
  if constexpr (TILES)
    return (cc >> 3) * 2048 + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
  else
    return r * gqa_row_pitch(D) + cc * 16;
}

// ----------------------------------------------------------- block streaming

// Pool row of token (block blk, row r) of the item for its KV head, or 0 past
// the item's end. The page-table load and the division by the page size
// happen here, ahead of use, not when the copy is issued.
__device__ __forceinline__ int64_t kv_row_of(const Stage1Args& a, const pkvd_work_item& it,
                                             const int32_t* pt, int blk, int nblk, int r) {
  const int tok = it.tok_begin + blk * BLK + r;
  if (blk >= nblk || tok >= it.tok_end) return 0;
  const int pidx = tok / a.page_size;
  int page = __ldg(pt + pidx);
  if (a.checks && (page < 0 || page >= a.num_pool_pages)) {
    atomicOr(a.status, kStatusBadPage);
    page = 0;
  }
  return (static_cast<int64_t>(page) * a.kv_heads + it.unit) * a.page_size +
         (tok - pidx * a.page_size);
}

// Issue the copies of block blk into `stage`. TILES: lane 0 copies the K
// tile, lane 1 the V tile (row = the block's first pool row). Otherwise lanes
// 0-15 copy K rows and lanes 16-31 V rows (row = this lane's token's row).
template <int D, bool TILES>
__device__ __forceinline__ void issue_block(const Stage1Args& a, const KvTensorMaps& maps,
                                            int blk, int n, int64_t row, uint8_t* stage,
                                            uint32_t bar, int lane) {
  constexpr int ROWB = D * 2;
  constexpr int TB = gqa_tile_bytes(D, TILES);
  const int nv = min(BLK, n - blk * BLK);
  if constexpr (TILES) {
    if (lane == 0) mbar_arrive_expect_tx(bar, 2u * TB);
    __syncwarp();
    if (lane < 2)
      tma_load_3d(smem_addr(stage + lane * TB), lane ? &maps.v : &maps.k, 0,
                  static_cast<int32_t>(row), 0, bar);
  } else {
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nv * ROWB * 2));
    __syncwarp();
    const int r = lane & (BLK - 1);
    const bool is_v = lane >= BLK;
    if (r < nv) {
      const uint8_t* pool = static_cast<const uint8_t*>(is_v ? a.v : a.k);
      const int64_t pitch_bytes = (is_v ? a.v_pitch : a.k_pitch) * 2;
      bulk_copy_g2s(smem_addr(stage + (is_v ? TB : 0) + r * gqa_row_pitch(D)),
                    pool + row * pitch_bytes, ROWB, bar);
    }
  }
}

// Pool rows of a warp's first blocks: the SPW blocks it copies first and
// the PF blocks after them (the page-id window). Loaded at the very start of
// the block, before the barrier set-up, so that the page-table round trip
// overlaps it.
template <int D, bool TILES>
struct WarpRows {
  static constexpr int SPW = gqa_stages_per_warp(D);
  static constexpr int PF = 4;     // page-id window (blocks)
  int64_t first[SPW];
  int64_t rows[PF];
  __device__ __forceinline__ WarpRows(const Stage1Args& a, const pkvd_work_item& it, int warp,
                                      int lane) {
    constexpr int W = gqa_warps(D);
    const int n = it.tok_end - it.tok_begin;
    const int nblk = (n + BLK - 1) / BLK;
    const int r = TILES ? 0 : (lane & (BLK - 1));
    const int32_t* pt = a.page_table + static_cast<int64_t>(it.request) * a.pt_stride;
#pragma unroll
    for (int s = 0; s < SPW; ++s) first[s] = kv_row_of(a, it, pt, warp + W * s, nblk, r);
#pragma unroll
    for (int i = 0; i < PF; ++i) rows[i] = kv_row_of(a, it, pt, warp + W * (SPW + i), nblk, r);
  }
};

// The per-warp pipeline: issue this warp's first SPW blocks, then for each of
// its blocks wait, run `process(nv, stage, k0)` (nv valid rows, k0 = the
// block's first token relative to the item), and refill the stage with the
// block SPW further on (prefetching further blocks into L2 was measured and
// did not pay). Returns false when a wait ran out (after waiting, bounded,
// for this warp's copies still in flight). The caller's `prologue` runs once
// the first copies are in flight.
template <int D, bool TILES, typename P, typename F>
__device__ __forceinline__ bool gqa_warp_loop(const Stage1Args& a, const KvTensorMaps& maps,
                                              const pkvd_work_item& it, WarpRows<D, TILES>& wr,
                                              uint8_t* stages, uint32_t bars, int warp, int lane,
                                              P&& prologue, F&& process) {
  constexpr int W = gqa_warps(D);
  constexpr int SPW = gqa_stages_per_warp(D);
  constexpr int SB = gqa_stage_bytes(D, TILES);
  constexpr int PF = WarpRows<D, TILES>::PF;
  const int n = it.tok_end - it.tok_begin;
  const int nblk = (n + BLK - 1) / BLK;
  const int nmine = nblk > warp ? (nblk - warp + W - 1) / W : 0;
  const int r = TILES ? 0 : (lane & (BLK - 1));
  const int32_t* pt = a.page_table + static_cast<int64_t>(it.request) * a.pt_stride;
  auto blk_of = [&](int k) { return warp + W * k; };
  auto stage_of = [&](int k) { return stages + (warp * SPW + k % SPW) * SB; };
  auto bar_of = [&](int k) { return bars + 8u * (warp * SPW + k % SPW); };
  int64_t (&rows)[PF] = wr.rows;

#pragma unroll
  for (int s = 0; s < SPW; ++s)
    if (s < nmine)
      issue_block<D, TILES>(a, maps, blk_of(s), n, wr.first[s], stage_of(s), bar_of(s), lane);
  prologue();

  bool ok = true;
  int k = 0;
  while (ok && k < nmine) {
#pragma unroll
    for (int i = 0; i < PF; ++i) {
      if (ok && k < nmine) {
        if (!__all_sync(kFull, mbar_wait(bar_of(k), (k / SPW) & 1))) {
          ok = false;
        } else {
          const int blk = blk_of(k);
          process(min(BLK, n - blk * BLK), stage_of(k), blk * BLK);
          __syncwarp();
          if (k + SPW < nmine)
            issue_block<D, TILES>(a, maps, blk_of(k + SPW), n, rows[i], stage_of(k), bar_of(k),
                                  lane);
          rows[i] = kv_row_of(a, it, pt, blk_of(k + SPW + PF), nblk, r);
          ++k;
        }
      }
    }
  }
  if (!ok && lane == 0) {
    // copies of this warp still in flight must land before the block exits
    for (int kk = k; kk < min(nmine, k + SPW); ++kk) mbar_wait(bar_of(kk), (kk / SPW) & 1);
  }
  return ok;
}

// Shared-memory carve-up: [stages (1 KB aligned)][barriers][p buffers][query tile].
template <int D, int G, bool TILES>
struct GqaSmem {
  uint8_t* stages;
  uint32_t bars;
  float* pbuf;
  uint8_t* qtile;
  __device__ __forceinline__ explicit GqaSmem(uint8_t* raw) {
    const uint32_t base = smem_addr(raw);
    stages = raw + ((kTileAlign - (base & (kTileAlign - 1))) & (kTileAlign - 1));
    uint8_t* b = stages + gqa_stage_area_bytes(D, G, TILES);
    bars = smem_addr(b);
    pbuf = reinterpret_cast<float*>(b + kBarrierBytes);
    qtile = b + kBarrierBytes + gqa_pbuf_bytes(D, G);
  }
};

// Barriers of all stages, initialised by thread 0 before any copy.
template <int D>
__device__ __forceinline__ void init_stage_barriers(uint32_t bars) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < gqa_stages(D); ++s) mbar_init(bars + 8 * s, 1);
    fence_barrier_init();
  }
  __syncthreads();
}

// Load CH consecutive 16-bit elements (8 or 4) and widen them to fp32.
template <typename T, int CH>
__device__ __forceinline__ void load_row(const uint8_t* p, float (&f)[CH]) {
  if constexpr (CH == 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    float2 x;
    x = unpack2<T>(w.x); f[0] = x.x; f[1] = x.y;
    x = unpack2<T>(w.y); f[2] = x.x; f[3] = x.y;
    x = unpack2<T>(w.z); f[4] = x.x; f[5] = x.y;
    x = unpack2<T>(w.w); f[6] = x.x; f[7] = x.y;
  } else {
    static_assert(CH == 4, "4 or 8 columns per lane");
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    float2 x;
    x = unpack2<T>(w.x); f[0] = x.x; f[1] = x.y;
    x = unpack2<T>(w.y); f[2] = x.x; f[3] = x.y;
  }
}

// Byte offset of lane `lane`'s CH columns of row `key` (CH = D / 32).
template <int D, bool TILES>
__device__ __forceinline__ int lane_cols_off(int key, int lane) {
  constexpr int CH = D / 32;
  if constexpr (CH == 8)
    return chunk_off<D, TILES>(key, lane);
  else
    return chunk_off<D, TILES>(key, lane >> 1) + (lane & 1) * 8;
}

// Transposing xor butterfly over N = 2^k partial sums per lane. Slot i of
// lane l must hold the partial of value index i ^ (l >> (5 - k)); after the
// halving steps (masks 16 .. 32/N) slot 0 holds value index l >> (5 - k)
// summed over 32 / (32/N) lanes, and the remaining masks finish the sum.
// The order of every addition is fixed by the lane id alone.
template <int N>
__device__ __forceinline__ float xfold(float (&v)[N]) {
  constexpr int LOGN = ilog2(N);
#pragma unroll
  for (int step = 0; step < LOGN; ++step) {
    const int half = N >> (step + 1);
    const int m = 16 >> step;
#pragma unroll
    for (int i = 0; i < half; ++i) v[i] += __shfl_xor_sync(kFull, v[i + half], m);
  }
#pragma unroll
  for (int m = (16 >> LOGN); m >= 1; m >>= 1) v[0] += __shfl_xor_sync(kFull, v[0], m);
  return v[0];
}

// Fixed-order merge of the warps' (m, l, o) for the item's NQ = q_len x G
// (query token, head) columns, column n = j * G + i being query token j's
// head kvh * G + i; writes the normalised partial rows and their
// log2-sum-exp2. mg holds [W][NQ] output rows
// of gqa_merge_row(D) floats, then [W][G] maxima, [W][G] sums and room for
// [W][G] weights. Thread h < G first folds head h's statistics in warp order
// into one weight per warp, w_wh = 2^(m_wh - M_h) / sum_w' 2^(m_w'h - M_h) l_w'h,
// and the head's lse; then every output element is sum_w w_wh o_wh[d] in
// warp order, four columns per thread.
// CAUSAL: several query tokens (q_len > 1); otherwise NQ == G and column n
// is head kvh * G + n.
template <int D, bool CAUSAL>
__device__ __forceinline__ void merge_warps(const Stage1Args& a, const pkvd_work_item& it,
                                            int G, int NQ, float* mg) {
  constexpr int W = gqa_warps(D);
  constexpr int RS = gqa_merge_row(D);
  const float* mm = mg + W * NQ * RS;
  const float* ml = mm + W * NQ;
  float* wt = mg + W * NQ * RS + 2 * W * NQ;
  const int VH = a.q_len * a.heads;
  // (query token, head) row of column n within the request's VH rows
  auto vrow = [&](int n) {
    return CAUSAL ? (n / G) * a.heads + it.unit * G + n % G : it.unit * G + n;
  };
  const int64_t row0 = static_cast<int64_t>(it.partial_row) * VH;
  if (threadIdx.x < NQ) {
    const int h = threadIdx.x;
    const int G_ = NQ;   // stride of the [W][NQ] statistics
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, mm[w * G_ + h]);
    float e[W];
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      e[w] = M == -INFINITY ? 0.f : exp2f(mm[w * G_ + h] - M);
      den += e[w] * ml[w * G_ + h];
    }
    const float inv = M == -INFINITY ? 0.f : 1.f / den;
#pragma unroll
    for (int w = 0; w < W; ++w) wt[w * G_ + h] = e[w] * inv;
    a.lse_part[vrow(h) * a.lse_stride + it.partial_row] =
        M == -INFINITY ? -INFINITY : M + log2f(den);
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < NQ * (D / 4); idx += W * 32) {
    const int h = idx / (D / 4), d = (idx % (D / 4)) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float c = wt[w * NQ + h];
      const float4 o = *reinterpret_cast<const float4*>(mg + (w * NQ + h) * RS + d);
      acc.x = fmaf(c, o.x, acc.x);
      acc.y = fmaf(c, o.y, acc.y);
      acc.z = fmaf(c, o.z, acc.z);
      acc.w = fmaf(c, o.w, acc.w);
    }
    *reinterpret_cast<float4*>(a.o_part + (row0 + vrow(h)) * a.dv + d) = acc;
  }
}

}  // namespace gqa
}  // namespace pkvd
