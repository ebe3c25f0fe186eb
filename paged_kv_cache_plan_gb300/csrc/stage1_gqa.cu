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
// Two consumers (the TensorFold pull 1932 page, "What this changes": separate
// kernel symbols per variant rather than a grid-uniform branch):
//   * gqa_fma: fp32 FMA. A warp scores four keys per pass; lane l holds
//     D/32 columns of each row and of every head's query, and the 4 x G
//     partial dot products are folded across the warp with xor shuffles
//     from 16 down to 1 in a fixed order (the same page: four keys a warp,
//     xor-fold wave sums). The fold is a transposing butterfly, so each
//     lane ends with one (key, head) score and no broadcast is needed.
//   * gqa_mma: mma.sync m16n8k16 with the 16 keys of a block as M and the
//     head group as N (8 per n-tile): S^T = K Q^T, then O^T += V^T P^T with
//     P^T formed in registers by movmatrix, as a 16-bit high part plus a
//     16-bit low remainder (two products), so P keeps ~16 significant bits.
#include "device.cuh"
#include "kernels.h"

namespace pkvd {
namespace {

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

// Warm L2 with block blk's K and V tiles (TILES only; lanes 0 and 1).
template <int D, bool TILES>
__device__ __forceinline__ void prefetch_block(const KvTensorMaps& maps, int64_t row, int lane) {
  if constexpr (TILES) {
    if (lane < 2) tma_prefetch_l2_3d(lane ? &maps.v : &maps.k, 0, static_cast<int32_t>(row), 0);
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
// its blocks wait, run `process(nv, stage)`, and refill the stage with the
// block SPW further on. With TILES, the blocks PFL beyond the next refill are
// also prefetched into L2 (off: it did not pay). Returns false when a wait ran
// out (after waiting, bounded, for this warp's copies still in flight). The
// caller's `prologue` runs once the first copies are in flight.
template <int D, bool TILES, typename P, typename F>
__device__ __forceinline__ bool gqa_warp_loop(const Stage1Args& a, const KvTensorMaps& maps,
                                              const pkvd_work_item& it, WarpRows<D, TILES>& wr,
                                              uint8_t* stages, uint32_t bars, int warp, int lane,
                                              P&& prologue, F&& process) {
  constexpr int W = gqa_warps(D);
  constexpr int SPW = gqa_stages_per_warp(D);
  constexpr int SB = gqa_stage_bytes(D, TILES);
  constexpr int PF = WarpRows<D, TILES>::PF;
  constexpr int PFL = 0;              // L2 prefetch distance past the next refill (off)
  static_assert(PFL < PF, "prefetched rows come from the page-id window");
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
#pragma unroll
  for (int i = 0; i < PFL; ++i)
    if (SPW + i < nmine) prefetch_block<D, TILES>(maps, rows[i], lane);
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
          process(min(BLK, n - blk * BLK), stage_of(k));
          __syncwarp();
          if (k + SPW < nmine)
            issue_block<D, TILES>(a, maps, blk_of(k + SPW), n, rows[i], stage_of(k), bar_of(k),
                                  lane);
          if (PFL > 0 && k + SPW + PFL < nmine)
            prefetch_block<D, TILES>(maps, rows[(i + PFL) % PF], lane);
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

// Fixed-order merge of the warps' (m, l, o) for G heads; writes the
// normalised partial row and its log2-sum-exp2. mg holds [W][G] output rows
// of gqa_merge_row(D) floats, then [W][G] maxima, [W][G] sums and room for
// [W][G] weights. Thread h < G first folds head h's statistics in warp order
// into one weight per warp, w_wh = 2^(m_wh - M_h) / sum_w' 2^(m_w'h - M_h) l_w'h,
// and the head's lse; then every output element is sum_w w_wh o_wh[d] in
// warp order, four columns per thread.
template <int D>
__device__ __forceinline__ void merge_warps(const Stage1Args& a, const pkvd_work_item& it, int G,
                                            int hq0, float* mg) {
  constexpr int W = gqa_warps(D);
  constexpr int RS = gqa_merge_row(D);
  const float* mm = mg + W * G * RS;
  const float* ml = mm + W * G;
  float* wt = mg + W * G * RS + 2 * W * G;
  const int64_t row0 = static_cast<int64_t>(it.partial_row) * a.heads + hq0;
  if (threadIdx.x < G) {
    const int h = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, mm[w * G + h]);
    float e[W];
    float den = 0.f;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      e[w] = M == -INFINITY ? 0.f : exp2f(mm[w * G + h] - M);
      den += e[w] * ml[w * G + h];
    }
    const float inv = M == -INFINITY ? 0.f : 1.f / den;
#pragma unroll
    for (int w = 0; w < W; ++w) wt[w * G + h] = e[w] * inv;
    a.lse_part[(hq0 + h) * a.lse_stride + it.partial_row] =
        M == -INFINITY ? -INFINITY : M + log2f(den);
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * (D / 4); idx += W * 32) {
    const int h = idx / (D / 4), d = (idx % (D / 4)) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const float c = wt[w * G + h];
      const float4 o = *reinterpret_cast<const float4*>(mg + (w * G + h) * RS + d);
      acc.x = fmaf(c, o.x, acc.x);
      acc.y = fmaf(c, o.y, acc.y);
      acc.z = fmaf(c, o.z, acc.z);
      acc.w = fmaf(c, o.w, acc.w);
    }
    *reinterpret_cast<float4*>(a.o_part + (row0 + h) * a.dv + d) = acc;
  }
}

// ---------------------------------------------------------------- FMA variant

template <typename T, int D, int G, bool TILES>
__global__ void __launch_bounds__(gqa_threads(D), 1)
    gqa_fma(const __grid_constant__ Stage1Args a, const __grid_constant__ KvTensorMaps maps) {
  constexpr int W = gqa_warps(D);
  constexpr int TB = gqa_tile_bytes(D, TILES);
  constexpr int CH = D / 32;              // columns per lane
  constexpr int N = 4 * G;                // partial sums per four-key pass
  constexpr int SHIFT = 5 - ilog2(N);     // lane >> SHIFT = value index held after the fold
  constexpr int LOGG = ilog2(G);
  constexpr int GP = G < 8 ? 8 : G;       // p-buffer row stride (floats)
  static_assert(N <= 32, "at most 8 heads per KV head on the FMA path");
  static_assert(gqa_merge_bytes(D, G) <= gqa_stage_area_bytes(D, G, TILES),
                "merge area must fit in the stage area");

  extern __shared__ uint8_t smem_raw[];
  if (TILES && threadIdx.x == 0) {
    tma_prefetch_desc(&maps.k);
    tma_prefetch_desc(&maps.v);
  }
  const pkvd_work_item it = a.items[blockIdx.x];
  pdl_launch_dependents();
  const GqaSmem<D, G, TILES> sm(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WarpRows<D, TILES> wr(a, it, warp, lane);
  init_stage_barriers<D>(sm.bars);

  float* pb = sm.pbuf + warp * (BLK * GP + GP);
  const int kvh = it.unit;
  const int f = lane >> SHIFT;            // (key in pass, head) this lane ends with
  const int fk = f >> LOGG;
  const int fh = f & (G - 1);
  const bool primary = (lane & ((1 << SHIFT) - 1)) == 0;

  // Query rows of the group, head order permuted by fh so that the partial
  // in slot (kk, h) is the one of value index (kk, h) ^ f (loaded once the
  // first KV copies are in flight).
  float qr[G][CH];
  auto load_q = [&]() {
    const uint8_t* qb = static_cast<const uint8_t*>(a.q) +
                        ((static_cast<int64_t>(it.request) * a.heads + kvh * G) * D + lane * CH) * 2;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      load_row<T, CH>(qb + static_cast<int64_t>(h ^ fh) * D * 2, qr[h]);
#pragma unroll
      for (int c = 0; c < CH; ++c) qr[h][c] *= a.scale_log2;
    }
  };

  float acc[G][CH];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int c = 0; c < CH; ++c) acc[h][c] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;

  const bool ok = gqa_warp_loop<D, TILES>(a, maps, it, wr, sm.stages, sm.bars, warp, lane, load_q,
                                          [&](int nv, const uint8_t* ks) {
    const uint8_t* vs = ks + TB;
    float sc[4];
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
      float part[N];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        float kf[CH];
        load_row<T, CH>(ks + lane_cols_off<D, TILES>(pass * 4 + (kk ^ fk), lane), kf);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float d = 0.f;
#pragma unroll
          for (int c = 0; c < CH; ++c) d = fmaf(qr[h][c], kf[c], d);
          part[kk * G + h] = d;
        }
      }
      sc[pass] = xfold<N>(part);
      if (pass * 4 + fk >= nv) sc[pass] = -INFINITY;
    }

    // Online softmax for this lane's head; lanes differing in bits 3-4 hold
    // the other keys of the pass.
    float bm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
    bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
    const float m_new = fmaxf(m_run, bm);
    const float alpha = exp2f(m_run - m_new);
    float p[4];
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) p[pass] = exp2f(sc[pass] - m_new);
    l_run = l_run * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
    m_run = m_new;

    if (primary) {
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) pb[(pass * 4 + fk) * GP + fh] = p[pass];
      if (fk == 0) pb[BLK * GP + fh] = alpha;
    }
    __syncwarp();

    if (!__all_sync(kFull, alpha == 1.f)) {   // some head's running max moved
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float al = pb[BLK * GP + h];
#pragma unroll
        for (int c = 0; c < CH; ++c) acc[h][c] *= al;
      }
    }
#pragma unroll
    for (int key = 0; key < BLK; ++key) {
      if (key < nv) {
        float vf[CH];
        load_row<T, CH>(vs + lane_cols_off<D, TILES>(key, lane), vf);
        float pk[GP];
#pragma unroll
        for (int h4 = 0; h4 < GP / 4; ++h4) {
          const float4 x = *reinterpret_cast<const float4*>(pb + key * GP + 4 * h4);
          pk[4 * h4 + 0] = x.x; pk[4 * h4 + 1] = x.y; pk[4 * h4 + 2] = x.z; pk[4 * h4 + 3] = x.w;
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int c = 0; c < CH; ++c) acc[h][c] = fmaf(pk[h], vf[c], acc[h][c]);
      }
    }
    __syncwarp();   // the p buffer is rewritten by the next block
  });

  // Head totals of l over the lanes that held the other keys.
  l_run += __shfl_xor_sync(kFull, l_run, 16);
  l_run += __shfl_xor_sync(kFull, l_run, 8);

  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusTimeout);
    return;
  }
  // All stages are consumed: reuse them for the cross-warp merge.
  constexpr int RS = gqa_merge_row(D);
  float* mg = reinterpret_cast<float*>(sm.stages);
  float* mo = mg + warp * G * RS;
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int c = 0; c < CH; c += 4)
      *reinterpret_cast<float4*>(mo + h * RS + lane * CH + c) =
          make_float4(acc[h][c], acc[h][c + 1], acc[h][c + 2], acc[h][c + 3]);
  if (primary && fk == 0) {
    mg[W * G * RS + warp * G + fh] = m_run;
    mg[W * G * RS + W * G + warp * G + fh] = l_run;
  }
  __syncthreads();
  merge_warps<D>(a, it, G, kvh * G, mg);
}

// ---------------------------------------------------------------- MMA variant

template <typename T, int D, int NT, bool TILES>
__global__ void __launch_bounds__(gqa_threads(D), NT == 1 ? 2 : 1)
    gqa_mma(const __grid_constant__ Stage1Args a, const __grid_constant__ KvTensorMaps maps) {
  constexpr int W = gqa_warps(D);
  constexpr int TB = gqa_tile_bytes(D, TILES);
  constexpr int KS = D / 16;              // k-steps of the score product = m-tiles of O^T
  constexpr int GMAX = 8 * NT;
  static_assert(gqa_merge_bytes(D, GMAX) <= gqa_stage_area_bytes(D, GMAX, TILES),
                "merge area must fit in the stage area");

  extern __shared__ uint8_t smem_raw[];
  if (TILES && threadIdx.x == 0) {
    tma_prefetch_desc(&maps.k);
    tma_prefetch_desc(&maps.v);
  }
  const pkvd_work_item it = a.items[blockIdx.x];
  pdl_launch_dependents();
  const GqaSmem<D, GMAX, TILES> sm(smem_raw);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = a.heads / a.kv_heads;
  const int kvh = it.unit;

  WarpRows<D, TILES> wr(a, it, warp, lane);
  init_stage_barriers<D>(sm.bars);

  // The group's query rows [GMAX][D] in padded rows (zero past G): the
  // source of the Q^T B fragments, read with ldmatrix each block. Loaded by
  // the whole block once every warp has its first KV copies in flight (all
  // warps run this exactly once, so the barrier inside is safe).
  auto load_q = [&]() {
    constexpr int CHUNKS = D * 2 / 16;
    const uint8_t* qg = static_cast<const uint8_t*>(a.q) +
                        (static_cast<int64_t>(it.request) * a.heads + kvh * G) * D * 2;
    for (int i = threadIdx.x; i < GMAX * CHUNKS; i += gqa_threads(D)) {
      const int h = i / CHUNKS, c = i % CHUNKS;
      *reinterpret_cast<uint4*>(sm.qtile + h * gqa_row_pitch(D) + c * 16) =
          h < G ? __ldg(reinterpret_cast<const uint4*>(qg + static_cast<int64_t>(h) * D * 2) + c)
                : make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
  };

  float o[KS][NT][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) o[mt][nt][i] = 0.f;
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      m_run[nt][e] = -INFINITY;
      l_run[nt][e] = 0.f;
    }

  // ldmatrix row / chunk of this lane: K (A of S^T) rows 0-15 with the high
  // lanes on the second 8 columns; V^T (A of O^T, transposing load) keys
  // 0-7 / 8-15 on lane bit 4 with the second 8 columns on lane bit 3.
  const int kr = lane & 15, khi = lane >> 4;
  const int vr = ((lane >> 4) & 1) * 8 + (lane & 7), vhi = (lane >> 3) & 1;
  const uint32_t qaddr = smem_addr(sm.qtile + (lane & 7) * gqa_row_pitch(D) + (lane >> 3) * 16);

  const bool ok = gqa_warp_loop<D, TILES>(a, maps, it, wr, sm.stages, sm.bars, warp, lane, load_q,
                                          [&](int nv, uint8_t* ks_) {
    uint8_t* vs = ks_ + TB;
    if (nv < BLK) {
      // P is zero past the end, but those V rows could hold non-finite bits.
      constexpr int CHUNKS = D * 2 / 16;
      for (int i = lane; i < (BLK - nv) * CHUNKS; i += 32)
        *reinterpret_cast<uint4*>(vs + chunk_off<D, TILES>(nv + i / CHUNKS, i % CHUNKS)) =
            make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
      __syncwarp();
    }

    // S^T = K Q^T, two accumulator chains per n-tile.
    float c[NT][2][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int i = 0; i < 4; ++i) c[nt][ch][i] = 0.f;
    const uint32_t kbase = smem_addr(ks_);
#pragma unroll
    for (int k = 0; k < KS; k += 2) {
      // Q^T B fragments of k-steps k, k+1 (ldmatrix of the query rows:
      // matrix m = d columns 16k + 8m .. +7 of heads nt*8 .. nt*8+7)
      uint32_t qf[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        ldmatrix_x4(qaddr + nt * 8 * gqa_row_pitch(D) + k * 32, qf[nt][0], qf[nt][1], qf[nt][2],
                    qf[nt][3]);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        uint32_t af[4];
        ldmatrix_x4(kbase + chunk_off<D, TILES>(kr, 2 * (k + kk) + khi), af[0], af[1], af[2],
                    af[3]);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
          mma_16816<T>(c[nt][kk], af, qf[nt][2 * kk], qf[nt][2 * kk + 1]);
      }
    }

    const bool v0 = g < nv, v1 = g + 8 < nv;
    uint32_t pf[NT][2][2];   // [n-tile][high, low part][k rows 0-7, 8-15]
    float alpha[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float s0 = v0 ? (c[nt][0][e] + c[nt][1][e]) * a.scale_log2 : -INFINITY;
        const float s1 = v1 ? (c[nt][0][2 + e] + c[nt][1][2 + e]) * a.scale_log2 : -INFINITY;
        float bm = fmaxf(s0, s1);
        bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
        const float m_new = fmaxf(m_run[nt][e], bm);
        alpha[nt][e] = exp2f(m_run[nt][e] - m_new);
        m_run[nt][e] = m_new;
        p[e] = exp2f(s0 - m_new);
        p[2 + e] = exp2f(s1 - m_new);
        l_run[nt][e] = l_run[nt][e] * alpha[nt][e] + (p[e] + p[2 + e]);
      }
      // C fragment (keys x heads) -> B fragment of P^T (keys as k, heads as n),
      // as a 16-bit high part plus the 16-bit rounding of the remainder.
      const uint32_t hi0 = pack2<T>(p[0], p[1]), hi1 = pack2<T>(p[2], p[3]);
      const float2 r0 = unpack2<T>(hi0), r1 = unpack2<T>(hi1);
      pf[nt][0][0] = movmatrix_trans(hi0);
      pf[nt][0][1] = movmatrix_trans(hi1);
      pf[nt][1][0] = movmatrix_trans(pack2<T>(p[0] - r0.x, p[1] - r0.y));
      pf[nt][1][1] = movmatrix_trans(pack2<T>(p[2] - r1.x, p[3] - r1.y));
    }

    bool same = true;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) same = same && alpha[nt][0] == 1.f && alpha[nt][1] == 1.f;
    if (!__all_sync(kFull, same)) {   // some head's running max moved
#pragma unroll
      for (int mt = 0; mt < KS; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          o[mt][nt][0] *= alpha[nt][0];
          o[mt][nt][1] *= alpha[nt][1];
          o[mt][nt][2] *= alpha[nt][0];
          o[mt][nt][3] *= alpha[nt][1];
        }
    }
    // O^T += V^T P^T: A = V^T by transposing ldmatrix of the V rows.
    const uint32_t vbase = smem_addr(vs);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t vf[4];
      ldmatrix_x4_trans(vbase + chunk_off<D, TILES>(vr, 2 * mt + vhi), vf[0], vf[1], vf[2],
                        vf[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_16816<T>(o[mt][nt], vf, pf[nt][0][0], pf[nt][0][1]);
        mma_16816<T>(o[mt][nt], vf, pf[nt][1][0], pf[nt][1][1]);
      }
    }
  });

#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float l = l_run[nt][e];
      l += __shfl_xor_sync(kFull, l, 4);
      l += __shfl_xor_sync(kFull, l, 8);
      l += __shfl_xor_sync(kFull, l, 16);
      l_run[nt][e] = l;
    }

  if (__syncthreads_or(!ok)) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusTimeout);
    return;
  }
  constexpr int RS = gqa_merge_row(D);
  float* mg = reinterpret_cast<float*>(sm.stages);
  float* mo = mg + warp * G * RS;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h0 = nt * 8 + 2 * t, d0 = mt * 16 + g;
      if (h0 < G) {
        mo[h0 * RS + d0] = o[mt][nt][0];
        mo[h0 * RS + d0 + 8] = o[mt][nt][2];
      }
      if (h0 + 1 < G) {
        mo[(h0 + 1) * RS + d0] = o[mt][nt][1];
        mo[(h0 + 1) * RS + d0 + 8] = o[mt][nt][3];
      }
    }
  if (g == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = nt * 8 + 2 * t + e;
        if (h < G) {
          mg[W * G * RS + warp * G + h] = m_run[nt][e];
          mg[W * G * RS + W * G + warp * G + h] = l_run[nt][e];
        }
      }
  }
  __syncthreads();
  merge_warps<D>(a, it, G, kvh * G, mg);
}

template <typename T, int D, int G, bool TILES>
void fma_entry(KernelEntry* e) {
  e->func = reinterpret_cast<const void*>(&gqa_fma<T, D, G, TILES>);
  e->threads = gqa_threads(D);
  e->smem = gqa_smem_bytes(D, G, TILES);
  e->block_tokens = kGqaBlockTokens;
  e->stages = gqa_stages(D);
  e->tiles = TILES;
}

template <typename T, int D, int NT, bool TILES>
void mma_entry(KernelEntry* e) {
  e->func = reinterpret_cast<const void*>(&gqa_mma<T, D, NT, TILES>);
  e->threads = gqa_threads(D);
  e->smem = gqa_smem_bytes(D, 8 * NT, TILES);
  e->block_tokens = kGqaBlockTokens;
  e->stages = gqa_stages(D);
  e->tiles = TILES;
}

template <typename T, int D, bool TILES>
bool fma_by_group(int group, KernelEntry* e) {
  switch (group) {
    case 1: fma_entry<T, D, 1, TILES>(e); return true;
    case 2: fma_entry<T, D, 2, TILES>(e); return true;
    case 4: fma_entry<T, D, 4, TILES>(e); return true;
    case 8: fma_entry<T, D, 8, TILES>(e); return true;
    default: return false;
  }
}

template <typename T, bool TILES>
bool fma_by_dim(int head_dim, int group, KernelEntry* e) {
  if (head_dim == 128) return fma_by_group<T, 128, TILES>(group, e);
  if (head_dim == 256) return fma_by_group<T, 256, TILES>(group, e);
  return false;
}

template <typename T, bool TILES>
bool mma_by_dim(int head_dim, int group, KernelEntry* e) {
  if (group < 1 || group > 16) return false;
  const bool two = group > 8;
  if (head_dim == 128) {
    two ? mma_entry<T, 128, 2, TILES>(e) : mma_entry<T, 128, 1, TILES>(e);
    return true;
  }
  if (head_dim == 256) {
    two ? mma_entry<T, 256, 2, TILES>(e) : mma_entry<T, 256, 1, TILES>(e);
    return true;
  }
  return false;
}

}  // namespace

bool gqa_fma_kernel(int dtype, int head_dim, int group, bool tiles, KernelEntry* e) {
  if (dtype == PKVD_FP16)
    return tiles ? fma_by_dim<__half, true>(head_dim, group, e)
                 : fma_by_dim<__half, false>(head_dim, group, e);
  return tiles ? fma_by_dim<__nv_bfloat16, true>(head_dim, group, e)
               : fma_by_dim<__nv_bfloat16, false>(head_dim, group, e);
}

bool gqa_mma_kernel(int dtype, int head_dim, int group, bool tiles, KernelEntry* e) {
  if (dtype == PKVD_FP16)
    return tiles ? mma_by_dim<__half, true>(head_dim, group, e)
                 : mma_by_dim<__half, false>(head_dim, group, e);
  return tiles ? mma_by_dim<__nv_bfloat16, true>(head_dim, group, e)
               : mma_by_dim<__nv_bfloat16, false>(head_dim, group, e);
}

}  // namespace pkvd
