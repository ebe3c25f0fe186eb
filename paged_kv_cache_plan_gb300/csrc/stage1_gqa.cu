// Stage 1 for GQA: one block per work item (request b, KV head, split s).
// The block streams the split's K and V rows through a ring of shared-memory
// stages and leaves, for each of the group's query heads, the normalised P.V
// partial and its log2-sum-exp2 (scores are pre-multiplied by log2 e).
//
// Warp roles (warp-specialised):
//   * producer warp: reads page ids ahead of use (a register window of
//     PF blocks, so the page-number loads never wait at the head of the
//     loop -- the aiter pull 4758 page, Technical Details 1: retire only
//     the page-number copy early, keep several KV blocks in flight), then
//     issues one bulk TMA copy per K or V row into a padded shared-memory
//     row (lanes 0-15: K rows, lanes 16-31: V rows of a 16-token block).
//     Every stage completes on its own mbarrier, so up to STAGES blocks are
//     in flight at once.
//   * 4 consumer warps: take whole 16-token blocks round-robin, each with
//     its own online softmax; a fixed-order merge of the warps ends the item.
//
// Two consumers exist (the TensorFold pull 1932 page, "What this changes":
// separate kernel symbols per variant rather than a grid-uniform branch):
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
constexpr int kPrefetchBlocks = 8;

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

// ------------------------------------------------------------------ producer

template <int D, int STAGES>
__device__ __forceinline__ void gqa_producer(const Stage1Args& a, const pkvd_work_item& it,
                                             uint8_t* stages, uint32_t bar_full,
                                             uint32_t bar_empty, int lane) {
  constexpr int BLK = kGqaBlockTokens;
  constexpr int ROWB = D * 2;
  constexpr int PITCH = gqa_row_pitch(D);
  constexpr int SB = gqa_stage_bytes(D);
  constexpr int PF = kPrefetchBlocks;

  const int n = it.tok_end - it.tok_begin;
  const int nblk = (n + BLK - 1) / BLK;
  const int r = lane & (BLK - 1);
  const bool is_v = lane >= BLK;
  const uint8_t* pool = static_cast<const uint8_t*>(is_v ? a.v : a.k);
  const int64_t pitch_bytes = (is_v ? a.v_pitch : a.k_pitch) * 2;
  const int32_t* pt = a.page_table + static_cast<int64_t>(it.request) * a.pt_stride;

  auto fetch = [&](int j) -> int {
    const int tok = it.tok_begin + j * BLK + r;
    if (j >= nblk || tok >= it.tok_end) return 0;
    int page = __ldg(pt + tok / a.page_size);
    if (a.checks && (page < 0 || page >= a.num_pool_pages)) {
      atomicOr(a.status, kStatusBadPage);
      page = 0;
    }
    return page;
  };

  int ids[PF];
#pragma unroll
  for (int i = 0; i < PF; ++i) ids[i] = fetch(i);

  int j = 0;
  bool ok = true;
  for (; j < nblk; ++j) {
    const int page = ids[0];
#pragma unroll
    for (int i = 0; i < PF - 1; ++i) ids[i] = ids[i + 1];
    ids[PF - 1] = fetch(j + PF);

    const int s = j % STAGES;
    if (j >= STAGES) {
      bool freed = true;
      if (lane == 0) freed = mbar_wait(bar_empty + 8 * s, ((j / STAGES) & 1) ^ 1);
      if (!__shfl_sync(kFull, freed, 0)) {
        ok = false;
        break;
      }
    }
    const int nv = min(BLK, n - j * BLK);
    if (lane == 0) mbar_arrive_expect_tx(bar_full + 8 * s, static_cast<uint32_t>(nv * ROWB * 2));
    __syncwarp();
    if (r < nv) {
      const int tok = it.tok_begin + j * BLK + r;
      const int64_t row =
          (static_cast<int64_t>(page) * a.kv_heads + it.unit) * a.page_size + tok % a.page_size;
      const uint32_t dst = smem_addr(stages + s * SB + (is_v ? BLK * PITCH : 0) + r * PITCH);
      bulk_copy_g2s(dst, pool + row * pitch_bytes, ROWB, bar_full + 8 * s);
    }
  }
  if (!ok && lane == 0) atomicOr(a.status, kStatusTimeout);
  // No copy into this block's shared memory may outlive the block.
  if (lane == 0)
    for (int jj = max(0, j - STAGES); jj < j; ++jj)
      mbar_wait(bar_full + 8 * (jj % STAGES), (jj / STAGES) & 1);
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

// Fixed-order merge of the consumer warps' (m, l, o) for G heads; writes the
// normalised partial row and its log2-sum-exp2. mg holds [W][G*D] outputs,
// then [W][G] maxima, then [W][G] sums.
template <int D>
__device__ __forceinline__ void merge_warps(const Stage1Args& a, const pkvd_work_item& it, int G,
                                            int hq0, const float* mg) {
  const float* mm = mg + kConsumerWarps * G * D;
  const float* ml = mm + kConsumerWarps * G;
  for (int idx = threadIdx.x; idx < G * D; idx += kConsumerWarps * 32) {
    const int h = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mm[w * G + h]);
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float e = exp2f(mm[w * G + h] - M);
        den += e * ml[w * G + h];
        num += e * mg[w * G * D + h * D + d];
      }
    }
    const int64_t row = static_cast<int64_t>(it.partial_row) * a.heads + hq0 + h;
    a.o_part[row * a.dv + d] = (M == -INFINITY) ? 0.f : num / den;
    if (d == 0) a.lse_part[row] = (M == -INFINITY) ? -INFINITY : M + log2f(den);
  }
}

// Prologue shared by both variants: barriers, then the producer branch.
template <int D>
__device__ __forceinline__ bool gqa_prologue(const Stage1Args& a, const pkvd_work_item& it,
                                             uint8_t* smem) {
  constexpr int STAGES = gqa_stages(D);
  const uint32_t bar_full = smem_addr(smem);
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  if ((threadIdx.x >> 5) == kConsumerWarps) {
    gqa_producer<D, STAGES>(a, it, smem + kBarrierBytes, bar_full, bar_empty, threadIdx.x & 31);
    return false;
  }
  return true;
}

// ---------------------------------------------------------------- FMA variant

template <typename T, int D, int G>
__global__ void __launch_bounds__(kStage1Threads, 1)
    gqa_fma(const __grid_constant__ Stage1Args a) {
  constexpr int BLK = kGqaBlockTokens;
  constexpr int STAGES = gqa_stages(D);
  constexpr int PITCH = gqa_row_pitch(D);
  constexpr int SB = gqa_stage_bytes(D);
  constexpr int CH = D / 32;              // columns per lane
  constexpr int N = 4 * G;                // partial sums per four-key pass
  constexpr int SHIFT = 5 - ilog2(N);     // lane >> SHIFT = value index held after the fold
  constexpr int LOGG = ilog2(G);
  constexpr int GP = G < 8 ? 8 : G;       // p-buffer row stride (floats)
  static_assert(N <= 32, "at most 8 heads per KV head on the FMA path");
  static_assert(gqa_merge_bytes(D, G) <= STAGES * SB, "merge area must fit in the stages");

  extern __shared__ __align__(128) uint8_t smem[];
  const pkvd_work_item it = a.items[blockIdx.x];
  pdl_launch_dependents();
  if (!gqa_prologue<D>(a, it, smem)) return;

  const uint32_t bar_full = smem_addr(smem);
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  uint8_t* stages = smem + kBarrierBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* pb = reinterpret_cast<float*>(stages + STAGES * SB) + warp * (BLK * GP + GP);

  const int n = it.tok_end - it.tok_begin;
  const int nblk = (n + BLK - 1) / BLK;
  const int kvh = it.unit;
  const int f = lane >> SHIFT;            // (key in pass, head) this lane ends with
  const int fk = f >> LOGG;
  const int fh = f & (G - 1);
  const bool primary = (lane & ((1 << SHIFT) - 1)) == 0;

  // Query rows of the group, head order permuted by fh so that the partial
  // in slot (kk, h) is the one of value index (kk, h) ^ f.
  float qr[G][CH];
  {
    const uint8_t* qb = static_cast<const uint8_t*>(a.q) +
                        ((static_cast<int64_t>(it.request) * a.heads + kvh * G) * D + lane * CH) * 2;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      load_row<T, CH>(qb + static_cast<int64_t>(h ^ fh) * D * 2, qr[h]);
#pragma unroll
      for (int c = 0; c < CH; ++c) qr[h][c] *= a.scale_log2;
    }
  }

  float acc[G][CH];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int c = 0; c < CH; ++c) acc[h][c] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  bool ok = true;

  for (int j = warp; j < nblk; j += kConsumerWarps) {
    const int s = j % STAGES;
    if (!__all_sync(kFull, mbar_wait(bar_full + 8 * s, (j / STAGES) & 1))) {
      ok = false;
      break;
    }
    const int nv = min(BLK, n - j * BLK);
    const uint8_t* ks = stages + s * SB;
    const uint8_t* vs = ks + BLK * PITCH;

    float sc[4];
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
      float part[N];
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        float kf[CH];
        load_row<T, CH>(ks + (pass * 4 + (kk ^ fk)) * PITCH + lane * CH * 2, kf);
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

#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float al = pb[BLK * GP + h];
#pragma unroll
      for (int c = 0; c < CH; ++c) acc[h][c] *= al;
    }
#pragma unroll
    for (int key = 0; key < BLK; ++key) {
      if (key < nv) {
        float vf[CH];
        load_row<T, CH>(vs + key * PITCH + lane * CH * 2, vf);
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
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
  }

  // Head totals of l over the lanes that held the other keys.
  l_run += __shfl_xor_sync(kFull, l_run, 16);
  l_run += __shfl_xor_sync(kFull, l_run, 8);

  if (consumer_sync_or(!ok)) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusTimeout);
    return;
  }
  // All stages are consumed: reuse them for the cross-warp merge.
  float* mg = reinterpret_cast<float*>(stages);
  float* mo = mg + warp * G * D;
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int c = 0; c < CH; ++c) mo[h * D + lane * CH + c] = acc[h][c];
  if (primary && fk == 0) {
    mg[kConsumerWarps * G * D + warp * G + fh] = m_run;
    mg[kConsumerWarps * G * D + kConsumerWarps * G + warp * G + fh] = l_run;
  }
  consumer_sync();
  merge_warps<D>(a, it, G, kvh * G, mg);
}

// ---------------------------------------------------------------- MMA variant

template <typename T, int D, int NT>
__global__ void __launch_bounds__(kStage1Threads, 1)
    gqa_mma(const __grid_constant__ Stage1Args a) {
  constexpr int BLK = kGqaBlockTokens;
  constexpr int STAGES = gqa_stages(D);
  constexpr int PITCH = gqa_row_pitch(D);
  constexpr int SB = gqa_stage_bytes(D);
  constexpr int KS = D / 16;              // k-steps of the score product = m-tiles of O^T
  constexpr int GMAX = 8 * NT;
  static_assert(gqa_merge_bytes(D, GMAX) <= STAGES * SB, "merge area must fit in the stages");

  extern __shared__ __align__(128) uint8_t smem[];
  const pkvd_work_item it = a.items[blockIdx.x];
  pdl_launch_dependents();
  if (!gqa_prologue<D>(a, it, smem)) return;

  const uint32_t bar_full = smem_addr(smem);
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  uint8_t* stages = smem + kBarrierBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int G = a.heads / a.kv_heads;
  const int n = it.tok_end - it.tok_begin;
  const int nblk = (n + BLK - 1) / BLK;
  const int kvh = it.unit;

  // Q^T as the B operand: lane holds head (nt*8 + g), dims 16ks + 2t (+1, +8, +9).
  uint32_t qb[KS][NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int h = nt * 8 + g;
    const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
        static_cast<const uint8_t*>(a.q) +
        (static_cast<int64_t>(it.request) * a.heads + kvh * G + (h < G ? h : 0)) * D * 2);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qb[ks][nt][0] = h < G ? __ldg(qrow + ks * 8 + t) : 0u;
      qb[ks][nt][1] = h < G ? __ldg(qrow + ks * 8 + 4 + t) : 0u;
    }
  }

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
  bool ok = true;

  for (int j = warp; j < nblk; j += kConsumerWarps) {
    const int s = j % STAGES;
    if (!__all_sync(kFull, mbar_wait(bar_full + 8 * s, (j / STAGES) & 1))) {
      ok = false;
      break;
    }
    const int nv = min(BLK, n - j * BLK);
    uint8_t* ks_ = stages + s * SB;
    uint8_t* vs = ks_ + BLK * PITCH;
    if (nv < BLK) {
      // P is zero past the end, but stale rows could hold non-finite bits.
      constexpr int CHUNKS = D * 2 / 16;
      for (int i = lane; i < (BLK - nv) * CHUNKS; i += 32)
        *reinterpret_cast<uint4*>(vs + (nv + i / CHUNKS) * PITCH + (i % CHUNKS) * 16) =
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
    const uint32_t kaddr = smem_addr(ks_ + (lane & 15) * PITCH + (lane >> 4) * 16);
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      uint32_t af[4];
      ldmatrix_x4(kaddr + k * 32, af[0], af[1], af[2], af[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma_16816<T>(c[nt][k & 1], af, qb[k][nt][0], qb[k][nt][1]);
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
      // C fragment (keys x heads) -> B fragment of P^T (keys as k, heads as n).
      // P goes to the tensor cores as a 16-bit high part plus the 16-bit
      // rounding of its remainder, so P.V keeps ~16 significant bits of P.
      const uint32_t hi0 = pack2<T>(p[0], p[1]), hi1 = pack2<T>(p[2], p[3]);
      const float2 r0 = unpack2<T>(hi0), r1 = unpack2<T>(hi1);
      pf[nt][0][0] = movmatrix_trans(hi0);
      pf[nt][0][1] = movmatrix_trans(hi1);
      pf[nt][1][0] = movmatrix_trans(pack2<T>(p[0] - r0.x, p[1] - r0.y));
      pf[nt][1][1] = movmatrix_trans(pack2<T>(p[2] - r1.x, p[3] - r1.y));
    }

#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        o[mt][nt][0] *= alpha[nt][0];
        o[mt][nt][1] *= alpha[nt][1];
        o[mt][nt][2] *= alpha[nt][0];
        o[mt][nt][3] *= alpha[nt][1];
      }
    // O^T += V^T P^T: A = V^T by transposing ldmatrix of the V rows.
    const uint32_t vaddr =
        smem_addr(vs + (((lane >> 4) & 1) * 8 + (lane & 7)) * PITCH + ((lane >> 3) & 1) * 16);
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      uint32_t vf[4];
      ldmatrix_x4_trans(vaddr + mt * 32, vf[0], vf[1], vf[2], vf[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma_16816<T>(o[mt][nt], vf, pf[nt][0][0], pf[nt][0][1]);
        mma_16816<T>(o[mt][nt], vf, pf[nt][1][0], pf[nt][1][1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
  }

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

  if (consumer_sync_or(!ok)) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusTimeout);
    return;
  }
  float* mg = reinterpret_cast<float*>(stages);
  float* mo = mg + warp * G * D;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h0 = nt * 8 + 2 * t, d0 = mt * 16 + g;
      if (h0 < G) {
        mo[h0 * D + d0] = o[mt][nt][0];
        mo[h0 * D + d0 + 8] = o[mt][nt][2];
      }
      if (h0 + 1 < G) {
        mo[(h0 + 1) * D + d0] = o[mt][nt][1];
        mo[(h0 + 1) * D + d0 + 8] = o[mt][nt][3];
      }
    }
  if (g == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = nt * 8 + 2 * t + e;
        if (h < G) {
          mg[kConsumerWarps * G * D + warp * G + h] = m_run[nt][e];
          mg[kConsumerWarps * G * D + kConsumerWarps * G + warp * G + h] = l_run[nt][e];
        }
      }
  }
  consumer_sync();
  merge_warps<D>(a, it, G, kvh * G, mg);
}

template <typename T, int D, int G>
void fma_entry(KernelEntry* e) {
  e->func = reinterpret_cast<const void*>(&gqa_fma<T, D, G>);
  e->threads = kStage1Threads;
  e->smem = gqa_smem_bytes(D, G);
  e->block_tokens = kGqaBlockTokens;
  e->stages = gqa_stages(D);
}

template <typename T, int D, int NT>
void mma_entry(KernelEntry* e) {
  e->func = reinterpret_cast<const void*>(&gqa_mma<T, D, NT>);
  e->threads = kStage1Threads;
  e->smem = gqa_smem_bytes(D, 8 * NT);
  e->block_tokens = kGqaBlockTokens;
  e->stages = gqa_stages(D);
}

template <typename T, int D>
bool fma_by_group(int group, KernelEntry* e) {
  switch (group) {
    case 1: fma_entry<T, D, 1>(e); return true;
    case 2: fma_entry<T, D, 2>(e); return true;
    case 4: fma_entry<T, D, 4>(e); return true;
    case 8: fma_entry<T, D, 8>(e); return true;
    default: return false;
  }
}

template <typename T>
bool fma_by_dim(int head_dim, int group, KernelEntry* e) {
  if (head_dim == 128) return fma_by_group<T, 128>(group, e);
  if (head_dim == 256) return fma_by_group<T, 256>(group, e);
  return false;
}

template <typename T>
bool mma_by_dim(int head_dim, int group, KernelEntry* e) {
  if (group < 1 || group > 16) return false;
  const bool two = group > 8;
  if (head_dim == 128) { two ? mma_entry<T, 128, 2>(e) : mma_entry<T, 128, 1>(e); return true; }
  if (head_dim == 256) { two ? mma_entry<T, 256, 2>(e) : mma_entry<T, 256, 1>(e); return true; }
  return false;
}

}  // namespace

bool gqa_fma_kernel(int dtype, int head_dim, int group, KernelEntry* e) {
  return dtype == PKVD_FP16 ? fma_by_dim<__half>(head_dim, group, e)
                            : fma_by_dim<__nv_bfloat16>(head_dim, group, e);
}

bool gqa_mma_kernel(int dtype, int head_dim, int group, KernelEntry* e) {
  return dtype == PKVD_FP16 ? mma_by_dim<__half>(head_dim, group, e)
                            : mma_by_dim<__nv_bfloat16>(head_dim, group, e);
}

}  // namespace pkvd
