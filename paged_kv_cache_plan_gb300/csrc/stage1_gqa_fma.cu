// Stage 1 for GQA, fp32 FMA consumer (shared parts in stage1_gqa.cuh).
//
// Two consumers (the TensorFold pull 1932 page, "What this changes": separate
// kernel symbols per variant rather than a grid-uniform branch):
//   * gqa_fma: fp32 FMA. A warp scores four keys per pass; lane l holds
//     D/32 columns of each row and of every head's query, and the 4 x G
//     partial dot products are folded across the warp with xor shuffles
//     from 16 down to 1 in a fixed order (the same page: four keys a warp,
//     xor-fold wave sums). The fold is a transposing butterfly, so each
//     lane ends with one (key, head) score and no broadcast is needed.
#include "stage1_gqa.cuh"

namespace pkvd {
namespace {

using namespace gqa;

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
                                          [&](int nv, const uint8_t* ks, int) {
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
  merge_warps<D, false>(a, it, G, G, mg);   // one query token (the planner's rule)
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

}  // namespace

bool gqa_fma_kernel(int dtype, int head_dim, int group, bool tiles, KernelEntry* e) {
  if (dtype == PKVD_FP16)
    return tiles ? fma_by_dim<__half, true>(head_dim, group, e)
                 : fma_by_dim<__half, false>(head_dim, group, e);
  return tiles ? fma_by_dim<__nv_bfloat16, true>(head_dim, group, e)
               : fma_by_dim<__nv_bfloat16, false>(head_dim, group, e);
}

}  // namespace pkvd
