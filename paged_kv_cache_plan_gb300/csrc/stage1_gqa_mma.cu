// Stage 1 for GQA, tensor-core (mma.sync) consumer (shared parts in
// stage1_gqa.cuh).
//
// Two consumers (the TensorFold pull 1932 page, "What this changes": separate
// kernel symbols per variant rather than a grid-uniform branch); this one:
//   * gqa_mma: mma.sync m16n8k16 with the 16 keys of a block as M and the
//     head group as N (8 per n-tile): S^T = K Q^T, then O^T += V^T P^T with
//     P^T formed in registers by movmatrix, as a 16-bit high part plus a
//     16-bit low remainder (two products), so P keeps ~16 significant bits.
#include "stage1_gqa.cuh"

namespace pkvd {
namespace {

using namespace gqa;

// CAUSAL: several query tokens per request (q_len > 1), each column cut at
// its token's position; the one-token kernel has no per-column cut.
template <typename T, int D, int NT, bool TILES, bool CAUSAL>
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
  const int NQ = a.q_len * G;             // columns: query token j's head kvh*G + i at j*G + i
  const int kvh = it.unit;

  WarpRows<D, TILES> wr(a, it, warp, lane);
  init_stage_barriers<D>(sm.bars);

  // The item's query rows [GMAX][D] in padded rows (zero past NQ): the
  // source of the Q^T B fragments, read with ldmatrix each block. Loaded by
  // the whole block once every warp has its first KV copies in flight (all
  // warps run this exactly once, so the barrier inside is safe), with
  // cp.async so that all of its loads are in flight together.
  auto load_q = [&]() {
    constexpr int CHUNKS = D * 2 / 16;
    for (int i = threadIdx.x; i < GMAX * CHUNKS; i += gqa_threads(D)) {
      const int h = i / CHUNKS, c = i % CHUNKS;
      const int64_t qrow =
          CAUSAL ? (static_cast<int64_t>(it.request) * a.q_len + h / G) * a.heads + kvh * G + h % G
                 : static_cast<int64_t>(it.request) * a.heads + kvh * G + h;
      uint8_t* dst = sm.qtile + h * gqa_row_pitch(D) + c * 16;
      if (h < NQ)
        cp_async16(smem_addr(dst), static_cast<const uint8_t*>(a.q) + qrow * D * 2 + c * 16);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    cp_async_wait_all();
    __syncthreads();
  };
  // Last visible token (relative to the item) of this lane's C-fragment
  // columns nt*8 + 2t + e: query token j = column / G sees tokens up to
  // query_pos + j. With one query token nothing in the item is cut.
  int lim[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e)
      lim[nt][e] = CAUSAL ? it.query_pos + (nt * 8 + 2 * t + e) / G - it.tok_begin : 0;

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
                                          [&](int nv, uint8_t* ks_, int k0) {
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

    uint32_t pf[NT][2][2];   // [n-tile][high, low part][k rows 0-7, 8-15]
    float alpha[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        // keys visible to this column: the block's valid rows, cut (several
        // query tokens) at the column's token position
        const int kl = CAUSAL ? min(nv, lim[nt][e] - k0 + 1) : nv;
        const bool v0 = g < kl, v1 = g + 8 < kl;
        const float s0 = v0 ? (c[nt][0][e] + c[nt][1][e]) * a.scale_log2 : -INFINITY;
        const float s1 = v1 ? (c[nt][0][2 + e] + c[nt][1][2 + e]) * a.scale_log2 : -INFINITY;
        float bm = fmaxf(s0, s1);
        bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
        bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
        bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
        const float m_new = fmaxf(m_run[nt][e], bm);
        // a column with no visible token yet keeps m = -inf, p = 0, alpha = 0
        // (with one query token every block has a visible token)
        const float m_ref = CAUSAL && m_new == -INFINITY ? 0.f : m_new;
        alpha[nt][e] = exp2f(m_run[nt][e] - m_ref);
        m_run[nt][e] = m_new;
        p[e] = exp2f(s0 - m_ref);
        p[2 + e] = exp2f(s1 - m_ref);
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
  float* mo = mg + warp * NQ * RS;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int h0 = nt * 8 + 2 * t, d0 = mt * 16 + g;
      if (h0 < NQ) {
        mo[h0 * RS + d0] = o[mt][nt][0];
        mo[h0 * RS + d0 + 8] = o[mt][nt][2];
      }
      if (h0 + 1 < NQ) {
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
        if (h < NQ) {
          mg[W * NQ * RS + warp * NQ + h] = m_run[nt][e];
          mg[W * NQ * RS + W * NQ + warp * NQ + h] = l_run[nt][e];
        }
      }
  }
  __syncthreads();
  merge_warps<D, CAUSAL>(a, it, G, NQ, mg);
}

template <typename T, int D, int NT, bool TILES, bool CAUSAL>
void mma_entry(KernelEntry* e) {
  e->func = reinterpret_cast<const void*>(&gqa_mma<T, D, NT, TILES, CAUSAL>);
  e->threads = gqa_threads(D);
  e->smem = gqa_smem_bytes(D, 8 * NT, TILES);
  e->block_tokens = kGqaBlockTokens;
  e->stages = gqa_stages(D);
  e->tiles = TILES;
}

template <typename T, int D, bool TILES, bool CAUSAL>
void mma_by_cols(int cols, KernelEntry* e) {
  cols > 8 ? mma_entry<T, D, 2, TILES, CAUSAL>(e) : mma_entry<T, D, 1, TILES, CAUSAL>(e);
}

// cols: the q_len x group (query token, head) columns of an item
template <typename T, bool TILES, bool CAUSAL>
bool mma_by_dim(int head_dim, int cols, KernelEntry* e) {
  if (cols < 1 || cols > 16) return false;
  if (head_dim == 128) {
    mma_by_cols<T, 128, TILES, CAUSAL>(cols, e);
    return true;
  }
  if (head_dim == 256) {
    mma_by_cols<T, 256, TILES, CAUSAL>(cols, e);
    return true;
  }
  return false;
}

template <typename T>
bool mma_by_tiles(int head_dim, int cols, bool tiles, bool causal, KernelEntry* e) {
  if (causal)
    return tiles ? mma_by_dim<T, true, true>(head_dim, cols, e)
                 : mma_by_dim<T, false, true>(head_dim, cols, e);
  return tiles ? mma_by_dim<T, true, false>(head_dim, cols, e)
               : mma_by_dim<T, false, false>(head_dim, cols, e);
}

}  // namespace

bool gqa_mma_kernel(int dtype, int head_dim, int cols, bool tiles, bool causal, KernelEntry* e) {
  return dtype == PKVD_FP16 ? mma_by_tiles<__half>(head_dim, cols, tiles, causal, e)
                            : mma_by_tiles<__nv_bfloat16>(head_dim, cols, tiles, causal, e);
}

}  // namespace pkvd
