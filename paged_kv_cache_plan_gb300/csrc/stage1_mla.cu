// Stage 1 for MLA: one block per work item (request b, block of 16 heads,
// split s). All heads share one 576-wide latent row per token (512 no-rope
// + 64 rope); V is the first 512 elements of the same row. This is the
// "bh16" stage-1 regime of the aiter pull 4758 page (Motivation, Technical
// Details 1): a program walks the KV blocks of one (request, split, head
// block), keeps several blocks in flight, and leaves a partial plus LSE.
//
// Warp roles:
//   * producer warp: page ids read ahead in a register window, one bulk TMA
//     copy per 1,152-byte row into a padded shared-memory row (lane l copies
//     rows l and l + 32 of a 64-token block); two stages in flight.
//   * 4 consumer warps, all on the same block:
//       S  = Q K^T      warp w takes keys 16w .. 16w+15 (mma.sync m16n8k16,
//                       M = the 16 heads, K = 576);
//       one named barrier shares the per-warp head maxima, then P is written
//       to shared memory in the inputs' 16-bit type as a high part plus the
//       rounding of its remainder (two products, ~16 significant bits of P);
//       O += P V        warp w owns output columns 128w .. 128w+127.
//     Every warp sees the same running maxima, so the per-warp row sums can
//     be added at the end in warp order.
#include "device.cuh"
#include "kernels.h"

namespace pkvd {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kPrefetchBlocks = 6;

template <typename T>
__global__ void __launch_bounds__(kStage1Threads, 1)
    mla_mma(const __grid_constant__ Stage1Args a, const __grid_constant__ KvTensorMaps) {
  constexpr int BLK = kMlaBlockTokens;
  constexpr int STAGES = kMlaStages;
  constexpr int HB = kMlaHeads;
  constexpr int PITCH = kMlaRowPitch;
  constexpr int SB = kMlaStageBytes;
  constexpr int ROWB = kMlaDk * 2;
  constexpr int KS = kMlaDk / 16;   // 36 k-steps of the score product
  constexpr int NCOL = kMlaDv / kConsumerWarps;   // 128 output columns per warp
  constexpr int NTO = NCOL / 8;     // 16 n-tiles of O per warp

  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t bar_full = smem_addr(smem);
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  uint8_t* stages = smem + kBarrierBytes;
  uint8_t* qs = stages + STAGES * SB;
  uint8_t* ps = qs + kMlaQBytes;
  float* wmax = reinterpret_cast<float*>(ps + kMlaPBytes);     // [4][16]
  float* wsum = wmax + kConsumerWarps * HB;                      // [4][16]

  const pkvd_work_item it = a.items[blockIdx.x];
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = it.tok_end - it.tok_begin;
  const int nblk = (n + BLK - 1) / BLK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    constexpr int PF = kPrefetchBlocks;
    const int32_t* pt = a.page_table + static_cast<int64_t>(it.request) * a.pt_stride;
    const uint8_t* pool = static_cast<const uint8_t*>(a.k);
    const int64_t pitch_bytes = a.k_pitch * 2;
    auto fetch = [&](int j, int r) -> int {
      const int tok = it.tok_begin + j * BLK + r;
      if (j >= nblk || tok >= it.tok_end) return 0;
      int page = __ldg(pt + tok / a.page_size);
      if (a.checks && (page < 0 || page >= a.num_pool_pages)) {
        atomicOr(a.status, kStatusBadPage);
        page = 0;
      }
      return page;
    };
    // Page ids of blocks j .. j + PF - 1 in a statically indexed register
    // window (unrolled by PF): no register move waits on a pending load.
    int ids[PF][2];
#pragma unroll
    for (int i = 0; i < PF; ++i) {
      ids[i][0] = fetch(i, lane);
      ids[i][1] = fetch(i, lane + 32);
    }
    int j = 0;
    bool ok = true;
    while (ok && j < nblk) {
#pragma unroll
      for (int i = 0; i < PF; ++i) {
        if (j < nblk && ok) {
          const int p0 = ids[i][0], p1 = ids[i][1];
          ids[i][0] = fetch(j + PF, lane);
          ids[i][1] = fetch(j + PF, lane + 32);
          const int s = j % STAGES;
          if (j >= STAGES) {
            bool freed = true;
            if (lane == 0) freed = mbar_wait(bar_empty + 8 * s, ((j / STAGES) & 1) ^ 1);
            ok = __shfl_sync(kFull, freed, 0);
          }
          if (ok) {
            const int nv = min(BLK, n - j * BLK);
            if (lane == 0)
              mbar_arrive_expect_tx(bar_full + 8 * s, static_cast<uint32_t>(nv * ROWB));
            __syncwarp();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int r = lane + 32 * h;
              if (r < nv) {
                const int tok = it.tok_begin + j * BLK + r;
                const int64_t row = (static_cast<int64_t>(h ? p1 : p0) * a.kv_heads) *
                                        a.page_size + tok % a.page_size;
                bulk_copy_g2s(smem_addr(stages + s * SB + r * PITCH), pool + row * pitch_bytes,
                              ROWB, bar_full + 8 * s);
              }
            }
            ++j;
          }
        }
      }
    }
    if (!ok && lane == 0) atomicOr(a.status, kStatusTimeout);
    if (lane == 0)
      for (int jj = max(0, j - STAGES); jj < j; ++jj)
        mbar_wait(bar_full + 8 * (jj % STAGES), (jj / STAGES) & 1);
    return;
  }

  // ------------------------------------------------------------ consumers
  const int g = lane >> 2, t = lane & 3;
  const int h0 = it.unit * HB;   // first query head of this block

  // Q tile [16 heads][576] into padded rows.
  {
    const uint8_t* qg = static_cast<const uint8_t*>(a.q) +
                        (static_cast<int64_t>(it.request) * a.heads + h0) * kMlaDk * 2;
    constexpr int CHUNKS = kMlaDk * 2 / 16;   // 72 per row
    for (int i = threadIdx.x; i < HB * CHUNKS; i += kConsumerWarps * 32) {
      const int r = i / CHUNKS, c = i % CHUNKS;
      *reinterpret_cast<uint4*>(qs + r * PITCH + c * 16) =
          __ldg(reinterpret_cast<const uint4*>(qg + static_cast<int64_t>(r) * kMlaDk * 2) + c);
    }
  }
  consumer_sync();

  float o[NTO][4];
#pragma unroll
  for (int i = 0; i < NTO; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};   // heads g, g + 8 (same in every warp)
  float l_run[2] = {0.f, 0.f};               // this lane's keys only

  const uint32_t qaddr = smem_addr(qs + (lane & 15) * PITCH + (lane >> 4) * 16);
  const uint32_t paddr = smem_addr(ps + (lane & 15) * kMlaPPitch + (lane >> 4) * 16);
  bool abort = false;

  for (int j = 0; j < nblk; ++j) {
    const int s = j % STAGES;
    const bool got = __all_sync(kFull, mbar_wait(bar_full + 8 * s, (j / STAGES) & 1));
    const int nv = min(BLK, n - j * BLK);
    uint8_t* kv = stages + s * SB;
    if (got && nv < BLK) {
      // Rows past the end: zero their V part (P is 0 there, stale bits may not be finite).
      constexpr int CHUNKS = kMlaDv * 2 / 16;   // 64 per row
      for (int i = threadIdx.x; i < (BLK - nv) * CHUNKS; i += kConsumerWarps * 32)
        *reinterpret_cast<uint4*>(kv + (nv + i / CHUNKS) * PITCH + (i % CHUNKS) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
    }

    // S = Q K^T for keys 16w .. 16w + 15: two n-tiles, two chains each.
    float c[2][2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int ch = 0; ch < 2; ++ch)
#pragma unroll
        for (int e = 0; e < 4; ++e) c[nt][ch][e] = 0.f;
    if (got) {
      const uint32_t kaddr = smem_addr(kv + (warp * 16 + (lane >> 4) * 8 + (lane & 7)) * PITCH +
                                       ((lane >> 3) & 1) * 16);
#pragma unroll 6
      for (int k = 0; k < KS; ++k) {
        uint32_t af[4], bf[4];
        ldmatrix_x4(qaddr + k * 32, af[0], af[1], af[2], af[3]);
        ldmatrix_x4(kaddr + k * 32, bf[0], bf[1], bf[2], bf[3]);
        mma_16816<T>(c[0][k & 1], af, bf[0], bf[1]);
        mma_16816<T>(c[1][k & 1], af, bf[2], bf[3]);
      }
    }
    // lane holds heads g (e = 0, 1) and g + 8 (e = 2, 3) for keys
    // 16w + 8nt + 2t + (e & 1)
    float sc[2][4];
    float lm[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = warp * 16 + nt * 8 + 2 * t + (e & 1);
        const float v = (c[nt][0][e] + c[nt][1][e]) * a.scale_log2;
        sc[nt][e] = key < nv ? v : -INFINITY;
        lm[e >> 1] = fmaxf(lm[e >> 1], sc[nt][e]);
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      lm[r] = fmaxf(lm[r], __shfl_xor_sync(kFull, lm[r], 1));
      lm[r] = fmaxf(lm[r], __shfl_xor_sync(kFull, lm[r], 2));
    }
    if (t == 0) {
      wmax[warp * HB + g] = lm[0];
      wmax[warp * HB + g + 8] = lm[1];
    }
    if (consumer_sync_or(!got)) {
      abort = true;
      break;
    }
    float alpha[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int h = g + 8 * r;
      float bm = wmax[h];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) bm = fmaxf(bm, wmax[w * HB + h]);
      const float m_new = fmaxf(m_run[r], bm);
      alpha[r] = exp2f(m_run[r] - m_new);
      m_run[r] = m_new;
    }
    float psum[2] = {0.f, 0.f};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      float p[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        p[e] = exp2f(sc[nt][e] - m_run[e >> 1]);
        psum[e >> 1] += p[e];
      }
      // P as a 16-bit high part (rows 0-15) plus the 16-bit rounding of the
      // remainder (rows 16-31): two products keep ~16 significant bits of P.
      const int col = warp * 16 + nt * 8 + 2 * t;
      const uint32_t hi0 = pack2<T>(p[0], p[1]), hi1 = pack2<T>(p[2], p[3]);
      const float2 r0 = unpack2<T>(hi0), r1 = unpack2<T>(hi1);
      *reinterpret_cast<uint32_t*>(ps + g * kMlaPPitch + col * 2) = hi0;
      *reinterpret_cast<uint32_t*>(ps + (g + 8) * kMlaPPitch + col * 2) = hi1;
      *reinterpret_cast<uint32_t*>(ps + (g + HB) * kMlaPPitch + col * 2) =
          pack2<T>(p[0] - r0.x, p[1] - r0.y);
      *reinterpret_cast<uint32_t*>(ps + (g + 8 + HB) * kMlaPPitch + col * 2) =
          pack2<T>(p[2] - r1.x, p[3] - r1.y);
    }
    l_run[0] = l_run[0] * alpha[0] + psum[0];
    l_run[1] = l_run[1] * alpha[1] + psum[1];
    consumer_sync();

    // O[:, 128w .. 128w+127] = O * alpha + P V
#pragma unroll
    for (int i = 0; i < NTO; ++i) {
      o[i][0] *= alpha[0];
      o[i][1] *= alpha[0];
      o[i][2] *= alpha[1];
      o[i][3] *= alpha[1];
    }
    const uint32_t vaddr = smem_addr(kv + (((lane >> 3) & 1) * 8 + (lane & 7)) * PITCH +
                                     (warp * NCOL + (lane >> 4) * 8) * 2);
#pragma unroll
    for (int kk = 0; kk < BLK / 16; ++kk) {
      uint32_t ah[4], al[4];
      ldmatrix_x4(paddr + kk * 32, ah[0], ah[1], ah[2], ah[3]);
      ldmatrix_x4(paddr + HB * kMlaPPitch + kk * 32, al[0], al[1], al[2], al[3]);
#pragma unroll
      for (int np = 0; np < NTO / 2; ++np) {
        uint32_t bf[4];
        ldmatrix_x4_trans(vaddr + kk * 16 * PITCH + np * 32, bf[0], bf[1], bf[2], bf[3]);
        mma_16816<T>(o[2 * np], ah, bf[0], bf[1]);
        mma_16816<T>(o[2 * np + 1], ah, bf[2], bf[3]);
        mma_16816<T>(o[2 * np], al, bf[0], bf[1]);
        mma_16816<T>(o[2 * np + 1], al, bf[2], bf[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
  }

  if (abort) {
    if (threadIdx.x == 0) atomicOr(a.status, kStatusTimeout);
    return;
  }

  // Row sums: this warp's keys, then all warps in order.
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] += __shfl_xor_sync(kFull, l_run[r], 1);
    l_run[r] += __shfl_xor_sync(kFull, l_run[r], 2);
  }
  if (t == 0) {
    wsum[warp * HB + g] = l_run[0];
    wsum[warp * HB + g + 8] = l_run[1];
  }
  consumer_sync();
  float lt[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int h = g + 8 * r;
    float l = wsum[h];
#pragma unroll
    for (int w = 1; w < kConsumerWarps; ++w) l += wsum[w * HB + h];
    lt[r] = l;
  }
  const int64_t row0 = static_cast<int64_t>(it.partial_row) * a.heads + h0;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int h = g + 8 * r;
    const bool empty = m_run[r] == -INFINITY;
    const float inv = empty ? 0.f : 1.f / lt[r];
    float* orow = a.o_part + (row0 + h) * a.dv + warp * NCOL + 2 * t;
#pragma unroll
    for (int i = 0; i < NTO; ++i)
      *reinterpret_cast<float2*>(orow + i * 8) =
          make_float2(o[i][2 * r] * inv, o[i][2 * r + 1] * inv);
    if (warp == 0 && t == 0)
      a.lse_part[row0 + h] = empty ? -INFINITY : m_run[r] + log2f(lt[r]);
  }
}

}  // namespace

bool mla_mma_kernel(int dtype, KernelEntry* e) {
  e->func = dtype == PKVD_FP16 ? reinterpret_cast<const void*>(&mla_mma<__half>)
                               : reinterpret_cast<const void*>(&mla_mma<__nv_bfloat16>);
  e->threads = kStage1Threads;
  e->smem = kMlaSmemBytes;
  e->block_tokens = kMlaBlockTokens;
  e->stages = kMlaStages;
  return true;
}

}  // namespace pkvd
