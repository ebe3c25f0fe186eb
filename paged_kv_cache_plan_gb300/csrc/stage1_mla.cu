// Stage 1 for MLA: one block per work item (request b, block of 16 heads,
// split s). All heads share one 576-wide latent row per token (512 no-rope
// + 64 rope); V is the first 512 elements of the same row. This is the
// "bh16" stage-1 regime of the aiter pull 4758 page (Motivation, Technical
// Details 1): a program walks the KV blocks of one (request, split, head
// block), keeps several blocks in flight, and leaves a partial plus LSE.
//
// Four warps, no producer warp. A block is 16 tokens; warp w issues the bulk
// copies of rows 4w .. 4w+3 of every block (one 1,152-byte copy per row, into
// rows padded to 1,168 bytes), so four warps' copies are in flight at once.
// Five stages: the copies of block j+4 are issued while block j is scored.
// Page ids are read eight blocks ahead into a register window.
//
// Per block, on mma.sync m16n8k16 (M = the 16 heads):
//   S = Q K^T       warp w multiplies over dims 144w .. 144w+143 (nine
//                   k-steps, its Q fragments held in registers for the whole
//                   item) for all 16 keys, and stores the partial tile;
//   one block barrier, then every warp adds the four partials in warp order,
//                   so all warps hold the same S, the same running maxima
//                   and the same P (the block barrier also frees the stage
//                   of the previous block for refilling);
//   O += P V        warp w owns output columns 128w .. 128w+127. P stays in
//                   registers (the accumulator layout of S is the A-operand
//                   layout of P), as a 16-bit high part plus the rounding of
//                   its remainder: two products keep ~16 significant bits.
#include "device.cuh"
#include "kernels.h"

namespace pkvd {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kPageWindow = 8;   // blocks of page ids read ahead

// __syncthreads that also ORs a flag over the block.
__device__ __forceinline__ bool block_sync_or(bool flag) { return __syncthreads_or(flag) != 0; }

// CAUSAL: several query tokens per request (q_len > 1), each row cut at its
// token's position; the one-token kernel has no per-row cut.
template <typename T, bool CAUSAL>
__global__ void __launch_bounds__(kMlaThreads, 2)
    mla_mma(const __grid_constant__ Stage1Args a, const __grid_constant__ KvTensorMaps) {
  constexpr int BLK = kMlaBlockTokens;
  constexpr int STAGES = kMlaStages;
  constexpr int W = kMlaWarps;
  constexpr int HB = kMlaHeads;
  constexpr int PITCH = kMlaRowPitch;
  constexpr int SB = kMlaStageBytes;
  constexpr int ROWB = kMlaDk * 2;
  constexpr int KSW = kMlaDk / 16 / W;   // 9 k-steps of the score product per warp
  constexpr int NCOL = kMlaDv / W;       // 128 output columns per warp
  constexpr int NTO = NCOL / 8;          // 16 n-tiles of O per warp
  constexpr int RPW = BLK / W;           // rows each warp copies per block
  constexpr int PF = kPageWindow;
  static_assert(BLK == 16 && KSW * W * 16 == kMlaDk && RPW * W == BLK, "block shape");
  static_assert(PF >= STAGES, "the page window covers the prologue");
  static_assert(kMlaSmemBytes == kBarrierBytes + STAGES * SB + 2 * W * 2 * 32 * 16, "layout");

  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t bars = smem_addr(smem);   // one full barrier per stage
  uint8_t* stages = smem + kBarrierBytes;
  float4* red = reinterpret_cast<float4*>(stages + STAGES * SB);   // [2][W][2][32]

  const pkvd_work_item it = a.items[blockIdx.x];
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int n = it.tok_end - it.tok_begin;
  const int nblk = (n + BLK - 1) / BLK;
  const int32_t* pt = a.page_table + static_cast<int64_t>(it.request) * a.pt_stride;
  const uint8_t* pool = static_cast<const uint8_t*>(a.k);
  const int64_t pitch_bytes = a.k_pitch * 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) mbar_init(bars + 8 * s, W);
    fence_barrier_init();
  }
  __syncthreads();

  // Page id of this lane's row (lanes < RPW) of block j, 0 past the end: a
  // load issued PF blocks before the row is formed from it (row_at), so its
  // latency never stalls the warp.
  auto page_of = [&](int j) -> int {
    const int tok = it.tok_begin + j * BLK + warp * RPW + lane;
    if (lane >= RPW || j >= nblk || tok >= it.tok_end) return 0;
    return ld_pinned(pt + tok / a.page_size);
  };
  // Pool row of this lane's row of block j from its page id; 0 past the end.
  auto row_at = [&](int j, int page) -> int64_t {
    const int tok = it.tok_begin + j * BLK + warp * RPW + lane;
    if (lane >= RPW || j >= nblk || tok >= it.tok_end) return 0;
    const int pidx = tok / a.page_size;
    if (a.checks && (page < 0 || page >= a.num_pool_pages)) {
      atomicOr(a.status, kStatusBadPage);
      page = 0;
    }
    return static_cast<int64_t>(page) * a.page_size + (tok - pidx * a.page_size);
  };
  // This warp's share of block j's copies. Rows past the item's end get a
  // zero V part instead (P is 0 there, but stale bits may not be finite).
  auto issue = [&](int j, int64_t row) {
    const int s = j % STAGES;
    uint8_t* st = stages + s * SB;
    const uint32_t bar = bars + 8 * s;
    const int nv = min(BLK, n - j * BLK);
    const int mine = max(0, min(RPW, nv - warp * RPW));
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(mine * ROWB));
    __syncwarp();
    if (lane < mine)
      bulk_copy_g2s(smem_addr(st + (warp * RPW + lane) * PITCH), pool + row * pitch_bytes, ROWB,
                    bar);
    if (mine < RPW) {
      constexpr int CH = kMlaDv * 2 / 16;   // 16-byte chunks of a V row
      for (int i = lane; i < (RPW - mine) * CH; i += 32)
        *reinterpret_cast<uint4*>(st + (warp * RPW + mine + i / CH) * PITCH + (i % CH) * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      fence_proxy_async_smem();
    }
  };

  int pages[PF];
#pragma unroll
  for (int i = 0; i < PF; ++i) pages[i] = page_of(i);
#pragma unroll
  for (int i = 0; i < STAGES; ++i) {
    if (i < nblk) issue(i, row_at(i, pages[i]));
    pages[i] = page_of(i + PF);
  }
  int issued = min(nblk, STAGES);

  // Q fragments of this warp's nine k-steps, rows g and g + 8 of the
  // item's 16 (query token, head) rows unit * 16 .. unit * 16 + 15 (row v of
  // a request is query token v / heads, head v % heads).
  const int VH = a.q_len * a.heads;
  uint32_t qf[KSW][4];
  {
    const T* qg = static_cast<const T*>(a.q) +
                  (static_cast<int64_t>(it.request) * VH + it.unit * HB) * kMlaDk;
#pragma unroll
    for (int i = 0; i < KSW; ++i) {
      const int d = (warp * KSW + i) * 16 + 2 * t;
      qf[i][0] = ldg_pair(qg + g * kMlaDk + d);
      qf[i][1] = ldg_pair(qg + (g + 8) * kMlaDk + d);
      qf[i][2] = ldg_pair(qg + g * kMlaDk + d + 8);
      qf[i][3] = ldg_pair(qg + (g + 8) * kMlaDk + d + 8);
    }
  }

  float o[NTO][4];
#pragma unroll
  for (int i = 0; i < NTO; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY};   // rows g, g + 8 (same in every warp)
  // last visible token of rows g, g + 8, relative to the item
  const int lim[2] = {CAUSAL ? it.query_pos + (it.unit * HB + g) / a.heads - it.tok_begin : 0,
                      CAUSAL ? it.query_pos + (it.unit * HB + g + 8) / a.heads - it.tok_begin
                             : 0};
  float l_run[2] = {0.f, 0.f};               // this lane's keys only

  // ldmatrix row addresses: K rows (keys) for the B operand of S, and V rows
  // (keys, transposed on load) for the B operand of O.
  const uint32_t kbase = smem_addr(stages) +
                         ((lane >> 4) * 8 + (lane & 7)) * PITCH + ((lane >> 3) & 1) * 16 +
                         warp * KSW * 32;
  const uint32_t vbase = smem_addr(stages) + (((lane >> 3) & 1) * 8 + (lane & 7)) * PITCH +
                         (warp * NCOL + (lane >> 4) * 8) * 2;
  bool ok = true;
  int j = 0;

  for (int j0 = 0; ok && j0 < nblk; j0 += PF) {
#pragma unroll
    for (int i = 0; i < PF; ++i) {
      if (ok && j0 + i < nblk) {
        j = j0 + i;
        const int s = j % STAGES;
        const bool got = __all_sync(kFull, mbar_wait(bars + 8 * s, (j / STAGES) & 1));

        // Partial S over this warp's dims: two n-tiles (keys 0-7, 8-15), two
        // chains each.
        float c[2][2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int ch = 0; ch < 2; ++ch)
#pragma unroll
            for (int e = 0; e < 4; ++e) c[nt][ch][e] = 0.f;
        if (got) {
          const uint32_t kaddr = kbase + s * SB;
#pragma unroll
          for (int kk = 0; kk < KSW; ++kk) {
            uint32_t b[4];
            ldmatrix_x4(kaddr + kk * 32, b[0], b[1], b[2], b[3]);
            mma_16816<T>(c[0][kk & 1], qf[kk], b[0], b[1]);
            mma_16816<T>(c[1][kk & 1], qf[kk], b[2], b[3]);
          }
        }
        float4* rb = red + (j & 1) * (W * 2 * 32);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          rb[(warp * 2 + nt) * 32 + lane] =
              make_float4(c[nt][0][0] + c[nt][1][0], c[nt][0][1] + c[nt][1][1],
                          c[nt][0][2] + c[nt][1][2], c[nt][0][3] + c[nt][1][3]);
        if (block_sync_or(!got)) {
          ok = false;
        } else {
          // Every warp is past block j - 1: refill its stage with block j + STAGES - 1.
          if (j >= 1) {
            if (j + STAGES - 1 < nblk) {
              issue(j + STAGES - 1, row_at(j + STAGES - 1, pages[(i + STAGES - 1) % PF]));
              issued = j + STAGES;
            }
            pages[(i + STAGES - 1) % PF] = page_of(j + STAGES - 1 + PF);
          }

          // Full scores: the four partials in warp order. Keys at or past
          // kl[r] are past the item's end or not yet visible to row r.
          const int nv = min(BLK, n - j * BLK);
          const int kl[2] = {CAUSAL ? min(nv, lim[0] - j * BLK + 1) : nv,
                             CAUSAL ? min(nv, lim[1] - j * BLK + 1) : nv};
          float sc[2][4];
          float lm[2] = {-INFINITY, -INFINITY};
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            float4 acc = rb[nt * 32 + lane];
#pragma unroll
            for (int w = 1; w < W; ++w) {
              const float4 p = rb[(w * 2 + nt) * 32 + lane];
              acc.x += p.x;
              acc.y += p.y;
              acc.z += p.z;
              acc.w += p.w;
            }
            const float v[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = nt * 8 + 2 * t + (e & 1);
              sc[nt][e] = key < kl[e >> 1] ? v[e] * a.scale_log2 : -INFINITY;
              lm[e >> 1] = fmaxf(lm[e >> 1], sc[nt][e]);
            }
          }
          float alpha[2], m_ref[2];
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            lm[r] = fmaxf(lm[r], __shfl_xor_sync(kFull, lm[r], 1));
            lm[r] = fmaxf(lm[r], __shfl_xor_sync(kFull, lm[r], 2));
            const float m_new = fmaxf(m_run[r], lm[r]);
            // a row with no visible token yet keeps m = -inf, p = 0
            m_ref[r] = CAUSAL && m_new == -INFINITY ? 0.f : m_new;
            alpha[r] = exp2f(m_run[r] - m_ref[r]);
            m_run[r] = m_new;
          }
          // P in the A-operand layout: rows g / g + 8, keys 2t, 2t+1 (n-tile
          // 0) and 8+2t, 9+2t (n-tile 1).
          uint32_t ph[4], pl[4];
          float psum[2] = {0.f, 0.f};
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            float p[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              p[e] = exp2f(sc[nt][e] - m_ref[e >> 1]);
              psum[e >> 1] += p[e];
            }
            const uint32_t h0 = pack2<T>(p[0], p[1]), h1 = pack2<T>(p[2], p[3]);
            const float2 r0 = unpack2<T>(h0), r1 = unpack2<T>(h1);
            ph[2 * nt] = h0;
            ph[2 * nt + 1] = h1;
            pl[2 * nt] = pack2<T>(p[0] - r0.x, p[1] - r0.y);
            pl[2 * nt + 1] = pack2<T>(p[2] - r1.x, p[3] - r1.y);
          }
          l_run[0] = l_run[0] * alpha[0] + psum[0];
          l_run[1] = l_run[1] * alpha[1] + psum[1];
          if (__any_sync(kFull, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int q = 0; q < NTO; ++q) {
              o[q][0] *= alpha[0];
              o[q][1] *= alpha[0];
              o[q][2] *= alpha[1];
              o[q][3] *= alpha[1];
            }
          }
          // O[:, 128w .. 128w+127] += P V over the block's 16 keys.
          const uint32_t ah[4] = {ph[0], ph[1], ph[2], ph[3]};
          const uint32_t al[4] = {pl[0], pl[1], pl[2], pl[3]};
          const uint32_t vaddr = vbase + s * SB;
#pragma unroll
          for (int np = 0; np < NTO / 2; ++np) {
            uint32_t b[4];
            ldmatrix_x4_trans(vaddr + np * 32, b[0], b[1], b[2], b[3]);
            mma_16816<T>(o[2 * np], ah, b[0], b[1]);
            mma_16816<T>(o[2 * np + 1], ah, b[2], b[3]);
            mma_16816<T>(o[2 * np], al, b[0], b[1]);
            mma_16816<T>(o[2 * np + 1], al, b[2], b[3]);
          }
        }
      }
    }
  }

  if (!ok) {
    if (threadIdx.x == 0) {
      atomicOr(a.status, kStatusTimeout);
      // copies still in flight must land before the block exits
      for (int q = j; q < issued; ++q) mbar_wait(bars + 8 * (q % STAGES), (q / STAGES) & 1);
    }
    pdl_wait_prerequisites();   // see the end of the kernel
    return;
  }

  // Row sums over the quad's keys (identical in every warp).
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l_run[r] += __shfl_xor_sync(kFull, l_run[r], 1);
    l_run[r] += __shfl_xor_sync(kFull, l_run[r], 2);
  }
  const int64_t row0 = static_cast<int64_t>(it.partial_row) * VH + it.unit * HB;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int h = g + 8 * r;
    const bool empty = m_run[r] == -INFINITY;
    const float inv = empty ? 0.f : 1.f / l_run[r];
    float* orow = a.o_part + (row0 + h) * a.dv + warp * NCOL + 2 * t;
#pragma unroll
    for (int q = 0; q < NTO; ++q)
      *reinterpret_cast<float2*>(orow + q * 8) =
          make_float2(o[q][2 * r] * inv, o[q][2 * r + 1] * inv);
    if (warp == 0 && t == 0)
      a.lse_part[(it.unit * HB + h) * a.lse_stride + it.partial_row] =
          empty ? -INFINITY : m_run[r] + log2f(l_run[r]);
  }
  // Launched after shared-prefix items (programmatic dependent launch, so
  // that these blocks fill SMs the prefix items leave): the block finishes
  // only once the prefix grid has, so the merge, which waits on this grid,
  // sees the prefix partials too. Without a prerequisite grid this returns
  // at once.
  pdl_wait_prerequisites();
}

}  // namespace

bool mla_mma_kernel(int dtype, bool causal, KernelEntry* e) {
  if (causal)
    e->func = dtype == PKVD_FP16 ? reinterpret_cast<const void*>(&mla_mma<__half, true>)
                                 : reinterpret_cast<const void*>(&mla_mma<__nv_bfloat16, true>);
  else
    e->func = dtype == PKVD_FP16 ? reinterpret_cast<const void*>(&mla_mma<__half, false>)
                                 : reinterpret_cast<const void*>(&mla_mma<__nv_bfloat16, false>);
  e->threads = kMlaThreads;
  e->smem = kMlaSmemBytes;
  e->block_tokens = kMlaBlockTokens;
  e->stages = kMlaStages;
  return true;
}

}  // namespace pkvd
