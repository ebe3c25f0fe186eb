// Stage 2: merge the split partials of every (request, query token, head)
// row (one query token: every (request, head)); `heads` below counts these
// rows per request.
//
// For request b with S splits (partial rows r0 .. r0 + S - 1), head h:
//     M = max_s lse_s,  w_s = 2^(lse_s - M)          (log2 domain)
//     out = sum_s w_s o_s / sum_s w_s,  lse = ln 2 * (M + log2 sum_s w_s)
// Splits of an empty range carry lse = -inf and weight 0; no split at all
// (an empty request) gives out = 0 and lse = -inf.
//
// Grid: (B * rows, tiles). With tiles > 1 each block owns a disjoint slice of
// the Dv output columns and re-derives M and sum_s w_s on its own, so the
// slices never communicate -- the head-dim-tiled stage-2 reduce of the
// aiter pull 4758 page (Technical Details 3). The merge waits on stage 1
// with griddepcontrol.wait, so it can be launched early (programmatic
// dependent launch).
//
// Bit-identical results for every tiling: every warp computes M and the
// weight sum itself, from the split lse values in the same lane-strided
// order with a xor butterfly (so all lanes and warps hold the same bits),
// and each float4 column is summed in a layout fixed by the split index
// alone (below), whichever block or thread owns the column.
#include "device.cuh"
#include "kernels.h"

namespace pkvd {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kSplitGroups = 32;    // splits s = g, g + 32, g + 64, ... per group
constexpr int kColThreads = 8;      // float4 columns per pass
constexpr int kWarps = kMergeThreads / 32;
static_assert(kMergeThreads == kSplitGroups * kColThreads, "merge block shape");
static_assert(stage2_smem_bytes(4) == kWarps * 16, "one float4 per warp and column");

__device__ __forceinline__ void fma4(float4& acc, float w, const float4& x) {
  acc.x = fmaf(w, x.x, acc.x);
  acc.y = fmaf(w, x.y, acc.y);
  acc.z = fmaf(w, x.z, acc.z);
  acc.w = fmaf(w, x.w, acc.w);
}

__device__ __forceinline__ void add_xor4(float4& v, int m) {
  v.x += __shfl_xor_sync(kFull, v.x, m);
  v.y += __shfl_xor_sync(kFull, v.y, m);
  v.z += __shfl_xor_sync(kFull, v.z, m);
  v.w += __shfl_xor_sync(kFull, v.w, m);
}

// Block layout: thread (g, c) = (tid / 8, tid % 8) sums, for each of its
// float4 columns c, c + 8, ..., the weighted partials of splits s = g mod 32
// in increasing s. The four groups of a warp are added by a xor butterfly
// over lane bits 3-4, the eight warps' sums in warp order. Each lane holds
// kLseRegs lse values (lane-strided) and the weights of its first kLseRegs
// own splits in registers; further splits are read as they come. A thread
// takes kU of its columns (c, c + 8, ...) at a time with kPre of each
// column's splits in flight, kU x kPre loads at once; those of its first
// columns are issued together with the lse values, before the weights are
// known. The grouping changes no addition: every column sums its splits in
// the same order whatever kU, kPre and the tiling. Variants: <8, 8, 1> for
// small grids of narrow slices (a tiled Dv: one column per thread), <4, 8, 4>
// for small grids of wide rows, <2, 2, 4> and <2, 2, 1> for large grids,
// where registers would cost occupancy.
template <int kPre, int kLseRegs, int kU>
__global__ void __launch_bounds__(kMergeThreads, kPre > 2 ? 2 : 3)
    merge_splits(const __grid_constant__ Stage2Args a) {
  static_assert(kLseRegs % kPre == 0, "prefetch depth divides the register window");
  extern __shared__ float4 wsum4[];   // [kWarps][C4] warp sums

  const int bh = blockIdx.x;
  const int b = bh / a.heads;
  const int h = bh - b * a.heads;
  const int dt = a.dv / a.tiles;
  const int C4 = dt / 4;
  const int d0 = blockIdx.y * dt;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int grp = threadIdx.x / kColThreads;
  const int ct = threadIdx.x % kColThreads;

  // The split table is written at plan time, not by stage 1: read it before
  // the wait, while stage 1 finishes.
  const int r0 = a.split_base[b];
  const int S = a.split_base[b + 1] - r0;

  pdl_wait_prerequisites();

  const int64_t stride = static_cast<int64_t>(a.heads) * a.dv;
  const float* base = a.o_part + (static_cast<int64_t>(r0) * a.heads + h) * a.dv + d0;
  const float* lp = a.lse_part + h * a.lse_stride + r0;   // this head's splits
  auto part = [&](int s, int c) {   // partial of split s, float4 column c (0 past the ends)
    return c < C4 && s < S ? __ldg(reinterpret_cast<const float4*>(base + s * stride) + c)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
  };

  // One round trip: the first kPre partials of this thread's first kU
  // columns (x holds the loads in flight), and the lse values (lane-strided,
  // for M and the weight sum; and those of this thread's own splits grp + 32 i).
  float4 x[kU][kPre];
#pragma unroll
  for (int u = 0; u < kU; ++u)
#pragma unroll
    for (int j = 0; j < kPre; ++j) x[u][j] = part(grp + j * kSplitGroups, u * kColThreads + ct);
  float lv[kLseRegs], lo[kLseRegs];
#pragma unroll
  for (int i = 0; i < kLseRegs; ++i) {
    const int s = lane + 32 * i, so = grp + kSplitGroups * i;
    lv[i] = s < S ? __ldg(lp + s) : -INFINITY;
    lo[i] = so < S ? __ldg(lp + so) : -INFINITY;
  }

  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < kLseRegs; ++i) m = fmaxf(m, lv[i]);
  for (int s = lane + 32 * kLseRegs; s < S; s += 32)
    m = fmaxf(m, __ldg(lp + s));
#pragma unroll
  for (int x = 16; x >= 1; x >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, x));
  const bool empty = (m == -INFINITY);
  float ws = 0.f;
  if (!empty) {
#pragma unroll
    for (int i = 0; i < kLseRegs; ++i) ws += exp2f(lv[i] - m);
    for (int s = lane + 32 * kLseRegs; s < S; s += 32)
      ws += exp2f(__ldg(lp + s) - m);
  }
#pragma unroll
  for (int x = 16; x >= 1; x >>= 1) ws += __shfl_xor_sync(kFull, ws, x);
  const float inv = empty ? 0.f : 1.f / ws;
  auto weight = [&](float l) { return empty ? 0.f : exp2f(l - m); };
  float wo[kLseRegs];
#pragma unroll
  for (int i = 0; i < kLseRegs; ++i) wo[i] = weight(lo[i]);

  for (int c0 = 0; c0 < C4; c0 += kColThreads * kU) {
    float4 acc[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    // own splits below 32 kLseRegs (the terms past S are zero, so stopping
    // there changes no bits)
#pragma unroll
    for (int i0 = 0; i0 < kLseRegs; i0 += kPre) {
      if (grp + kSplitGroups * i0 >= S) break;
      if (i0 > 0 || c0 > 0) {   // the first chunk was loaded before the weights
#pragma unroll
        for (int u = 0; u < kU; ++u)
#pragma unroll
          for (int j = 0; j < kPre; ++j)
            x[u][j] = part(grp + kSplitGroups * (i0 + j), c0 + u * kColThreads + ct);
      }
#pragma unroll
      for (int u = 0; u < kU; ++u)
#pragma unroll
        for (int j = 0; j < kPre; ++j) fma4(acc[u], wo[i0 + j], x[u][j]);
    }
    for (int s = grp + kSplitGroups * kLseRegs; s < S; s += kSplitGroups) {
      const float w = weight(__ldg(lp + s));
#pragma unroll
      for (int u = 0; u < kU; ++u) fma4(acc[u], w, part(s, c0 + u * kColThreads + ct));
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int c = c0 + u * kColThreads + ct;
      add_xor4(acc[u], 8);
      add_xor4(acc[u], 16);
      if (lane < kColThreads && c < C4) wsum4[warp * C4 + c] = acc[u];
    }
  }
  __syncthreads();
  float* out = a.out + static_cast<int64_t>(bh) * a.dv + d0;
  for (int c = threadIdx.x; c < C4; c += kMergeThreads) {
    float4 t = wsum4[c];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) {
      const float4 x = wsum4[w * C4 + c];
      t.x += x.x;
      t.y += x.y;
      t.z += x.z;
      t.w += x.w;
    }
    reinterpret_cast<float4*>(out)[c] = make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
  }
  if (blockIdx.y == 0 && threadIdx.x == 0)
    a.lse[bh] = empty ? -INFINITY : (m + log2f(ws)) * 0.69314718055994530942f;
}

// Few splits (S <= kMergeColMaxSplits for every request): one thread per
// float4 column, all S partials in flight at once. The column sum is formed
// in exactly the order merge_splits uses for such S -- product w_s o_s per
// split (split s alone in its residue group), xor butterfly over groups
// (0+1)+(2+3) and (4+5)+(6+7) within a warp, then warp 0's sum plus warp
// 1's -- and M and the weight sum by the same warp code, so both kernels
// give identical bits.
__global__ void __launch_bounds__(128) merge_cols(const __grid_constant__ Stage2Args a) {
  constexpr int NS = kMergeColMaxSplits;
  static_assert(NS == 8, "the fixed summation tree below covers eight splits");
  const int bh = blockIdx.x;
  const int b = bh / a.heads;
  const int h = bh - b * a.heads;
  const int dt = a.dv / a.tiles;
  const int C4 = dt / 4;
  const int d0 = blockIdx.y * dt;
  const int lane = threadIdx.x & 31;

  // The split table is written at plan time, not by stage 1: read it before
  // the wait, while stage 1 finishes.
  const int r0 = a.split_base[b];
  const int S = a.split_base[b + 1] - r0;

  pdl_wait_prerequisites();

  const int64_t stride = static_cast<int64_t>(a.heads) * a.dv;
  const float* base = a.o_part + (static_cast<int64_t>(r0) * a.heads + h) * a.dv + d0;
  const float* lp = a.lse_part + h * a.lse_stride + r0;   // this head's splits

  float ls[NS];
#pragma unroll
  for (int s = 0; s < NS; ++s) ls[s] = s < S ? __ldg(lp + s) : -INFINITY;
  // M and the weight sum as merge_splits' warps form them (lane s holds split s)
  float lv = -INFINITY;
#pragma unroll
  for (int s = 0; s < NS; ++s)
    if (lane == s) lv = ls[s];
  float m = lv;
#pragma unroll
  for (int x = 16; x >= 1; x >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, x));
  const bool empty = (m == -INFINITY);
  float ws = empty ? 0.f : exp2f(lv - m);
#pragma unroll
  for (int x = 16; x >= 1; x >>= 1) ws += __shfl_xor_sync(kFull, ws, x);
  const float inv = empty ? 0.f : 1.f / ws;
  float w[NS];
#pragma unroll
  for (int s = 0; s < NS; ++s) w[s] = empty ? 0.f : exp2f(ls[s] - m);

  float* out = a.out + static_cast<int64_t>(bh) * a.dv + d0;
  for (int c = threadIdx.x; c < C4; c += blockDim.x) {
    float4 t[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s)
      t[s] = s < S ? __ldg(reinterpret_cast<const float4*>(base + s * stride) + c)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      float4 p = make_float4(0.f, 0.f, 0.f, 0.f);
      fma4(p, w[s], t[s]);
      t[s] = p;
    }
    auto add = [](const float4& x, const float4& y) {
      return make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w);
    };
    const float4 w0 = add(add(t[0], t[1]), add(t[2], t[3]));
    const float4 w1 = add(add(t[4], t[5]), add(t[6], t[7]));
    const float4 r = add(w0, w1);
    reinterpret_cast<float4*>(out)[c] = make_float4(r.x * inv, r.y * inv, r.z * inv, r.w * inv);
  }
  if (blockIdx.y == 0 && threadIdx.x == 0)
    a.lse[bh] = empty ? -INFINITY : (m + log2f(ws)) * 0.69314718055994530942f;
}

// Merge of context-parallel ranks: each rank's decode over its own token
// range of every request leaves a normalised output row and its natural-log
// lse; the rows of n ranks are combined by the same log-sum-exp merge (aiter
// pull 4758, Technical Details 3), one block per (request, query token, head)
// row and one thread per float4 column, the ranks summed in rank order:
//     M = max_r lse_r,  w_r = e^(lse_r - M),
//     out = sum_r w_r o_r / sum_r w_r,  lse = M + ln sum_r w_r.
// A rank whose range held no token of the request has lse -inf, weight 0.
__global__ void __launch_bounds__(128) merge_ranks(const float* __restrict__ o,
                                                   const float* __restrict__ lse_in, int n,
                                                   int64_t rows, int dv, float* __restrict__ out,
                                                   float* __restrict__ lse) {
  const int64_t row = blockIdx.x;
  const int c = threadIdx.x;   // float4 column
  const int cols = dv / 4;
  float m = -INFINITY;
  for (int r = 0; r < n; ++r) m = fmaxf(m, __ldg(lse_in + r * rows + row));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float ws = 0.f;
  if (m != -INFINITY) {
    for (int r = 0; r < n; ++r) {
      const float l = __ldg(lse_in + r * rows + row);
      if (l == -INFINITY) continue;
      const float w = expf(l - m);
      ws += w;
      if (c < cols) fma4(acc, w, __ldg(reinterpret_cast<const float4*>(o + (r * rows + row) * dv) + c));
    }
  }
  const float inv = m == -INFINITY ? 0.f : 1.f / ws;
  if (c < cols)
    reinterpret_cast<float4*>(out + row * dv)[c] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (c == 0) lse[row] = m == -INFINITY ? -INFINITY : m + logf(ws);
}

}  // namespace

int launch_merge_ranks(int n, int64_t rows, int dv, const float* o, const float* lse_in,
                       float* out, float* lse, cudaStream_t stream) {
  if (rows == 0) return PKVD_OK;
  merge_ranks<<<dim3(static_cast<unsigned>(rows)), dim3(128), 0, stream>>>(o, lse_in, n, rows, dv,
                                                                        out, lse);
  return cudaGetLastError() == cudaSuccess ? PKVD_OK : PKVD_ECUDA;
}

bool stage2_kernel(const pkvd_plan_info& info, int batch, int heads, int dv, KernelEntry* e) {
  const int tiles = info.stage2_tiles > 0 ? info.stage2_tiles : 1;
  if (info.max_splits <= kMergeColMaxSplits) {
    e->func = reinterpret_cast<const void*>(&merge_cols);
    e->threads = merge_col_threads(dv / tiles);
    e->smem = 0;
  } else {
    const bool deep = static_cast<int64_t>(batch) * heads * tiles <= 2LL * info.num_sms;
    const bool wide = dv / tiles / 4 > kColThreads;   // several columns per thread
    e->func = deep ? (wide ? reinterpret_cast<const void*>(&merge_splits<4, 8, 4>)
                           : reinterpret_cast<const void*>(&merge_splits<8, 8, 1>))
                   : (wide ? reinterpret_cast<const void*>(&merge_splits<2, 2, 4>)
                           : reinterpret_cast<const void*>(&merge_splits<2, 2, 1>));
    e->threads = kMergeThreads;
    e->smem = stage2_smem_bytes(dv / tiles);
  }
  return e->threads == info.stage2_threads;
}

}  // namespace pkvd
