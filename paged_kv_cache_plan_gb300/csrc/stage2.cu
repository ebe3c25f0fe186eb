// Stage 2: merge the split partials of every (request, head).
//
// For request b with S splits (partial rows r0 .. r0 + S - 1), head h:
//     M = max_s lse_s,  w_s = 2^(lse_s - M)          (log2 domain)
//     out = sum_s w_s o_s / sum_s w_s,  lse = ln 2 * (M + log2 sum_s w_s)
// Splits of an empty range carry lse = -inf and weight 0; no split at all
// (an empty request) gives out = 0 and lse = -inf.
//
// Grid: (B * Hq, tiles). With tiles > 1 each block owns a disjoint slice of
// the Dv output columns and re-derives M and sum_s w_s on its own, so the
// slices never communicate -- the head-dim-tiled stage-2 reduce of the
// aiter pull 4758 page (Technical Details 3). M and the weight sum are
// always computed by warp 0 in the same lane-strided order, and the weighted
// sums run over a fixed split-residue layout, so every tiling gives
// identical bits. The merge waits on stage 1 with griddepcontrol.wait,
// so it can be launched early (programmatic dependent launch).
#include "device.cuh"
#include "kernels.h"

namespace pkvd {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kSplitGroups = 16;    // splits s = g, g + 16, g + 32, ... per group
constexpr int kColThreads = 16;     // float4 columns per pass
static_assert(kMergeThreads == kSplitGroups * kColThreads, "merge block shape");

// Block layout: thread (g, c) = (tid / 16, tid % 16) sums, for each of its
// float4 columns c, c + 16, ..., the weighted partials of splits s = g mod 16
// in increasing s; the 16 group sums are then added in group order. The
// order of every addition depends only on s and the column, never on the
// tiling, so all tilings give identical bits.
// kPre: partials per thread loaded before the weights are known. Deep (8)
// when the merge grid is small and latency-bound; shallow (2) when it is
// large, where the extra registers would cost occupancy.
template <int kPre>
__global__ void __launch_bounds__(kMergeThreads) merge_splits(const __grid_constant__ Stage2Args a) {
  extern __shared__ float4 dyn[];   // [16][C4] group sums, then [S] weights
  __shared__ float stats[2];        // M, sum of weights

  const int bh = blockIdx.x;
  const int b = bh / a.heads;
  const int h = bh - b * a.heads;
  const int dt = a.dv / a.tiles;
  const int C4 = dt / 4;
  const int d0 = blockIdx.y * dt;
  float4* gsum = dyn;
  float* w_s = reinterpret_cast<float*>(dyn + kSplitGroups * C4);

  pdl_wait_prerequisites();

  const int r0 = a.split_base[b];
  const int S = a.split_base[b + 1] - r0;
  const int grp = threadIdx.x / kColThreads;
  const int ct = threadIdx.x % kColThreads;
  const int64_t stride = static_cast<int64_t>(a.heads) * a.dv;
  const float* base = a.o_part + (static_cast<int64_t>(r0) * a.heads + h) * a.dv + d0;

  // The first kPre partials of this thread's first column are loaded right
  // away, in flight together with the split log-sum-exps: the weights need
  // the lse values, the loads do not.
  float4 pre[kPre];
#pragma unroll
  for (int u = 0; u < kPre; ++u) {
    const int s = grp + u * kSplitGroups;
    pre[u] = ct < C4 && s < S ? __ldg(reinterpret_cast<const float4*>(base + s * stride) + ct)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int s = threadIdx.x; s < S; s += kMergeThreads)
    w_s[s] = a.lse_part[static_cast<int64_t>(r0 + s) * a.heads + h];
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float m = -INFINITY;
    for (int s = lane; s < S; s += 32) m = fmaxf(m, w_s[s]);
#pragma unroll
    for (int x = 16; x >= 1; x >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, x));
    float ws = 0.f;
    for (int s = lane; s < S; s += 32) {
      const float w = (m == -INFINITY) ? 0.f : exp2f(w_s[s] - m);
      w_s[s] = w;
      ws += w;
    }
#pragma unroll
    for (int x = 16; x >= 1; x >>= 1) ws += __shfl_xor_sync(kFull, ws, x);
    if (lane == 0) {
      stats[0] = m;
      stats[1] = ws;
    }
  }
  __syncthreads();
  const float M = stats[0];
  const float wsum = stats[1];
  const bool empty = (M == -INFINITY);
  const float inv = empty ? 0.f : 1.f / wsum;

  auto fma4 = [](float4& acc, float w, const float4& x) {
    acc.x = fmaf(w, x.x, acc.x);
    acc.y = fmaf(w, x.y, acc.y);
    acc.z = fmaf(w, x.z, acc.z);
    acc.w = fmaf(w, x.w, acc.w);
  };
  for (int c = ct; c < C4; c += kColThreads) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = grp;
    if (c == ct) {
#pragma unroll
      for (int u = 0; u < kPre; ++u, s += kSplitGroups)
        if (s < S) fma4(acc, w_s[s], pre[u]);
    }
    for (; s + 3 * kSplitGroups < S; s += 4 * kSplitGroups) {
      float4 x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        x[u] = __ldg(reinterpret_cast<const float4*>(base + (s + u * kSplitGroups) * stride) + c);
#pragma unroll
      for (int u = 0; u < 4; ++u) fma4(acc, w_s[s + u * kSplitGroups], x[u]);
    }
    for (; s < S; s += kSplitGroups)
      fma4(acc, w_s[s], __ldg(reinterpret_cast<const float4*>(base + s * stride) + c));
    gsum[grp * C4 + c] = acc;
  }
  __syncthreads();
  float* out = a.out + static_cast<int64_t>(bh) * a.dv + d0;
  for (int c = threadIdx.x; c < C4; c += kMergeThreads) {
    float4 t = gsum[c];
#pragma unroll
    for (int g = 1; g < kSplitGroups; ++g) {
      const float4 x = gsum[g * C4 + c];
      t.x += x.x;
      t.y += x.y;
      t.z += x.z;
      t.w += x.w;
    }
    reinterpret_cast<float4*>(out)[c] = make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
  }
  if (blockIdx.y == 0 && threadIdx.x == 0)
    a.lse[bh] = empty ? -INFINITY : (M + log2f(wsum)) * 0.69314718055994530942f;
}

}  // namespace

bool stage2_kernel(bool deep_prefetch, KernelEntry* e) {
  e->func = deep_prefetch ? reinterpret_cast<const void*>(&merge_splits<8>)
                          : reinterpret_cast<const void*>(&merge_splits<2>);
  e->threads = kMergeThreads;
  e->smem = 0;      // per plan: stage2_smem_bytes(Dv / tiles, max splits)
  return true;
}

}  // namespace pkvd
