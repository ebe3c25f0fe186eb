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
// always computed by warp 0 in the same lane-strided order, so every tiling
// gives identical bits. The merge waits on stage 1 with griddepcontrol.wait,
// so it can be launched early (programmatic dependent launch).
#include "device.cuh"
#include "kernels.h"

namespace pkvd {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__global__ void __launch_bounds__(256) merge_splits(const __grid_constant__ Stage2Args a) {
  extern __shared__ float w_s[];   // [S] weights
  __shared__ float stats[2];       // M, sum of weights

  const int bh = blockIdx.x;
  const int b = bh / a.heads;
  const int h = bh - b * a.heads;
  const int dt = a.dv / a.tiles;
  const int d0 = blockIdx.y * dt;

  pdl_wait_prerequisites();

  const int r0 = a.split_base[b];
  const int S = a.split_base[b + 1] - r0;

  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float m = -INFINITY;
    for (int s = lane; s < S; s += 32)
      m = fmaxf(m, a.lse_part[static_cast<int64_t>(r0 + s) * a.heads + h]);
#pragma unroll
    for (int x = 16; x >= 1; x >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, x));
    float ws = 0.f;
    for (int s = lane; s < S; s += 32) {
      const float l = a.lse_part[static_cast<int64_t>(r0 + s) * a.heads + h];
      const float w = (m == -INFINITY) ? 0.f : exp2f(l - m);
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

  const float* base = a.o_part + (static_cast<int64_t>(r0) * a.heads + h) * a.dv;
  const int64_t stride = static_cast<int64_t>(a.heads) * a.dv;
  float* out = a.out + static_cast<int64_t>(bh) * a.dv;
  for (int d = d0 + 4 * threadIdx.x; d < d0 + dt; d += 4 * blockDim.x) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int s = 0;
    for (; s + 4 <= S; s += 4) {
      float4 x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        x[u] = __ldg(reinterpret_cast<const float4*>(base + (s + u) * stride + d));
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float w = w_s[s + u];
        acc.x = fmaf(w, x[u].x, acc.x);
        acc.y = fmaf(w, x[u].y, acc.y);
        acc.z = fmaf(w, x[u].z, acc.z);
        acc.w = fmaf(w, x[u].w, acc.w);
      }
    }
    for (; s < S; ++s) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(base + s * stride + d));
      const float w = w_s[s];
      acc.x = fmaf(w, x.x, acc.x);
      acc.y = fmaf(w, x.y, acc.y);
      acc.z = fmaf(w, x.z, acc.z);
      acc.w = fmaf(w, x.w, acc.w);
    }
    *reinterpret_cast<float4*>(out + d) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (blockIdx.y == 0 && threadIdx.x == 0)
    a.lse[bh] = empty ? -INFINITY : (M + log2f(wsum)) * 0.69314718055994530942f;
}

}  // namespace

bool stage2_kernel(KernelEntry* e) {
  e->func = reinterpret_cast<const void*>(&merge_splits);
  e->threads = 0;   // chosen per plan
  e->smem = 0;      // S floats, per plan
  return true;
}

}  // namespace pkvd
