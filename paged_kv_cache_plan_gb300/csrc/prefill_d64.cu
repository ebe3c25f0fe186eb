// Dense causal prefill attention at head_dim 64 (prefill_d64_run in
// include/pkvd.h): every token of a prompt attends to the tokens at or before
// it. The rocm-libraries pull 10102 page (Motivation, Technical Details) is
// about this kernel's shared-memory layout at D = 64: there a 64-element row
// is half of one DMA row group, a per-row pad cannot be placed, and the pad
// goes between row groups to spread the LDS banks. Here a 64-element bf16 row
// is exactly one 128-byte swizzle row, so every tile moves with TMA in the
// canonical 128-byte-swizzled layout (16-byte chunk c of row r at
// r * 128 + ((c ^ (r % 8)) * 16) within 1 KB atoms): eight consecutive rows
// of a chunk land in eight distinct bank groups with no pad at all, and the
// tensor cores read the tiles through descriptors.
//
// One block per (request, query head, 128-query tile); six warps:
//   * warps 0-3: softmax, one query row per thread (tensor-memory lane =
//     row); the row's scores of a key tile are read from tensor memory once
//     into registers, masked on the diagonal tiles, P = exp2(s - m) goes to
//     shared memory, running sums in fp32;
//   * warp 4: TMA producer (the query tile once, then K and V tiles through
//     several stages, so the next tiles' copies are in flight during the
//     current tile's compute);
//   * warp 5: tensor-memory allocation and the MMA issue: S = Q K^T
//     (M = 128 queries, N = the tile's keys, K = 64) into an S buffer, then
//     O += P V (M = 128, N = 64, K = the tile's keys).
// Two shapes (PfShape below): query tiles before kOnePartFrom tokens keep P
// as a 16-bit high part plus the 16-bit rounding of its remainder (two
// products, ~16 significant bits: their first rows have a handful of keys,
// where one rounding of P would not average out) with 128-key tiles, one
// block per SM; later tiles use one part and 64-key tiles, small enough for
// three blocks per SM. The running maximum is lazy (raised only when a
// block's maximum exceeds it by more than 2^8); a raise rescales the
// thread's O row in tensor memory after the previous O product is complete.
// Causality: key tiles up to the diagonal of query tile qt; the diagonal
// tiles mask keys after the row's own position. Every wait is bounded; a
// wait that runs out sets the status word, and every role drains what it
// issued before the block frees its tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <type_traits>

#include "device.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pkvd {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int PD = 64;                 // head dim (K and V)
constexpr int BM = 128;                // queries per block
constexpr int TILE_Q = BM * PD * 2;    // 16 KB: the query tile
constexpr int PSLAB = BM * 128;        // 16 KB: 128 rows x 64 keys of P
constexpr int kThreads = 192;
constexpr int kSoftmaxWarps = 4, kProducerWarp = 4, kMmaWarp = 5;
constexpr float kLazyRescale = 8.f;    // log2 units
constexpr int kOnePartFrom = 1024;     // query positions from which P is one 16-bit part
constexpr int MISC = 256;

// Two shapes of the kernel. Query tiles before kOnePartFrom tokens (rows
// with few keys) keep P in two 16-bit parts and take 128-key tiles through
// four stages (208 KB, one block per SM); the later ones use one part and
// 64-key tiles (96 KB and 256 tensor-memory columns: two blocks per SM, so
// that two blocks' softmax warps share each SM sub-partition).
// Shared memory: [Q][K stages][V stages][P (high, low)][misc]; one P tile
// (the softmax writes P of tile j once O of tile j - 1 has read P of j - 1).
// Tensor memory: two S buffers of BN columns, then O (64 columns).
template <int kBN, int kStages, bool kTwoPart, int kMinBlocks, int kSBuf>
struct PfShape {
  static constexpr int SBUF = kSBuf;             // S buffers in tensor memory
  static constexpr int BN = kBN;                 // keys per tile
  static constexpr int STAGES = kStages;
  static constexpr bool TWO = kTwoPart;
  static constexpr int MINB = kMinBlocks;        // resident blocks per SM
  static constexpr int TILE_KV = BN * PD * 2;    // a K or V tile
  static constexpr int PPART = BM * BN * 2;      // one part of P
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + TILE_Q;
  static constexpr int OFF_V = OFF_K + STAGES * TILE_KV;
  static constexpr int OFF_P = OFF_V + STAGES * TILE_KV;
  static constexpr int OFF_MISC = OFF_P + (TWO ? 2 : 1) * PPART;
  static constexpr int SMEM = 1024 + OFF_MISC + MISC;   // 1 KB alignment slack
  static constexpr uint32_t OCOL = SBUF * BN;            // O after the S buffers
  static constexpr uint32_t TCOLS = OCOL + PD <= 128 ? 128 : OCOL + PD <= 256 ? 256 : 512;
  static_assert(SMEM * MINB + 1024 * MINB <= 233472, "shared memory per SM");
  static_assert(TCOLS * MINB <= 512, "tensor memory per SM");
  static_assert(BM % BN == 0 && BN % 64 == 0, "key tiles of 64 or 128");
};
using EarlyShape = PfShape<128, 4, true, 1, 2>;
using LateShape = PfShape<64, 2, false, 3, 1>;

struct PrefillArgs {
  float* out;            // [B, L, Hq, 64]
  float* lse;            // [B, L, Hq] natural log
  int32_t* status;       // device status word (kStatus* bits)
  int32_t batch, heads, kv_heads, seq_len;
  int32_t qt_first;      // query tiles qt_first .. qt_first + qt_count - 1
  int32_t qt_count;
  float scale_log2;
};

struct PrefillMaps {
  CUtensorMap q;         // {64, Hq, L, B}, box {64, 1, 128, 1}
  CUtensorMap k;         // {64, L, B * Hkv}, box {64, BN, 1}
  CUtensorMap v;
};

// byte offset of 16-byte chunk c (0..15: keys 8c .. 8c+7) of row r in a P part
__device__ __forceinline__ uint32_t p_off(int r, int c) {
  return (c >> 3) * PSLAB + (r >> 3) * 1024 + (r & 7) * 128 + ((((c & 7) ^ (r & 7))) << 4);
}

template <typename T, typename C>
__global__ void __launch_bounds__(kThreads, C::MINB)
    prefill_d64(const __grid_constant__ PrefillArgs a, const __grid_constant__ PrefillMaps maps) {
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr int BN = C::BN, kStages = C::STAGES, TILE = C::TILE_KV, PPART = C::PPART;
  constexpr int OFF_Q = C::OFF_Q, OFF_K = C::OFF_K, OFF_V = C::OFF_V, OFF_P = C::OFF_P;
  constexpr bool two_part = C::TWO;
  constexpr uint32_t TCOLS = C::TCOLS;
  constexpr uint32_t kIdS = tc::idesc_f16(kBf16, BM, BN, false, false);
  constexpr uint32_t kIdO = tc::idesc_f16(kBf16, BM, PD, false, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
  uint8_t* misc = sm + C::OFF_MISC;
  const uint32_t bars = smem_addr(misc);
  const uint32_t qfull = bars, kvfull = bars + 8, kvempty = bars + 8 + 8 * kStages,
                 sfull = bars + 8 + 16 * kStages, sfree = sfull + 16, pfull = sfree + 16,
                 pfree = pfull + 8, drain = pfree + 8;
  static_assert(8 + 16 * kStages + 16 + 16 + 8 + 8 + 8 <= 128, "barriers before the slot");
  uint32_t* tslot = reinterpret_cast<uint32_t*>(misc + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 132);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heavy (late) query tiles first
  const int bh_count = a.batch * a.heads;
  const int qt = a.qt_first + a.qt_count - 1 - static_cast<int>(blockIdx.x) / bh_count;
  const int bh = static_cast<int>(blockIdx.x) % bh_count;
  const int b = bh / a.heads, h = bh % a.heads;
  const int kvh = h / (a.heads / a.kv_heads);
  constexpr int kPer = BM / BN;                // key tiles per query tile
  const int nkv = (qt + 1) * kPer;             // key tiles up to the diagonal
  const int jdiag = qt * kPer;                 // first key tile that needs the causal mask

  pdl_launch_dependents();   // the second launch may take SMs this grid's tail leaves
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&maps.q);
    tma_prefetch_desc(&maps.k);
    tma_prefetch_desc(&maps.v);
    mbar_init(qfull, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(kvfull + 8 * i, 1);
      mbar_init(kvempty + 8 * i, 1);
    }
    for (int i = 0; i < C::SBUF; ++i) {
      mbar_init(sfull + 8 * i, 1);
      mbar_init(sfree + 8 * i, kSoftmaxWarps);
    }
    mbar_init(pfull, kSoftmaxWarps);
    mbar_init(pfree, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tc::alloc(smem_addr(tslot), TCOLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tslot;
  auto fail = [&]() {
    *abort_flag = 1;
    atomicOr(a.status, kStatusTimeout);
  };

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ TMA
    if (lane == 0) {
      const int kvrow = b * a.kv_heads + kvh;
      mbar_arrive_expect_tx(qfull, TILE_Q);
      tma_load_4d(smem_addr(sm + OFF_Q), &maps.q, 0, h, qt * BM, b, qfull);
      int issued = 0;
      for (int j = 0; j < nkv; ++j) {
        const int s = j % kStages;
        if (j >= kStages &&
            (*abort_flag || !mbar_wait(kvempty + 8 * s, (j / kStages - 1) & 1))) {
          fail();
          break;
        }
        mbar_arrive_expect_tx(kvfull + 8 * s, 2 * TILE);
        tma_load_3d(smem_addr(sm + OFF_K + s * TILE), &maps.k, 0, j * BN, kvrow, kvfull + 8 * s);
        tma_load_3d(smem_addr(sm + OFF_V + s * TILE), &maps.v, 0, j * BN, kvrow, kvfull + 8 * s);
        issued = j + 1;
      }
      // copies still in flight must land before the block exits
      mbar_wait(qfull, 0);
      for (int j = (issued >= kStages ? issued - kStages : 0); j < issued; ++j)
        mbar_wait(kvfull + 8 * (j % kStages), (j / kStages) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint64_t dq = tc::sdesc(smem_addr(sm + OFF_Q), 16, 1024);          // K-major
      const uint64_t dk0 = tc::sdesc(smem_addr(sm + OFF_K), 16, 1024);         // K-major
      const uint64_t dv0 = tc::sdesc(smem_addr(sm + OFF_V), TILE, 1024);       // MN-major
      const uint64_t dp0 = tc::sdesc(smem_addr(sm + OFF_P), 16, 1024);         // K-major
      constexpr uint64_t kTileStep = TILE >> 4, kPartStep = PPART >> 4, kSlabStep = PSLAB >> 4;
      const uint32_t tO = tbase + C::OCOL;
      bool ok = mbar_wait(qfull, 0);
      auto issue_s = [&](int j) -> bool {
        const int s = j % kStages, sb = j % C::SBUF;
        if (*abort_flag || !mbar_wait(kvfull + 8 * s, (j / kStages) & 1)) return false;
        if (j >= C::SBUF &&
            (*abort_flag || !mbar_wait(sfree + 8 * sb, (j / C::SBUF - 1) & 1)))
          return false;
        tc::fence_after();
        const uint32_t d = tbase + sb * BN;
        const uint64_t dk = dk0 + s * kTileStep;
#pragma unroll
        for (int k = 0; k < PD / 16; ++k) tc::mma_f16(d, dq + 2 * k, dk + 2 * k, kIdS, k > 0);
        tc::commit(sfull + 8 * sb);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < nkv; ++j) {
        if (j + 1 < nkv && !issue_s(j + 1)) {
          ok = false;
          break;
        }
        const int s = j % kStages;
        if (*abort_flag || !mbar_wait(pfull, j & 1)) {
          ok = false;
          break;
        }
        tc::fence_after();
        const uint64_t dv = dv0 + s * kTileStep;
        const uint64_t dph = dp0, dpl = dp0 + kPartStep;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t koff = (k >> 2) * kSlabStep + (k & 3) * 2;
          tc::mma_f16(tO, dph + koff, dv + k * (2048 >> 4), kIdO, j > 0 || k > 0);
          if (two_part) tc::mma_f16(tO, dpl + koff, dv + k * (2048 >> 4), kIdO, true);
        }
        tc::commit(kvempty + 8 * s);
        tc::commit(pfree);
      }
      if (!ok) fail();
      // every product issued must be complete before the memory is freed
      tc::commit(drain);
      mbar_wait(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;                           // query row of this thread
    const int qi = qt * BM + r;                          // its position
    const uint32_t lanes = static_cast<uint32_t>(32 * warp) << 16;
    const float sl2 = a.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool bad = false;
    auto wait_all = [&](uint32_t bar, uint32_t parity) {
      return __all_sync(kFull, !*abort_flag && mbar_wait(bar, parity));
    };
    for (int j = 0; j < nkv; ++j) {
      const int s = j % C::SBUF;   // S buffer
      if (!wait_all(sfull + 8 * s, (j / C::SBUF) & 1)) {
        bad = true;
        break;
      }
      tc::fence_after();
      // the row's unscaled scores, read once (keys after the row's own
      // position masked on the diagonal tile); the scale is folded into the
      // exponent's fused multiply-add below
      const uint32_t ts = tbase + lanes + s * BN;
      float sc[BN];
#pragma unroll
      for (int c4 = 0; c4 < BN / 32; ++c4) {
        uint32_t x[32];
        tc::ld32(ts + 32 * c4, x);
#pragma unroll
        for (int i = 0; i < 32; ++i) sc[32 * c4 + i] = __uint_as_float(x[i]);
      }
      // S buffer s is in registers: the MMA may overwrite it
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfree + 8 * s);
      if (j >= jdiag) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (j * BN + c > qi) sc[c] = -INFINITY;
      }
      // block maximum as eight independent chains (a single chain of 128
      // dependent maxima would cost its full latency every tile), on the
      // unscaled scores (the scale is positive), then scaled
      float mx[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx[k] = sc[k];
#pragma unroll
      for (int c = 8; c < BN; ++c) mx[c & 7] = fmaxf(mx[c & 7], sc[c]);
      const float mb = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
      bool need = false;
      float alpha = 1.f;
      if (j == 0) {
        m = mb;
      } else if (mb > m + kLazyRescale) {
        need = true;
        alpha = ex2(m - mb);
        m = mb;
        l *= alpha;
      }
      // P = exp2(s * scale - m): one paired fused multiply-add forms two
      // exponents, one paired add takes two P into the row sum (four chains
      // of pairs)
      {
        const uint64_t scale2 = f32x2(sl2, sl2), negm2 = f32x2(-m, -m);
        uint64_t ls[4] = {0ull, 0ull, 0ull, 0ull};   // +0.0f pairs
#pragma unroll
        for (int c = 0; c < BN; c += 2) {
          const float2 e = f32x2_split(ffma_x2(f32x2(sc[c], sc[c + 1]), scale2, negm2));
          sc[c] = ex2(e.x);
          sc[c + 1] = ex2(e.y);
          ls[(c >> 1) & 3] = fadd_x2(ls[(c >> 1) & 3], f32x2(sc[c], sc[c + 1]));
        }
        const float2 l01 = f32x2_split(fadd_x2(ls[0], ls[1]));
        const float2 l23 = f32x2_split(fadd_x2(ls[2], ls[3]));
        l += (l01.x + l01.y) + (l23.x + l23.y);
      }
      // O of tile j - 1 must be complete before its P tile is rewritten and
      // before O is rescaled
      if (j >= 1 && !wait_all(pfree, (j - 1) & 1)) {
        bad = true;
        break;
      }
      if (__any_sync(kFull, need)) {
        tc::fence_after();
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t o[32];
          tc::ld32(tbase + lanes + C::OCOL + 32 * half, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tc::st32(tbase + lanes + C::OCOL + 32 * half, o);
        }
        tc::wait_st();
      }
      uint8_t* ph = sm + OFF_P;
      uint8_t* pl = ph + PPART;
#pragma unroll
      for (int g = 0; g < BN / 8; ++g) {   // 16-byte chunks of 8 keys
        uint32_t hi[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) hi[e] = pack2<T>(sc[8 * g + 2 * e], sc[8 * g + 2 * e + 1]);
        const uint32_t off = p_off(r, g);
        *reinterpret_cast<uint4*>(ph + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        if (two_part) {
          uint32_t lo[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 rh = unpack2<T>(hi[e]);
            lo[e] = pack2<T>(sc[8 * g + 2 * e] - rh.x, sc[8 * g + 2 * e + 1] - rh.y);
          }
          *reinterpret_cast<uint4*>(pl + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
      }
      // P (generic-proxy writes) goes to the tensor cores (async proxy)
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull);
    }
    if (bad) {
      if (lane == 0) fail();
    } else if (wait_all(pfree, (nkv - 1) & 1)) {
      tc::fence_after();
      uint32_t o[2][32];
      tc::ld32(tbase + lanes + C::OCOL, o[0]);
      tc::ld32(tbase + lanes + C::OCOL + 32, o[1]);
      if (qi < a.seq_len) {
        const float inv = 1.f / l;
        const int64_t row = (static_cast<int64_t>(b) * a.seq_len + qi) * a.heads + h;
        float4* dst = reinterpret_cast<float4*>(a.out + row * PD);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[8 * hh + i] = make_float4(__uint_as_float(o[hh][4 * i]) * inv,
                                          __uint_as_float(o[hh][4 * i + 1]) * inv,
                                          __uint_as_float(o[hh][4 * i + 2]) * inv,
                                          __uint_as_float(o[hh][4 * i + 3]) * inv);
        a.lse[row] = (m + log2f(l)) * 0.69314718055994530942f;
      }
    } else if (lane == 0) {
      fail();
    }
  }

  tc::fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after();
    tc::dealloc(tbase, TCOLS);
  }
  // The second launch (programmatic dependent launch) finishes only once the
  // first has, so whatever follows in the stream sees both; for the first
  // launch this returns at once.
  pdl_wait_prerequisites();
}

}  // namespace
}  // namespace pkvd

extern "C" int prefill_d64_run(const pkvd_prefill_desc* desc, const void* q, const void* k,
                               const void* v, float* out, float* lse, int32_t* status,
                               pkvd_stream_t stream) {
  using namespace pkvd;
  if (!desc || !q || !k || !v || !out || !lse || !status) return PKVD_EINVAL;
  const pkvd_prefill_desc& d = *desc;
  if (d.batch < 1 || d.heads < 1 || d.kv_heads < 1 || d.seq_len < 1 || d.reserved[0] ||
      d.reserved[1] || !(d.scale >= 0.f))
    return PKVD_EINVAL;
  if (d.dtype != PKVD_BF16 && d.dtype != PKVD_FP16) return PKVD_EINVAL;
  if (d.heads % d.kv_heads != 0) return PKVD_EUNSUPPORTED;
  for (const void* p : {q, k, v, static_cast<const void*>(out), static_cast<const void*>(lse)})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return PKVD_EINVAL;
  const int64_t q_tiles = (static_cast<int64_t>(d.seq_len) + BM - 1) / BM;
  const int64_t blocks = q_tiles * d.batch * d.heads;
  if (blocks > 0x7fffffffLL || static_cast<int64_t>(d.batch) * d.kv_heads > 0x7fffffffLL)
    return PKVD_EUNSUPPORTED;

  PrefillArgs a;
  a.out = out;
  a.lse = lse;
  a.status = status;
  a.batch = d.batch;
  a.heads = d.heads;
  a.kv_heads = d.kv_heads;
  a.seq_len = d.seq_len;
  const float scale = d.scale > 0.f ? d.scale : 0.125f;   // 1 / sqrt(64)
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);

  const uint64_t L = static_cast<uint64_t>(d.seq_len);
  PrefillMaps maps;
  {
    const uint64_t dims[4] = {PD, static_cast<uint64_t>(d.heads), L, static_cast<uint64_t>(d.batch)};
    const uint64_t strides[3] = {PD * 2, static_cast<uint64_t>(d.heads) * PD * 2,
                                 L * d.heads * PD * 2};
    const uint32_t box[4] = {PD, 1, BM, 1};
    const int rc = encode_tiled_map(d.dtype, q, 4, dims, strides, box, &maps.q);
    if (rc != PKVD_OK) return rc;
  }
  // one launch per kernel shape: query tiles before kOnePartFrom tokens, then the rest
  const int64_t early = std::min<int64_t>(q_tiles, kOnePartFrom / BM);
  bool after_first = false;   // the second launch overlaps the first's tail
  auto launch = [&](auto shape, int64_t qt_first, int64_t qt_count) -> int {
    using C = decltype(shape);
    if (qt_count <= 0) return PKVD_OK;
    const uint64_t dims[3] = {PD, L, static_cast<uint64_t>(d.batch) * d.kv_heads};
    const uint64_t strides[2] = {PD * 2, L * PD * 2};
    const uint32_t box[3] = {PD, C::BN, 1};
    int rc = encode_tiled_map(d.dtype, k, 3, dims, strides, box, &maps.k);
    if (rc == PKVD_OK) rc = encode_tiled_map(d.dtype, v, 3, dims, strides, box, &maps.v);
    if (rc != PKVD_OK) return rc;
    a.qt_first = static_cast<int32_t>(qt_first);
    a.qt_count = static_cast<int32_t>(qt_count);
    const void* fn = d.dtype == PKVD_FP16 ? reinterpret_cast<const void*>(&prefill_d64<__half, C>)
                                          : reinterpret_cast<const void*>(&prefill_d64<__nv_bfloat16, C>);
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
        cudaSuccess)
      return PKVD_ECUDA;
    void* args[] = {&a, &maps};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(qt_count * d.batch * d.heads));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(C::SMEM);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = after_first ? 1 : 0;
    if (cudaLaunchKernelExC(&cfg, fn, args) != cudaSuccess) return PKVD_ECUDA;
    after_first = true;
    return PKVD_OK;
  };
  // the long late tiles first, so the short early ones fill the tail
  int rc = launch(LateShape{}, early, q_tiles - early);
  if (rc == PKVD_OK) rc = launch(EarlyShape{}, 0, early);
  return rc;
}
