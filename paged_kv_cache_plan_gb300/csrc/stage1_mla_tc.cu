// Stage 1 for MLA on the fifth-generation tensor cores (tcgen05): one block
// per work item (request b, block of 64 (query token, head) rows, the last
// block of a request zero-padded when its rows are not a multiple of 64,
// split s; or, for a
// shared-prefix item, the heads of up to 64 / heads consecutive requests
// over their common prefix, read through the first member's page table,
// each head's partial going to its own request's partial row); all heads
// share the 576-wide latent row of each token and V is its first 512
// elements. This is the head-batched stage-1 of the aiter pull 4758 page
// (Motivation, Technical Details 1) with the keys, not the heads, as the M
// side of the products, because 64 heads x 512 fp32 output columns already
// fill half of the tensor memory:
//
//   S^T [64 keys x 64 heads] = K [64 keys x 576] . Q^T              (M = 64)
//   O^T [512 x 64 heads]    += V^T [512 x 64 keys] . P^T [64 keys x 64 heads]
//                                                      (four M = 128 tiles)
//
// Tensor memory (512 columns): O^T tile t in columns 64t .. 64t+63, two S^T
// buffers in columns 256 .. 383 (an M = 64 accumulator occupies lanes 0-15
// of each 32-lane quarter: row i sits in lane 32 (i / 16) + i % 16), and the
// softmax threads' running sums of P in columns 384 .. 447.
//
// Shared memory, all operands in the 128-byte-swizzled layout: the Q tile
// (K-major, rows = heads), two K/V stages of nine 64-column slabs (one tile
// serves as the K-major A operand of S^T and as the MN-major A operand of
// O^T), and the P^T tile (MN-major, rows = keys). Shared memory holds two
// stages.
//
// Roles:
//   warps 0-3   copy each block slab by slab as 16-byte cp.async chunks
//               placed directly in the swizzled layout (one page per token
//               leaves no contiguous tile to move); thread t copies rows
//               t / 8 + 16 i (i < 4), chunk t % 8 of every slab; a slab's
//               barrier completes when every copying thread's chunks of it
//               have landed. A stage is refilled once the O^T of the block
//               two back is complete (releasing it slab pair by slab pair as
//               the O^T tiles complete measured slower: the early copies
//               compete with O^T for shared-memory bandwidth);
//   warp 12     allocates the tensor memory; one thread issues each block's
//               S^T products three slabs at a time as the slabs land (after
//               a proxy fence: the copies wrote shared memory through the
//               generic proxy, the tensor cores read it through the async
//               proxy);
//   warp 13     one thread issues each block's O^T products as soon as its P
//               is ready (a separate issuer, so that neither kind of product
//               waits behind the other's barrier);
//   warps 4-11  the softmax. Warp w reads the S^T lanes of quarter w % 4 (16
//               keys) for 32 of the 64 heads with 16-lane tensor-memory
//               loads, which spread the 16 x 32 scores over all 32 threads
//               (two keys x eight heads each). The running maximum per head is
//               lazy: it is only raised when a block's scores exceed it by
//               more than 2^8, so most blocks need no cross-warp reduction at
//               all, only a vote; P = exp2(s - m) then lies below 2^8, which
//               the 16-bit P and the fp32 sums absorb. When a head's maximum
//               is raised, the block maxima are folded over threads (xor
//               shuffles) and quarters (shared memory), and O^T and the
//               running sums of that head are rescaled. P is rounded to one
//               16-bit value.
#include <type_traits>

#include "device.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace pkvd {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr float kLazyRescale = 8.f;   // log2 units
// Reference maximum of a row that sees no token of its item's first block
// (several query tokens: the causal cut). Finite, so P = exp2(-inf - m) = 0
// and a later raise scales the (zero) row by exp2(floor - m) = 0.
constexpr float kNoTokenMax = -1e30f;
constexpr int kSlabs = kMlaDk / 64;   // 9

// Byte offset, in a tile of 64-column slabs of `slab_bytes` each, of 16-byte
// chunk ch (0..71) of row r, 128-byte swizzle.
__device__ __forceinline__ uint32_t swz_off(int r, int ch, int slab_bytes) {
  return (ch >> 3) * slab_bytes + (r >> 3) * 1024 + (r & 7) * 128 + (((ch & 7) ^ (r & 7)) << 4);
}

// CAUSAL: several query tokens per request (q_len > 1), each row cut at its
// token's position; the one-token kernel has no per-row cut.
template <typename T, bool CAUSAL>
__global__ void __launch_bounds__(kMlaTcThreads, 1)
    mla_tc(const __grid_constant__ Stage1Args a, const __grid_constant__ KvTensorMaps) {
  constexpr int R = kMlaTcHeads;              // 64 heads = N of both products
  constexpr int BLK = kMlaTcBlockTokens;      // 64 keys
  constexpr int SLAB = kMlaTcSlabBytes;       // one 64-column slab of 64 rows
  constexpr int STAGE = kMlaTcStageBytes;
  constexpr int CH = kMlaDk * 2 / 16;         // 72 16-byte chunks per row
  constexpr int MMA_WARP = kMlaTcLoadWarps + kMlaTcSoftmaxWarps;   // S^T issue, tensor memory
  constexpr int O_WARP = MMA_WARP + 1;                              // O^T issue
  constexpr int LDT = kMlaTcLoadWarps * 32;   // copying threads
  constexpr int SMX = kMlaTcSoftmaxWarps * 32;
  constexpr int TCOLS = 512;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t kIdS = tc::idesc_f16(kBf16, BLK, R, false, false);
  constexpr uint32_t kIdO = tc::idesc_f16(kBf16, 128, R, true, true);
  static_assert(SLAB == R * 128, "the Q tile and the K/V stages share one slab size");
  static_assert(4 * R + 2 * R + 64 <= TCOLS, "tensor memory columns");
  static_assert(LDT == 2 * BLK && kMlaTcSoftmaxWarps == 8, "warp roles");

  extern __shared__ uint8_t raw[];
  uint8_t* sm = raw + ((kTileAlign - (smem_addr(raw) & (kTileAlign - 1))) & (kTileAlign - 1));
  uint8_t* qs = sm;
  uint8_t* stages = qs + kMlaTcQBytes;
  uint8_t* ps = stages + kMlaTcStages * STAGE;
  uint8_t* misc = ps + kMlaTcPBytes;
  const uint32_t bars = smem_addr(misc);
  const uint32_t full = bars;               // [2][9] slab landed (128 copying threads)
  const uint32_t empty = bars + 144;        // [2] O of the stage's block done (MMA commit)
  const uint32_t sfull = bars + 160;        // [2] S^T buffer written (MMA commit)
  const uint32_t sfree = bars + 176;        // [2] S^T buffer read out (8 softmax warps)
  const uint32_t pfull = bars + 192;        // P^T written, O rescaled if needed (8 warps)
  const uint32_t odone = bars + 200;        // O of the latest block done (MMA commit)
  const uint32_t drain = bars + 208;        // every S^T product done (at exit)
  const uint32_t drain_o = bars + 216;      // every O^T product done (at exit)
  const uint32_t qfull = bars + 224;        // the Q tile landed (every thread)
  uint32_t* tslot = reinterpret_cast<uint32_t*>(misc + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 260);
  volatile int* resc_flag = reinterpret_cast<volatile int*>(misc + 264);   // [2]
  float* m_ref = reinterpret_cast<float*>(misc + 512);      // [64] running maxima (log2)
  float* alpha_s = reinterpret_cast<float*>(misc + 768);    // [64] rescale factors, then 1 / l
  float* red = reinterpret_cast<float*>(misc + 1024);       // [4 quarters][64]
  static_assert(1024 + 4 * 64 * 4 <= kMlaTcMiscBytes, "scratch area");

  const pkvd_work_item it = a.items[blockIdx.x];
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = it.tok_end - it.tok_begin;
  const int nblk = (n + BLK - 1) / BLK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      for (int c = 0; c < kSlabs; ++c) mbar_init(full + 8 * (s * kSlabs + c), LDT);
      mbar_init(empty + 8 * s, 1);
      mbar_init(sfull + 8 * s, 1);
      mbar_init(sfree + 8 * s, kMlaTcSoftmaxWarps);
    }
    mbar_init(pfull, kMlaTcSoftmaxWarps);
    mbar_init(odone, 1);
    mbar_init(drain, 1);
    mbar_init(drain_o, 1);
    mbar_init(qfull, kMlaTcThreads);
    *abort_flag = 0;
    fence_barrier_init();
  }
  // (query token, head) rows of a request: row v is query token v / heads,
  // head v % heads (grouped shared-prefix items have one query token)
  const int VH = a.q_len * a.heads;
  // Query row r of the item: row unit * 64 + r of the request, or (grouped
  // shared-prefix item) head r % heads of member r / heads; -1 for the unused
  // rows (past the request's last row when its rows are not a multiple of
  // 64, or of a group with fewer members than fit).
  auto q_row = [&](int r) -> int64_t {
    if (!it.grouped)
      return it.unit * R + r < VH ? static_cast<int64_t>(it.request) * VH + it.unit * R + r : -1;
    const int m = r / a.heads;
    return m < it.unit ? static_cast<int64_t>(it.request + m) * a.heads + (r - m * a.heads) : -1;
  };
  // Partial-output row of query row r (-1: unused).
  auto out_row = [&](int r) -> int64_t {
    if (!it.grouped)
      return it.unit * R + r < VH ? static_cast<int64_t>(it.partial_row) * VH + it.unit * R + r
                                  : -1;
    const int m = r / a.heads;
    return m < it.unit
               ? static_cast<int64_t>(a.split_base[it.request + m] + it.split) * a.heads +
                     (r - m * a.heads)
               : -1;
  };
  // Partial-lse index of query row r (head-major lse array; -1: unused).
  auto lse_idx = [&](int r) -> int64_t {
    if (!it.grouped)
      return it.unit * R + r < VH
                 ? static_cast<int64_t>(it.unit * R + r) * a.lse_stride + it.partial_row
                 : -1;
    const int m = r / a.heads;
    return m < it.unit ? static_cast<int64_t>(r - m * a.heads) * a.lse_stride +
                             a.split_base[it.request + m] + it.split
                       : -1;
  };
  // K/V rows of the item: the request's page table; token of block row r of
  // block j (rows past the item's end repeat its last token, their keys are
  // masked). The page ids of a row are read ahead of use (page_of) and turned
  // into byte offsets later (off_of, in the copying warps).
  const int32_t* pt = a.page_table + static_cast<int64_t>(it.request) * a.pt_stride;
  auto tok_of = [&](int j, int r) -> int {
    const int tok = it.tok_begin + j * BLK + r;
    return tok < it.tok_end ? tok : it.tok_end - 1;
  };
  auto page_of = [&](int j, int r) -> int { return ld_pinned(pt + tok_of(j, r) / a.page_size); };
  // the copying threads' page ids of the first two blocks, read before the
  // query tile so that the two round trips overlap
  int pg0[4] = {0, 0, 0, 0}, pg1[4] = {0, 0, 0, 0};
  if (warp < kMlaTcLoadWarps) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (nblk > 0) pg0[i] = page_of(0, threadIdx.x / 8 + 16 * i);
      if (nblk > 1) pg1[i] = page_of(1, threadIdx.x / 8 + 16 * i);
    }
  }
  // Q tile: the 64 query rows, K-major, moved with cp.async so that all of
  // its loads are in flight together (an unused row's chunks copy no source
  // bytes and fill zeros). Nobody waits for it here: every thread arrives on
  // qfull once its chunks have landed, and only the S^T issue waits, so the
  // first K/V copies go out while the tile is still on its way.
  for (int i = threadIdx.x; i < R * CH; i += kMlaTcThreads) {
    const int r = i / CH, ch = i - r * CH;
    const int64_t qr = q_row(r);
    cp_async16_zfill(smem_addr(qs + swz_off(r, ch, SLAB)),
                     static_cast<const uint8_t*>(a.q) + (qr >= 0 ? qr * (kMlaDk * 2) + ch * 16 : 0),
                     qr >= 0 ? 16u : 0u);
  }
  if (warp == MMA_WARP) tc::alloc(smem_addr(tslot), TCOLS);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tslot;
  cp_async_arrive(qfull);   // the barrier's initialisation is visible after the sync

  if (warp < kMlaTcLoadWarps) {
    // ------------------------------------------------------------ copies
    const int tid = threadIdx.x;
    const int cq = tid & 7;                          // 16-byte chunk within a slab row
    const uint8_t* pool = static_cast<const uint8_t*>(a.k);
    const int64_t pitch_bytes = a.k_pitch * 2;
    // The page id of a row is loaded two blocks ahead, before that block's
    // copies, and its byte offset formed after the next block's copies
    // (page_of, then off_of), so that the cold page-table read never holds
    // up the copies being issued.
    auto off_of = [&](int j, int r, int page) -> int64_t {
      const int tok = tok_of(j, r);
      const int pidx = tok / a.page_size;
      if (a.checks) {
        // a grouped item reads the shared tokens through its first member's
        // page table: the other members must name the same pages
        for (int m = 1; it.grouped && m < it.unit; ++m)
          if (__ldg(pt + m * a.pt_stride + pidx) != page) atomicOr(a.status, kStatusBadPage);
        if (page < 0 || page >= a.num_pool_pages) {
          atomicOr(a.status, kStatusBadPage);
          page = 0;
        }
      }
      return (static_cast<int64_t>(page) * a.page_size + (tok - pidx * a.page_size)) *
             pitch_bytes;
    };
    // this thread's rows of a block: tid / 8 + 16 i
    int64_t cur[4];
    int pg[4];   // page ids of the next block's rows
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      cur[i] = nblk > 0 ? off_of(0, tid / 8 + 16 * i, pg0[i]) : 0;
      pg[i] = pg1[i];
    }
    for (int j = 0; j < nblk; ++j) {
      const int s = j & 1;
      int pg2[4];   // page ids of block j + 2
#pragma unroll
      for (int i = 0; i < 4; ++i) pg2[i] = j + 2 < nblk ? page_of(j + 2, tid / 8 + 16 * i) : 0;
      if (j >= 2) {
        const bool ok = !*abort_flag && mbar_wait(empty + 8 * s, ((j >> 1) - 1) & 1);
        if (!__all_sync(kFull, ok)) {
          if (lane == 0) {
            *abort_flag = 1;
            atomicOr(a.status, kStatusTimeout);
          }
          break;
        }
      }
      const uint32_t st = smem_addr(stages + s * STAGE);
      // Each slab is announced asynchronously once this thread's copies of it
      // have landed (cp.async arrive); the MMA thread fences them for the
      // async proxy before its tensor-core reads.
#pragma unroll 1
      for (int c = 0; c < kSlabs; ++c) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          cp_async16(st + swz_off(tid / 8 + 16 * i, 8 * c + cq, SLAB),
                     pool + cur[i] + (8 * c + cq) * 16);
        cp_async_arrive(full + 8 * (s * kSlabs + c));
      }
      // the next block's offsets from ids loaded a block ago
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (j + 1 < nblk) cur[i] = off_of(j + 1, tid / 8 + 16 * i, pg[i]);
        pg[i] = pg2[i];
      }
    }
    cp_async_wait_all();
  } else if (warp == MMA_WARP || warp == O_WARP) {
    // ------------------------------------------------------------ MMA issue
    // Two issuing threads, so that neither product waits behind the other's
    // barrier: warp 12 issues each block's S^T three slabs at a time as its
    // slabs land, warp 13 each block's O^T as soon as its P is ready. They write
    // disjoint tensor-memory columns and read different shared memory, and
    // each commits (and at the end drains) only what it issued itself.
    // Descriptors are built once; a byte offset d within the first 256 KB of
    // shared memory moves a descriptor by d / 16 in its start field, so every
    // product below is one add and one issue (an issuing thread is bound by
    // its instruction latency, not by the tensor pipe).
    if (lane == 0 && nblk > 0) {
      constexpr uint64_t kStageStep = STAGE >> 4, kSlabStep = SLAB >> 4;
      bool ok = true;
      if (warp == MMA_WARP) {
        const uint64_t dq = tc::sdesc(smem_addr(qs), 16, 1024);
        const uint64_t dk0 = tc::sdesc(smem_addr(stages), 16, 1024);   // K-major
        // the Q tile (fenced for the async proxy below, with the slabs)
        ok = mbar_wait(qfull, 0);
        for (int js = 0; ok && js < nblk; ++js) {
          // the S^T buffer must have been read out by block js - 2's softmax
          if (js >= 2) ok = !*abort_flag && mbar_wait(sfree + 8 * (js & 1), ((js >> 1) - 1) & 1);
          const uint32_t d = tbase + 4 * R + (js & 1) * R;
          const uint64_t dk = dk0 + (js & 1) * kStageStep;
          // a few slabs at a time: a copying thread's arrival on a slab's
          // barrier comes after all of its earlier copies, so the last
          // slab's barrier of a group covers the group (one wait and one pair
          // of fences per group: the issuing thread's own instructions, not
          // the tensor pipe, set the rate of these small products)
          constexpr int kGroupEnd[] = {2, 5, 8};   // last slab of each group
          constexpr int kGroups = sizeof(kGroupEnd) / sizeof(kGroupEnd[0]);
          static_assert(kGroupEnd[kGroups - 1] == kSlabs - 1, "the groups cover the slabs");
#pragma unroll
          for (int gr = 0; gr < kGroups; ++gr) {
            if (ok) ok = mbar_wait(full + 8 * ((js & 1) * kSlabs + kGroupEnd[gr]), (js >> 1) & 1);
            if (!ok) break;
            // the slabs landed through the generic proxy; the tensor cores
            // read them through the async proxy
            fence_proxy_async_smem();
            tc::fence_after();
#pragma unroll
            for (int c = gr == 0 ? 0 : kGroupEnd[gr - 1] + 1; c <= kGroupEnd[gr]; ++c)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                tc::mma_f16(d, dk + c * kSlabStep + 2 * k, dq + c * kSlabStep + 2 * k, kIdS,
                            c > 0 || k > 0);
          }
          if (ok) tc::commit(sfull + 8 * (js & 1));
        }
        // every product this thread issued must be done before the tensor
        // memory is freed
        tc::commit(drain);
        mbar_wait(drain, 0);
      } else {
        const uint64_t dv0 = tc::sdesc(smem_addr(stages), SLAB, 1024);   // MN-major
        const uint64_t dp = tc::sdesc(smem_addr(ps), SLAB, 1024);
        for (int jo = 0; ok && jo < nblk; ++jo) {
          ok = !*abort_flag && mbar_wait(pfull, jo & 1);
          if (!ok) break;
          tc::fence_after();
          const uint64_t dv = dv0 + (jo & 1) * kStageStep;
#pragma unroll
          for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int k = 0; k < BLK / 16; ++k)
              tc::mma_f16(tbase + t * R, dv + t * 2 * kSlabStep + k * (2048 >> 4),
                          dp + k * (2048 >> 4), kIdO, jo > 0 || k > 0);
          tc::commit(empty + 8 * (jo & 1));
          tc::commit(odone);
        }
        tc::commit(drain_o);
        mbar_wait(drain_o, 0);
      }
      if (!ok) {
        *abort_flag = 1;
        atomicOr(a.status, kStatusTimeout);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int q = warp & 3;                         // tensor-memory lane quarter
    const int h = (warp - kMlaTcLoadWarps) >> 2;    // heads 32h .. 32h+31
    const int cl = lane & 15;
    // The quarter's 16 keys x the warp's 32 rows are spread over all 32
    // threads (16-lane tensor-memory loads): value v (< 16) of this thread is
    // key key0 + 8 ((v / 2) % 2), column 8 (v / 4) + 2 tq4 + v % 2 of the 32.
    const int tq4 = lane & 3;
    const int key0 = 16 * q + (lane >> 2);
    auto col_of = [&](int v) { return 8 * (v >> 2) + 2 * tq4 + (v & 1); };
    const uint32_t lanes = static_cast<uint32_t>(32 * q) << 16;
    const bool decider = q == 0;                    // warps 4 and 8 finish the reductions
    const float sl2 = a.scale_log2;
    // running sums of P per (key slot, row), in the free tensor-memory
    // columns 384 + 32h .. in the same 16-lane layout (registers are the
    // scarce resource)
    const uint32_t lcols = tbase + lanes + 6 * R + 32 * h;
    // Causal cut among the query tokens: row c of this warp's 32 sees the
    // item's tokens up to vis0 + (query token of the row); blocks that end at
    // or before vis0 need no per-row test (all of them, with one token).
    const int vis0 = it.query_pos - it.tok_begin;
    const int row0 = it.grouped ? 0 : it.unit * R + 32 * h;   // first row of this warp
    // this thread's 16 scaled scores of block j (keys past the end or not yet
    // visible to the row: -inf)
    auto scores = [&](int j, int b, float (&x)[16]) {
      uint32_t r[16];
      tc::ld16x4(tbase + lanes + 4 * R + b * R + 32 * h, r);
      const int nv = min(BLK, n - j * BLK);
      const bool valid0 = key0 < nv, valid1 = key0 + 8 < nv;
      if (!CAUSAL || (j + 1) * BLK - 1 <= vis0) {
#pragma unroll
        for (int v = 0; v < 16; ++v)
          x[v] = ((v & 2) ? valid1 : valid0) ? __uint_as_float(r[v]) * sl2 : -INFINITY;
      } else {
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          const int kj = j * BLK + key0 + 4 * (v & 2);
          const int tok_j = it.grouped ? 0 : (row0 + col_of(v)) / a.heads;
          x[v] = ((v & 2) ? valid1 : valid0) && kj <= vis0 + tok_j ? __uint_as_float(r[v]) * sl2
                                                                 : -INFINITY;
        }
      }
    };
    bool bad = false;

    for (int j = 0; j < nblk; ++j) {
      const int b = j & 1;
      const bool ok = __all_sync(kFull, !*abort_flag && mbar_wait(sfull + 8 * b, (j >> 1) & 1));
      const bool o_prev = j == 0 || mbar_test(odone, (j - 1) & 1);
      float x[16];
      bool need = j == 0;
      if (ok) {
        tc::fence_after();
        scores(j, b, x);
        if (j > 0) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 m2 = *reinterpret_cast<const float2*>(m_ref + 32 * h + 8 * i + 2 * tq4);
            need |= x[4 * i] > m2.x + kLazyRescale;
            need |= x[4 * i + 1] > m2.y + kLazyRescale;
            need |= x[4 * i + 2] > m2.x + kLazyRescale;
            need |= x[4 * i + 3] > m2.y + kLazyRescale;
          }
        }
      } else {
        *abort_flag = 1;
      }
      // one vote per block: raise some maximum (or stop)
      bool o_ready = false;
      if (named_sync_or(1, SMX, need || !ok)) {
        if (*abort_flag) {
          bad = true;
          break;
        }
        // -------- slow path: raise the reference maxima of the heads that need it
        {
          // block maxima over this quarter's keys: the thread's two keys,
          // then the eight threads that share its columns
          float bm[8];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 2; ++e) bm[2 * i + e] = fmaxf(x[4 * i + e], x[4 * i + 2 + e]);
#pragma unroll
          for (int off = 4; off < 32; off <<= 1)
#pragma unroll
            for (int k = 0; k < 8; ++k) bm[k] = fmaxf(bm[k], __shfl_xor_sync(kFull, bm[k], off));
          if (lane < 4) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int e = 0; e < 2; ++e) red[q * 64 + 32 * h + 8 * i + 2 * lane + e] = bm[2 * i + e];
          }
        }
        named_sync(1, SMX);
        if (decider && lane < 16) {
          bool raise = false;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int col = 32 * h + 2 * cl + e;
            const float bm =
                fmaxf(fmaxf(red[col], red[64 + col]), fmaxf(red[128 + col], red[192 + col]));
            const float mo = m_ref[col];
            float mn = mo, al = 1.f;
            if (j == 0) {
              // a row that sees no token of the first block (causal cut)
              // starts from a finite floor, so that P = exp2(-inf - m) = 0
              mn = CAUSAL && bm == -INFINITY ? kNoTokenMax : bm;
            } else if (bm > mo + kLazyRescale) {
              mn = bm;
              al = ex2(mo - mn);
              raise = true;
            }
            m_ref[col] = mn;
            alpha_s[col] = al;
          }
          const bool any = __any_sync(0x0000ffffu, raise);
          if (lane == 0) resc_flag[h] = any ? 1 : 0;
        }
        named_sync(1, SMX);
        if (resc_flag[0] | resc_flag[1]) {
          // O of the previous block must be done before it is rescaled
          if (!__all_sync(kFull, !*abort_flag && mbar_wait(odone, (j - 1) & 1))) *abort_flag = 1;
          o_ready = true;
          tc::fence_after();
          // scale the O^T columns of this warp's heads (all four dv tiles,
          // this quarter's lanes) and the running sums
          // (the factors are re-read per tile: hoisted out of the loop they
          // would hold 32 more registers across it, on this rare path)
          const volatile float* al = alpha_s + 32 * h;
#pragma unroll 1
          for (int t = 0; t < 4; ++t) {
            const uint32_t cols = tbase + lanes + t * R + 32 * h;
            uint32_t o[32];
            tc::ld32(cols, o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * al[c]);
            tc::st32(cols, o);
          }
          {
            uint32_t lv[16];
            tc::ld16x4(lcols, lv);
#pragma unroll
            for (int v = 0; v < 16; ++v)
              lv[v] = __float_as_uint(__uint_as_float(lv[v]) * alpha_s[32 * h + col_of(v)]);
            tc::st16x4(lcols, lv);
          }
          tc::wait_st();
        }
        // read the scores again: keeping them live across the rescale costs
        // more registers than this rare second load
        scores(j, b, x);
      }
      // O of the previous block must be done before P^T is rewritten (a wait
      // that runs out stops the loop at the next vote)
      if (j >= 1 && !o_ready &&
          !__all_sync(kFull, o_prev || (!*abort_flag && mbar_wait(odone, (j - 1) & 1))))
        *abort_flag = 1;
      // P = exp2(s - m); P^T in the inputs' 16-bit type into shared memory
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 m2 = *reinterpret_cast<const float2*>(m_ref + 32 * h + 8 * i + 2 * tq4);
        x[4 * i] = ex2(x[4 * i] - m2.x);
        x[4 * i + 1] = ex2(x[4 * i + 1] - m2.y);
        x[4 * i + 2] = ex2(x[4 * i + 2] - m2.x);
        x[4 * i + 3] = ex2(x[4 * i + 3] - m2.y);
      }
      // two adjacent columns of one key per 4-byte store: row key, 16-byte
      // chunk 4h + i of the 128-byte-swizzled P^T tile, word tq4
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const int key = key0 + 8 * kk;
        uint8_t* prow = ps + (key >> 3) * 1024 + (key & 7) * 128 + 4 * tq4;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          *reinterpret_cast<uint32_t*>(prow + (((4 * h + i) ^ (key & 7)) << 4)) =
              pack2<T>(x[4 * i + 2 * kk], x[4 * i + 2 * kk + 1]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull);
      // S^T buffer b was read out before P
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sfree + 8 * b);
      // running sums of P in fp32 (the log-sum-exp needs them unrounded)
      {
        tc::fence_after();
        uint32_t l[16];
        if (j > 0) tc::ld16x4(lcols, l);
#pragma unroll
        for (int v = 0; v < 16; ++v)
          l[v] = __float_as_uint(j > 0 ? __uint_as_float(l[v]) + x[v] : x[v]);
        tc::st16x4(lcols, l);
        tc::wait_st();
      }
    }

    if (!bad) {
      const bool ok = __all_sync(
          kFull, nblk == 0 || (!*abort_flag && mbar_wait(odone, (nblk - 1) & 1)));
      // sums over this quarter's keys: the thread's two key slots, then the
      // eight threads that share its columns (fixed order)
      float lp[8];
      if (nblk > 0) {
        uint32_t l[16];
        tc::fence_after();
        tc::ld16x4(lcols, l);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            lp[2 * i + e] = __uint_as_float(l[4 * i + e]) + __uint_as_float(l[4 * i + 2 + e]);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) lp[k] = 0.f;
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)
#pragma unroll
        for (int k = 0; k < 8; ++k) lp[k] += __shfl_xor_sync(kFull, lp[k], off);
      if (named_sync_or(1, SMX, !ok)) {
        bad = true;
      } else {
        if (lane < 4) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int e = 0; e < 2; ++e) red[q * 64 + 32 * h + 8 * i + 2 * lane + e] = lp[2 * i + e];
        }
        named_sync(1, SMX);
        if (decider && lane < 16) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int col = 32 * h + 2 * cl + e;
            const float l = ((red[col] + red[64 + col]) + red[128 + col]) + red[192 + col];
            const bool seen = nblk > 0 && (!CAUSAL || l > 0.f);   // some token was visible
            alpha_s[col] = seen ? 1.f / l : 0.f;
            const int64_t li = lse_idx(col);
            if (li >= 0) a.lse_part[li] = seen ? m_ref[col] + log2f(l) : -INFINITY;
          }
        }
        named_sync(1, SMX);
        tc::fence_after();
        // the partial rows are staged as [64 rows][512] fp32 in the K/V stages
        // (idle now: every product is done) and written by bulk copies, one
        // 2 KB row each, instead of 128 scalar stores per thread
        float* ostage = reinterpret_cast<float*>(stages);
        static_assert(R * kMlaDv * 4 <= kMlaTcStages * STAGE, "partial rows fit the stages");
#pragma unroll 1
        for (int t = 0; t < 4; ++t) {
          uint32_t o[32];
          if (nblk > 0) {
            tc::ld32(tbase + lanes + t * R + 32 * h, o);
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = 0u;
          }
          const int dvi = 128 * t + 32 * q + lane;
#pragma unroll
          for (int c = 0; c < 32; ++c)
            ostage[(32 * h + c) * kMlaDv + dvi] = __uint_as_float(o[c]) * alpha_s[32 * h + c];
        }
        fence_proxy_async_smem();
        named_sync(1, SMX);
        {
          const int r = threadIdx.x - kMlaTcLoadWarps * 32;
          if (r < R) {
            const int64_t orow = out_row(r);
            if (orow >= 0)
              bulk_store_s2g(a.o_part + orow * a.dv, smem_addr(ostage + r * kMlaDv), kMlaDv * 4);
            bulk_store_commit_wait_read();
          }
        }
      }
    }
    if (bad && threadIdx.x == kMlaTcLoadWarps * 32) {
      *abort_flag = 1;
      atomicOr(a.status, kStatusTimeout);
    }
  }

  tc::fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc::fence_after();
    tc::dealloc(tbase, TCOLS);
  }
  // As the private-token kernel of a shared-prefix plan (programmatic
  // dependent launch): finish only once the prefix grid has, so the merge,
  // which waits on this grid, sees the prefix partials too. Without a
  // prerequisite grid this returns at once.
  pdl_wait_prerequisites();
}

}  // namespace

bool mla_tc_kernel(int dtype, bool causal, KernelEntry* e) {
  if (causal)
    e->func = dtype == PKVD_FP16 ? reinterpret_cast<const void*>(&mla_tc<__half, true>)
                                 : reinterpret_cast<const void*>(&mla_tc<__nv_bfloat16, true>);
  else
    e->func = dtype == PKVD_FP16 ? reinterpret_cast<const void*>(&mla_tc<__half, false>)
                                 : reinterpret_cast<const void*>(&mla_tc<__nv_bfloat16, false>);
  e->threads = kMlaTcThreads;
  e->smem = kMlaTcSmemBytes;
  e->block_tokens = kMlaTcBlockTokens;
  e->stages = kMlaTcStages;
  return true;
}

}  // namespace pkvd
