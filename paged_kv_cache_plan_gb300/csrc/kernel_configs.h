// Static shapes of the stage-1 kernels, in plain C++ so that the host
// planner can size splits without touching CUDA. The kernels static_assert
// that their shared-memory layouts match these numbers.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define PKVD_HD __host__ __device__
#else
#define PKVD_HD
#endif

namespace pkvd {

// Every K/V row lands in shared memory at a pitch 16 bytes wider than the
// row. Consecutive rows then start in different 16-byte bank groups, so the
// 8 rows an ldmatrix (or a quarter-warp of 128-bit loads) touches hit 8
// distinct groups: the bank-conflict-free pitch rule of the rocm-libraries
// pull 10102 page (Motivation: bank = (addr/4) % banks, pad the pitch so a
// wave's reads spread over all banks), redone for 32 banks x 4 bytes.
constexpr int kRowPad = 16;

// Mbarrier area at the front of dynamic shared memory.
constexpr int kBarrierBytes = 256;

// GQA stage 1: gqa_warps(D) warps per block. Each warp owns
// gqa_stages_per_warp(D) shared-memory stages and issues the copies of its
// own blocks: a warp's copies are issued one after another, so several
// issuing warps keep many copies in flight, and a second stage per warp keeps
// a copy in flight while the warp computes on the other.
// One stage = 16 tokens of K and 16 of V (one page at page size 16), moved
// either as two whole 16-row tiles through TMA tensor maps (128-byte swizzle,
// tiles = true) or as one bulk copy per row into padded rows (tiles = false).
constexpr int kGqaBlockTokens = 16;
constexpr int kTileAlign = 1024;    // swizzled tiles start on 1 KB boundaries
PKVD_HD constexpr int gqa_warps(int) { return 6; }
PKVD_HD constexpr int gqa_stages_per_warp(int D) { return D == 256 ? 1 : 2; }
PKVD_HD constexpr int gqa_threads(int D) { return gqa_warps(D) * 32; }
PKVD_HD constexpr int gqa_stages(int D) { return gqa_warps(D) * gqa_stages_per_warp(D); }
PKVD_HD constexpr int gqa_row_pitch(int D) { return D * 2 + kRowPad; }
PKVD_HD constexpr int gqa_tile_bytes(int D, bool tiles) {
  return tiles ? kGqaBlockTokens * D * 2 : kGqaBlockTokens * gqa_row_pitch(D);
}
PKVD_HD constexpr int gqa_stage_bytes(int D, bool tiles) { return 2 * gqa_tile_bytes(D, tiles); }
// p values and rescale factors each warp publishes per block (FMA variant)
PKVD_HD constexpr int gqa_pbuf_bytes(int D, int G) {
  return gqa_warps(D) * (kGqaBlockTokens * (G < 8 ? 8 : G) + (G < 8 ? 8 : G)) * 4;
}
// the group's query rows, padded like K/V rows (MMA variant: ldmatrix source
// of the Q^T fragments)
PKVD_HD constexpr int gqa_qtile_bytes(int D, int G) {
  return (G < 8 ? 8 : G) * gqa_row_pitch(D);
}
// cross-warp merge area, carved from the (by then idle) stage buffers:
// [W][G] output rows of gqa_merge_row(D) floats (4 floats of padding, so the
// quad lanes of an mma fragment, two heads apart, store to distinct banks),
// then [W][G] maxima, [W][G] sums and [W][G] merge weights
PKVD_HD constexpr int gqa_merge_row(int D) { return D + 4; }
PKVD_HD constexpr int gqa_merge_bytes(int D, int G) {
  return gqa_warps(D) * (G * gqa_merge_row(D) + 3 * G) * 4;
}
// the stage area, large enough to hold the merge area afterwards
PKVD_HD constexpr int gqa_stage_area_bytes(int D, int G, bool tiles) {
  return gqa_stages(D) * gqa_stage_bytes(D, tiles) > gqa_merge_bytes(D, G)
             ? gqa_stages(D) * gqa_stage_bytes(D, tiles)
             : gqa_merge_bytes(D, G);
}
// [align slack][stage area][barriers][p buffers][query tile]
PKVD_HD constexpr int gqa_smem_bytes(int D, int G, bool tiles) {
  return kTileAlign + gqa_stage_area_bytes(D, G, tiles) + kBarrierBytes + gqa_pbuf_bytes(D, G) +
         gqa_qtile_bytes(D, G);
}

// MLA (mma.sync consumer): a block of 16 heads per work item, 4 warps, one
// stage = 16 latent rows of 576 (V = the first 512 of each row) at the padded
// pitch. Warp w scores the 16 keys of a block over dims 144w .. 144w+143 and
// owns output columns 128w .. 128w+127; the four partial score tiles meet in
// a double-buffered reduction area. Sized for two blocks per SM.
constexpr int kMlaWarps = 4;
constexpr int kMlaThreads = kMlaWarps * 32;
constexpr int kMlaBlockTokens = 16;
constexpr int kMlaStages = 5;
constexpr int kMlaHeads = 16;
constexpr int kMlaDk = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaRowPitch = kMlaDk * 2 + kRowPad;                       // 1168 B
constexpr int kMlaStageBytes = kMlaBlockTokens * kMlaRowPitch;           // 18688 B
// partial scores: [2 buffers][4 warps][2 n-tiles][32 lanes] float4
constexpr int kMlaRedBytes = 2 * kMlaWarps * 2 * 32 * 16;                // 8192 B
constexpr int kMlaSmemBytes = kBarrierBytes + kMlaStages * kMlaStageBytes + kMlaRedBytes;

// MLA on the fifth-generation tensor cores (tcgen05): a block of 64 query
// heads per work item, 64-key blocks in two stages. Warps 0-3 copy K/V rows
// (16-byte cp.async chunks written straight into the 128-byte-swizzled
// operand layout), warps 4-11 run the softmax, warp 12 issues the S^T
// products and owns the tensor memory, warp 13 issues the O^T products. Shared memory: [align slack][Q tile][2 stages]
// [P tile][barriers and reduction scratch] = the whole 227 KB of a block.
constexpr int kMlaTcHeads = 64;
constexpr int kMlaTcBlockTokens = 64;
constexpr int kMlaTcStages = 2;
constexpr int kMlaTcLoadWarps = 4;
constexpr int kMlaTcSoftmaxWarps = 8;
constexpr int kMlaTcThreads = (kMlaTcLoadWarps + kMlaTcSoftmaxWarps + 2) * 32;   // 448
constexpr int kMlaTcSlabBytes = kMlaTcBlockTokens * 128;     // 64 rows x 64 columns
constexpr int kMlaTcStageBytes = (kMlaDk / 64) * kMlaTcSlabBytes;               // 73,728
constexpr int kMlaTcQBytes = (kMlaDk / 64) * kMlaTcHeads * 128;                 // 73,728
constexpr int kMlaTcPBytes = kMlaTcHeads * kMlaTcBlockTokens * 2;               // 8,192
constexpr int kMlaTcMiscBytes = 2048;
constexpr int kMlaTcSmemBytes = kTileAlign + kMlaTcQBytes + kMlaTcStages * kMlaTcStageBytes +
                                kMlaTcPBytes + kMlaTcMiscBytes;                  // 232,448
// The tcgen05 kernel rounds P to one 16-bit value (the mma.sync kernel keeps a
// second, low part). AUTO uses it only when every request has at least this
// many tokens, where the rounding errors of P average out far below the
// output tolerance.
constexpr int kMlaTcMinContext = 1024;

// Query tokens per request a plan takes (multi-token decode).
constexpr int kMaxQueryLen = 8;

// Ranks a context-parallel decode may spread one request over.
constexpr int kMaxCpRanks = 1024;

// Stage 2 keeps one float4 sum per warp (8 warps) and float4 column of its
// Dv slice in shared memory.
constexpr int kMaxSplits = 8192;
constexpr int kMergeThreads = 256;
PKVD_HD constexpr int stage2_smem_bytes(int dv_slice) {
  return (kMergeThreads / 32) * (dv_slice / 4) * 16;
}
// With at most kMergeColMaxSplits splits per request the merge runs one
// thread per float4 column instead (no shared memory), in blocks of
// merge_col_threads(Dv slice) threads.
constexpr int kMergeColMaxSplits = 8;
PKVD_HD constexpr int merge_col_threads(int dv_slice) {
  return ((dv_slice / 4 + 31) / 32) * 32 > 128 ? 128
         : ((dv_slice / 4 + 31) / 32) * 32 < 32 ? 32
                                                : ((dv_slice / 4 + 31) / 32) * 32;
}
// Threads per merge block for a plan whose requests have at most max_splits
// splits, with Dv slices of dv_slice columns.
PKVD_HD constexpr int merge_threads(int max_splits, int dv_slice) {
  return max_splits <= kMergeColMaxSplits ? merge_col_threads(dv_slice) : kMergeThreads;
}

// Usable shared memory per SM and per block on sm_103a.
constexpr int kSmemPerSm = 233472;     // 228 KB
constexpr int kSmemPerBlockMax = 232448;  // 227 KB
constexpr int kSmemReservedPerBlock = 1024;

}  // namespace pkvd
