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

// Producer warp + consumer warps per stage-1 block.
constexpr int kConsumerWarps = 4;
constexpr int kStage1Threads = (kConsumerWarps + 1) * 32;

// Every K/V row lands in shared memory at a pitch 16 bytes wider than the
// row. Consecutive rows then start in different 16-byte bank groups, so the
// 8 rows an ldmatrix (or a quarter-warp of 128-bit loads) touches hit 8
// distinct groups: the bank-conflict-free pitch rule of the rocm-libraries
// pull 10102 page (Motivation: bank = (addr/4) % banks, pad the pitch so a
// wave's reads spread over all banks), redone for 32 banks x 4 bytes.
constexpr int kRowPad = 16;

// Mbarrier area at the front of dynamic shared memory.
constexpr int kBarrierBytes = 256;

// GQA: one stage = 16 tokens of K and 16 of V (one page at page size 16).
constexpr int kGqaBlockTokens = 16;
PKVD_HD constexpr int gqa_stages(int D) { return D == 256 ? 6 : 8; }
PKVD_HD constexpr int gqa_row_pitch(int D) { return D * 2 + kRowPad; }
PKVD_HD constexpr int gqa_stage_bytes(int D) { return 2 * kGqaBlockTokens * gqa_row_pitch(D); }
// p values and rescale factors each consumer warp publishes per block
PKVD_HD constexpr int gqa_pbuf_bytes(int G) {
  return kConsumerWarps * (kGqaBlockTokens * G + G) * 4;
}
PKVD_HD constexpr int gqa_smem_bytes(int D, int G) {
  return kBarrierBytes + gqa_stages(D) * gqa_stage_bytes(D) + gqa_pbuf_bytes(G < 8 ? 8 : G);
}
// cross-warp merge area, carved from the (by then idle) stage buffers
PKVD_HD constexpr int gqa_merge_bytes(int D, int G) {
  return kConsumerWarps * (G * D + 2 * G) * 4;
}

// MLA: one stage = 64 latent rows of 576 (V = the first 512 of each row),
// a block of 16 heads per work item.
constexpr int kMlaBlockTokens = 64;
constexpr int kMlaStages = 2;
constexpr int kMlaHeads = 16;
constexpr int kMlaDk = 576;
constexpr int kMlaDv = 512;
constexpr int kMlaRowPitch = kMlaDk * 2 + kRowPad;                       // 1168 B
constexpr int kMlaStageBytes = kMlaBlockTokens * kMlaRowPitch;           // 74752 B
constexpr int kMlaQBytes = kMlaHeads * kMlaRowPitch;                     // 18688 B
constexpr int kMlaPPitch = (kMlaBlockTokens + 8) * 2;                    // 144 B
constexpr int kMlaPBytes = 2 * kMlaHeads * kMlaPPitch;   // P high + low parts, 4608 B
constexpr int kMlaRedBytes = 2 * kConsumerWarps * kMlaHeads * 4;         // 512 B
constexpr int kMlaSmemBytes = kBarrierBytes + kMlaStages * kMlaStageBytes + kMlaQBytes +
                              kMlaPBytes + kMlaRedBytes;

// Stage 2 keeps one weight per split in shared memory.
constexpr int kMaxSplits = 8192;

// Usable shared memory per SM and per block on sm_103a.
constexpr int kSmemPerSm = 233472;     // 228 KB
constexpr int kSmemPerBlockMax = 232448;  // 227 KB
constexpr int kSmemReservedPerBlock = 1024;

}  // namespace pkvd
