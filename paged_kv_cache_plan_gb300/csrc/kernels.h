// Kernel arguments and the per-variant kernel lookup shared by the host
// launcher and the kernel translation units.
#pragma once

#include <cuda.h>   // CUtensorMap (type only; the driver is reached through the runtime)
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/pkvd.h"

namespace pkvd {

// Arguments of every stage-1 kernel (one work item per block).
struct Stage1Args {
  const void* q;                 // [B, Hq, D] 16-bit
  const void* k;                 // K pool, rows of k_pitch elements
  const void* v;                 // V pool, rows of v_pitch elements
  const int32_t* page_table;     // [B, pt_stride]
  const pkvd_work_item* items;   // [grid]
  const int32_t* split_base;     // [B + 1] first partial row of each request (grouped items)
  float* o_part;                 // [rows, Hq, Dv] normalised partial outputs
  float* lse_part;               // [Hq, lse_stride] partial log2-sum-exp2 (log2 domain),
                                 // head-major: one head's splits are consecutive
  int64_t lse_stride;            // partial rows of the plan
  int32_t* status;               // device status word (kStatus* bits)
  int64_t pt_stride;             // entries per page_table row
  int64_t k_pitch;               // elements between K rows
  int64_t v_pitch;               // elements between V rows
  int64_t num_pool_pages;        // pages in the pools (checks only)
  int32_t heads;                 // Hq
  int32_t kv_heads;              // Hkv
  int32_t page_size;             // tokens per page
  int32_t dv;                    // Dv
  int32_t q_len;                 // query tokens per request: q is [B, q_len, Hq, D] and
                                 // the partials hold q_len * Hq rows per split
  float scale_log2;              // scale * log2(e): scores go straight to exp2
  int32_t checks;                // 1 = bounds-check page ids
};

// Arguments of the merge kernel (one block per (request, head, Dv slice)).
struct Stage2Args {
  const float* o_part;
  const float* lse_part;         // [q_len * Hq, lse_stride]
  int64_t lse_stride;
  const int32_t* split_base;     // [B + 1] first partial row of each request
  float* out;                    // [B, q_len * Hq, Dv]
  float* lse;                    // [B, q_len * Hq] natural log
  int32_t heads;                 // q_len * Hq (query token, head) rows
  int32_t dv;
  int32_t tiles;                 // Dv slices (gridDim.y)
};

// Tensor maps of the K and V pools for the whole-page tile path (unused,
// zero, for kernels that copy rows).
struct KvTensorMaps {
  CUtensorMap k;
  CUtensorMap v;
};

struct KernelEntry {
  const void* func = nullptr;    // __global__ symbol: (Stage1Args, KvTensorMaps) for stage 1,
                                 // (Stage2Args) for the merge
  int threads = 0;
  int smem = 0;                  // dynamic shared memory bytes
  int block_tokens = 0;
  int stages = 0;
  bool tiles = false;            // K/V move as TMA page tiles (needs tensor maps)
};

// Lookups; false when the combination has no kernel.
bool gqa_fma_kernel(int dtype, int head_dim, int group, bool tiles, KernelEntry* e);
// cols = q_len x group; causal: several query tokens per request (a cut per
// (query token, head) row); the one-token kernels have none.
bool gqa_mma_kernel(int dtype, int head_dim, int cols, bool tiles, bool causal, KernelEntry* e);
bool mla_mma_kernel(int dtype, bool causal, KernelEntry* e);
bool mla_tc_kernel(int dtype, bool causal, KernelEntry* e);
// The merge kernel of a plan (threads and shared memory filled in): one
// thread per column when no request has more than kMergeColMaxSplits
// splits; otherwise split-parallel, with deep prefetch when the merge grid
// (batch x rows x Dv slices blocks, rows = q_len x heads) is at most two
// blocks per SM.
bool stage2_kernel(const pkvd_plan_info& info, int batch, int heads, int dv, KernelEntry* e);

// Merge of n context-parallel ranks' normalised rows (o [n][rows][dv], lse
// [n][rows] natural log) into out [rows][dv], lse [rows]; dv a multiple of 4
// up to 512. Returns a pkvd_status.
int launch_merge_ranks(int n, int64_t rows, int dv, const float* o, const float* lse_in,
                       float* out, float* lse, cudaStream_t stream);

// Stage-1 kernel for a normalised plan description (variant resolved).
bool stage1_kernel(const pkvd_plan_desc& d, bool tiles, KernelEntry* e);

// A tiled tensor map with 128-byte swizzle over a 16-bit tensor: rank 2..5,
// dims innermost first, strides[i] = bytes between steps of dim i + 1, box
// the copied tile; out-of-range elements read as zero. Returns a pkvd_status.
int encode_tiled_map(int dtype, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box, CUtensorMap* out);

// Encode the K and V tensor maps of the page-tile path for the given pool
// pointers: {64 columns, pool rows, D/64 column blocks}, box {64, 16, D/64},
// 128-byte swizzle. Returns a pkvd_status.
int encode_kv_maps(const pkvd_plan_desc& d, const void* k, const void* v, KvTensorMaps* out);

}  // namespace pkvd
