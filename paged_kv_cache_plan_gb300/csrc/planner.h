// Host split planner: shape checks, variant choice, split sizes, work-list
// order and merge tiling. Plain C++; no CUDA call anywhere in it.
#pragma once

#include <cstdint>
#include <vector>

#include "../../include/pkvd.h"

namespace pkvd {

struct PlanLayout {
  pkvd_plan_desc desc{};             // normalised (defaults filled in)
  pkvd_plan_info info{};
  std::vector<int32_t> seq_lens;
  std::vector<int32_t> splits;       // S_b
  std::vector<int32_t> split_base;   // B + 1 prefix sums of S_b
  std::vector<pkvd_work_item> items; // stage-1 grid order
  // Shared-prefix plans: grouped prefix items (tensor-memory MLA kernel),
  // launched before `items`; empty otherwise.
  std::vector<pkvd_work_item> prefix_items;
};

// Static per-variant numbers the planner needs (block tokens, stages,
// threads, shared memory); false when the variant has no kernel for the shape.
struct VariantShape {
  int block_tokens;
  int stages;
  int threads;
  int smem;
};
bool variant_shape(int variant, int head_dim, int group, bool tiles, VariantShape* out);

// Whether the GQA kernels can move K/V as whole 16-row page tiles: the page
// size is a multiple of 16 and every split starts on a 16-token boundary.
bool plan_uses_tiles(const pkvd_plan_desc& normalised, const int32_t* seq_lens);

// Validate and normalise `in`; resolve the family and (if AUTO) the variant.
int normalise_desc(const pkvd_plan_desc& in, const int32_t* seq_lens, pkvd_plan_desc* out,
                   int* family);

// Full planning with desc->num_sms and desc->ctas_per_sm already set (> 0).
int plan_layout(const pkvd_plan_desc& desc, const int32_t* seq_lens, PlanLayout* out);

// The normalised description of a shared-prefix plan's per-request items:
// the full lengths fix the page-table width, the private lengths (what is
// left after the grouped prefixes) resolve the variant.
int prefix_private_desc(const pkvd_plan_desc& in, const int32_t* seq_lens,
                        const int32_t* prefix_group, const int32_t* prefix_len,
                        pkvd_plan_desc* out, int* family);

// Shared-prefix planning (see decode_plan_prefix): the per-request items of
// the private tokens, planned as plan_layout does, plus grouped prefix items
// for the tensor-memory MLA kernel (one resident block per SM).
int plan_layout_prefix(const pkvd_plan_desc& desc, const int32_t* seq_lens,
                       const int32_t* prefix_group, const int32_t* prefix_len, PlanLayout* out);

// Context parallel (one request's tokens spread over `world` ranks, each
// GPU holding the whole page table): rank `rank` takes of request b the
// tokens [begin[b], begin[b] + len[b]), ceil(ceil(L_b / world) / ps) pages
// per rank from the start (trailing ranks may be empty).
int cp_ranges(int world, int rank, int batch, int page_size, const int32_t* seq_lens,
              int32_t* begin, int32_t* len);

// The normalised description of a rank's plan (the full lengths fix the
// page-table width, the rank's lengths resolve the variant; one query token).
int cp_shard_desc(const pkvd_plan_desc& in, const int32_t* seq_lens, int world, int rank,
                  pkvd_plan_desc* out, int* family);

// A rank's plan: plan_layout on the rank's lengths with every item moved to
// the absolute token positions of its range.
int plan_layout_cp(const pkvd_plan_desc& in, const int32_t* seq_lens, int world, int rank,
                   PlanLayout* out);

}  // namespace pkvd
