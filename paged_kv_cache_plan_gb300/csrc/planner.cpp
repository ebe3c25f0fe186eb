// Split planner (host). See planner.h.
//
// Split policy. The aiter pull 4758 page (Motivation) gives each request
// about 256/batch splits on a 256-CU part, trading split count against how
// far each stage-1 program walks. Here the same trade is made against this
// GPU's stage-1 capacity: a uniform chunk of C tokens (a multiple of the
// kernel's block) is the smallest one for which the work items
//     sum_b units * ceil(L_b / C)
// fit in one wave of num_sms * ctas_per_sm resident blocks; request b then
// has S_b = ceil(L_b / C) splits. A forced split count S gives request b the
// chunk ceil(L_b / S) instead (so min(S, L_b) splits).
//
// Grid order (the same page, Technical Details 2): split-major puts all
// requests' items of one split next to each other (L2 reuse under prefix
// sharing); it is a pure relabelling, so results are bit-identical.
//
// Merge tiling (the same page, Technical Details 3): slice Dv only while
// the B * q_len * Hq merge blocks would leave SMs idle, up to 8 ways, and only into
// slices that divide Dv evenly.
#include "planner.h"

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "kernel_configs.h"

namespace pkvd {

namespace {

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

bool variant_shape(int variant, int head_dim, int group, bool tiles, VariantShape* out) {
  switch (variant) {
    case PKVD_VARIANT_GQA_FMA:
      if ((head_dim != 128 && head_dim != 256) || !is_pow2(group) || group > 8) return false;
      *out = {kGqaBlockTokens, gqa_stages(head_dim), gqa_threads(head_dim),
              gqa_smem_bytes(head_dim, group, tiles)};
      return true;
    case PKVD_VARIANT_GQA_MMA:
      if ((head_dim != 128 && head_dim != 256) || group < 1 || group > 16) return false;
      *out = {kGqaBlockTokens, gqa_stages(head_dim), gqa_threads(head_dim),
              gqa_smem_bytes(head_dim, group > 8 ? 16 : 8, tiles)};
      return true;
    case PKVD_VARIANT_MLA_MMA:
      if (head_dim != kMlaDk || tiles) return false;
      *out = {kMlaBlockTokens, kMlaStages, kMlaThreads, kMlaSmemBytes};
      return true;
    case PKVD_VARIANT_MLA_TC:
      if (head_dim != kMlaDk || tiles) return false;
      *out = {kMlaTcBlockTokens, kMlaTcStages, kMlaTcThreads, kMlaTcSmemBytes};
      return true;
    default:
      return false;
  }
}

bool plan_uses_tiles(const pkvd_plan_desc& d, const int32_t* seq_lens) {
  if (d.head_dim == kMlaDk || d.page_size % kGqaBlockTokens != 0) return false;
  if (d.splits > 0)
    for (int b = 0; b < d.batch; ++b) {
      const int64_t chunk = std::max<int64_t>(1, ceil_div(seq_lens[b], d.splits));
      if (ceil_div(seq_lens[b], chunk) > 1 && chunk % kGqaBlockTokens != 0) return false;
    }
  return true;   // planner chunks are multiples of the 16-token block
}

int normalise_desc(const pkvd_plan_desc& in, const int32_t* seq_lens, pkvd_plan_desc* out,
                   int* family) {
  pkvd_plan_desc d = in;
  if (!seq_lens && d.batch > 0) return PKVD_EINVAL;
  if (d.batch < 1 || d.heads < 1 || d.kv_heads < 1 || d.head_dim < 1 || d.page_size < 1)
    return PKVD_EINVAL;
  if (d.head_dim_v < 0 || d.splits < 0 || d.num_sms < 0 || d.ctas_per_sm < 0 ||
      d.min_chunk < 0 || d.max_pages_per_seq < 0 || d.num_pool_pages < 0 ||
      d.k_row_pitch < 0 || d.v_row_pitch < 0)
    return PKVD_EINVAL;
  if (d.reserved2 != 0 || d.q_len < 0) return PKVD_EINVAL;
  if (d.q_len == 0) d.q_len = 1;
  if (d.q_len > kMaxQueryLen) return PKVD_EUNSUPPORTED;
  if (d.dtype != PKVD_BF16 && d.dtype != PKVD_FP16) return PKVD_EINVAL;
  if (d.grid_order < PKVD_ORDER_AUTO || d.grid_order > PKVD_ORDER_REQUEST_MAJOR)
    return PKVD_EINVAL;
  if (d.stage2_tiles != 0 && d.stage2_tiles != 1 && d.stage2_tiles != 2 &&
      d.stage2_tiles != 4 && d.stage2_tiles != 8)
    return PKVD_EINVAL;
  if (d.checks != 0 && d.checks != 1) return PKVD_EINVAL;
  if (d.checks && d.num_pool_pages == 0) return PKVD_EINVAL;
  if (!(std::isfinite(d.scale)) || d.scale < 0.f) return PKVD_EINVAL;
  if (d.heads % d.kv_heads != 0) return PKVD_EUNSUPPORTED;

  const bool mla = d.head_dim == kMlaDk;
  if (mla) {
    if (d.head_dim_v == 0) d.head_dim_v = kMlaDv;
    if (d.head_dim_v != kMlaDv || d.kv_heads != 1 || d.heads % kMlaHeads != 0)
      return PKVD_EUNSUPPORTED;
    if (d.k_row_pitch == 0) d.k_row_pitch = kMlaDk;
    if (d.v_row_pitch == 0) d.v_row_pitch = kMlaDk;
    if (d.k_row_pitch != d.v_row_pitch) return PKVD_EUNSUPPORTED;   // V aliases K rows
  } else {
    if (d.head_dim != 128 && d.head_dim != 256) return PKVD_EUNSUPPORTED;
    if (d.head_dim_v == 0) d.head_dim_v = d.head_dim;
    if (d.head_dim_v != d.head_dim) return PKVD_EUNSUPPORTED;
    if (d.k_row_pitch == 0) d.k_row_pitch = d.head_dim;
    if (d.v_row_pitch == 0) d.v_row_pitch = d.head_dim_v;
  }
  if (d.k_row_pitch < d.head_dim || d.v_row_pitch < d.head_dim_v) return PKVD_EINVAL;
  if ((d.k_row_pitch * 2) % 16 != 0 || (d.v_row_pitch * 2) % 16 != 0) return PKVD_EINVAL;
  if (d.scale == 0.f) d.scale = 1.0f / std::sqrt(static_cast<float>(d.head_dim));

  int64_t max_pages = 0;
  for (int b = 0; b < d.batch; ++b) {
    if (seq_lens[b] < 0) return PKVD_EINVAL;
    if (seq_lens[b] > 0 && seq_lens[b] < d.q_len) return PKVD_EINVAL;   // queries are cached tokens
    max_pages = std::max<int64_t>(max_pages, ceil_div(seq_lens[b], d.page_size));
  }
  if (d.max_pages_per_seq == 0) d.max_pages_per_seq = std::max<int64_t>(1, max_pages);
  if (d.max_pages_per_seq < max_pages) return PKVD_EINVAL;

  // (query token, head) rows: a unit of the MLA kernels takes 16 or 64 of
  // them; a GQA unit (one KV head) takes the q_len x group rows of its heads
  const int group = d.heads / d.kv_heads;
  const int vheads = d.q_len * d.heads;
  if (mla) {
    // The tensor-memory kernel rounds P to one 16-bit value; it is only
    // taken (and only accepted) when every non-empty request has at least
    // kMlaTcMinContext tokens, where that rounding averages out far below
    // the output tolerance. Shorter contexts run on the mma.sync kernel,
    // which keeps a second, low part of P. Row counts that are not a
    // multiple of 64 take it too (its last unit zero-padded): with one
    // product per 64 keys the padding costs little, and it measured faster
    // than the 16-row mma.sync kernel at 16 heads.
    int64_t min_len = INT64_MAX;
    for (int b = 0; b < d.batch; ++b)
      if (seq_lens[b] > 0) min_len = std::min<int64_t>(min_len, seq_lens[b]);
    const bool long_enough = min_len >= kMlaTcMinContext;
    if (d.variant == PKVD_VARIANT_AUTO)
      d.variant = long_enough ? PKVD_VARIANT_MLA_TC : PKVD_VARIANT_MLA_MMA;
    if (d.variant != PKVD_VARIANT_MLA_MMA && d.variant != PKVD_VARIANT_MLA_TC)
      return PKVD_EUNSUPPORTED;
    if (d.variant == PKVD_VARIANT_MLA_TC && !long_enough) return PKVD_EUNSUPPORTED;
  } else {
    // The mma consumer is faster than the fp32 FMA consumer on every group
    // size measured on GB300 (the FMA path is issue-bound: about five
    // instructions per K/V byte pair at group 8, d 256), so it is the default.
    if (d.variant == PKVD_VARIANT_AUTO) d.variant = PKVD_VARIANT_GQA_MMA;
    if (d.variant != PKVD_VARIANT_GQA_FMA && d.variant != PKVD_VARIANT_GQA_MMA)
      return PKVD_EUNSUPPORTED;
    if (d.variant == PKVD_VARIANT_GQA_FMA && d.q_len != 1) return PKVD_EUNSUPPORTED;
  }
  VariantShape vs;
  if (!variant_shape(d.variant, d.head_dim, d.q_len * group, false, &vs))
    return PKVD_EUNSUPPORTED;
  *out = d;
  *family = mla ? PKVD_FAMILY_MLA : PKVD_FAMILY_GQA;
  return PKVD_OK;
}

int plan_layout(const pkvd_plan_desc& in, const int32_t* seq_lens, PlanLayout* out) {
  pkvd_plan_desc d;
  int family = 0;
  int rc = normalise_desc(in, seq_lens, &d, &family);
  if (rc != PKVD_OK) return rc;
  if (d.num_sms < 1 || d.ctas_per_sm < 1) return PKVD_EINVAL;

  const int B = d.batch;
  const int group = d.heads / d.kv_heads;
  const int vheads = d.q_len * d.heads;     // merge rows per request
  const bool kv_tiles = plan_uses_tiles(d, seq_lens);
  VariantShape vs;
  variant_shape(d.variant, d.head_dim, d.q_len * group, kv_tiles, &vs);
  const int blk = vs.block_tokens;

  PlanLayout& P = *out;
  P.desc = d;
  P.seq_lens.assign(seq_lens, seq_lens + B);
  P.splits.assign(B, 0);
  P.split_base.assign(B + 1, 0);
  P.items.clear();

  pkvd_plan_info& I = P.info;
  I = pkvd_plan_info{};
  I.family = family;
  I.variant = d.variant;
  I.num_sms = d.num_sms;
  I.ctas_per_sm = d.ctas_per_sm;
  if (family == PKVD_FAMILY_MLA) {
    I.heads_per_unit = d.variant == PKVD_VARIANT_MLA_TC ? kMlaTcHeads : kMlaHeads;
    // the tensor-memory kernel zero-pads a request's last 64-row unit
    I.units_per_request = static_cast<int>(ceil_div(vheads, I.heads_per_unit));
  } else {
    I.heads_per_unit = d.q_len * group;
    I.units_per_request = d.kv_heads;
  }
  I.block_tokens = blk;
  I.pipeline_stages = vs.stages;
  I.stage1_smem_bytes = vs.smem;
  I.stage1_threads = vs.threads;
  I.kv_tiles = kv_tiles ? 1 : 0;
  const int units = I.units_per_request;

  // --- split sizes
  std::vector<int64_t> chunk(B, 1);
  int64_t maxL = 0;
  for (int b = 0; b < B; ++b) maxL = std::max<int64_t>(maxL, P.seq_lens[b]);
  if (d.splits > 0) {
    for (int b = 0; b < B; ++b) {
      const int64_t L = P.seq_lens[b];
      chunk[b] = std::max<int64_t>(1, ceil_div(L, d.splits));
      P.splits[b] = L == 0 ? 0 : static_cast<int32_t>(ceil_div(L, chunk[b]));
    }
    bool uniform = true;
    for (int b = 1; b < B; ++b) uniform = uniform && chunk[b] == chunk[0];
    I.chunk = uniform ? chunk[0] : 0;
  } else {
    const int64_t target = static_cast<int64_t>(d.num_sms) * d.ctas_per_sm;
    const int64_t min_chunk =
        std::max<int64_t>(blk, ceil_div(d.min_chunk > 0 ? d.min_chunk : 2 * blk, blk) * blk);
    auto items_for = [&](int64_t C) {
      int64_t n = 0;
      for (int b = 0; b < B; ++b) n += ceil_div(P.seq_lens[b], C);
      return n * units;
    };
    // smallest multiple of blk (>= min_chunk) whose items fit one wave,
    // else one split per request
    const int64_t hi_c = std::max<int64_t>(min_chunk, ceil_div(std::max<int64_t>(maxL, 1), blk) * blk);
    int64_t C = hi_c;
    if (d.variant == PKVD_VARIANT_MLA_TC) {
      // One resident block per SM and long items: choose the uniform split
      // count that minimises waves x (tokens per item + a pipeline fill of
      // two blocks), so that a last, partly filled wave costs little.
      int64_t best = -1;
      for (int64_t S = 1; S <= 4 * target; ++S) {
        const int64_t c = std::max<int64_t>(min_chunk, ceil_div(ceil_div(std::max<int64_t>(maxL, 1), S), blk) * blk);
        const int64_t cost = ceil_div(items_for(c), target) * (c + 2 * blk);
        if (best < 0 || cost < best) {
          best = cost;
          C = c;
        }
      }
    } else if (items_for(hi_c) <= target) {
      int64_t lo = ceil_div(min_chunk, blk), hi = hi_c / blk;   // in blocks
      while (lo < hi) {
        const int64_t mid = (lo + hi) / 2;
        if (items_for(mid * blk) <= target) hi = mid; else lo = mid + 1;
      }
      C = lo * blk;
    }
    // the merge keeps one weight per split in shared memory
    while (ceil_div(maxL, C) > kMaxSplits) C += blk;
    for (int b = 0; b < B; ++b) {
      chunk[b] = C;
      P.splits[b] = static_cast<int32_t>(ceil_div(P.seq_lens[b], C));
    }
    I.chunk = C;
  }
  int max_s = 0;
  for (int b = 0; b < B; ++b) {
    if (P.splits[b] > kMaxSplits) return PKVD_EUNSUPPORTED;
    P.split_base[b + 1] = P.split_base[b] + P.splits[b];
    max_s = std::max(max_s, P.splits[b]);
  }
  I.num_partial_rows = P.split_base[B];
  I.max_splits = max_s;

  // --- work list
  int order = d.grid_order;
  if (order == PKVD_ORDER_AUTO) order = B > 1 ? PKVD_ORDER_SPLIT_MAJOR : PKVD_ORDER_REQUEST_MAJOR;
  I.grid_order = order;
  auto push = [&](int b, int u, int s) {
    pkvd_work_item w{};
    w.request = b;
    w.unit = u;
    w.split = s;
    w.partial_row = P.split_base[b] + s;
    w.tok_begin = static_cast<int32_t>(s * chunk[b]);
    w.tok_end = static_cast<int32_t>(std::min<int64_t>(P.seq_lens[b], (s + 1) * chunk[b]));
    w.query_pos = P.seq_lens[b] - d.q_len;
    P.items.push_back(w);
  };
  if (order == PKVD_ORDER_SPLIT_MAJOR) {
    for (int s = 0; s < max_s; ++s)
      for (int b = 0; b < B; ++b)
        if (s < P.splits[b])
          for (int u = 0; u < units; ++u) push(b, u, s);
  } else {
    for (int b = 0; b < B; ++b)
      for (int u = 0; u < units; ++u)
        for (int s = 0; s < P.splits[b]; ++s) push(b, u, s);
  }
  I.num_items = static_cast<int32_t>(P.items.size());

  // --- merge tiling
  const int dv = d.head_dim_v;
  int tiles = d.stage2_tiles;
  const int64_t base = static_cast<int64_t>(B) * vheads;
  if (tiles == 0) {
    tiles = 1;
    while (tiles < 8 && base * tiles * 2 <= d.num_sms && dv % (tiles * 2 * 32) == 0) tiles *= 2;
  } else if (dv % (tiles * 4) != 0) {
    return PKVD_EUNSUPPORTED;
  }
  I.stage2_tiles = tiles;
  I.stage2_threads = merge_threads(max_s, dv / tiles);

  // --- workspace: items, split table, partial outputs and lse, status word
  auto al = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t rows = I.num_partial_rows;
  I.workspace_bytes = al(static_cast<int64_t>(std::max<size_t>(P.items.size(), 1)) *
                         static_cast<int64_t>(sizeof(pkvd_work_item))) +
                      al(static_cast<int64_t>(B + 1) * 4) +
                      al(std::max<int64_t>(rows, 1) * vheads * dv * 4) +
                      al(std::max<int64_t>(rows, 1) * vheads * 4) + al(16);
  return PKVD_OK;
}

namespace {

struct Group {
  int first, count;
  int64_t len;
};

// Checks the sharing description and collects the groups that get grouped
// prefix items: runs of consecutive requests with one group id and one
// prefix length. A group whose prefix is shorter than kMlaTcMinContext is
// dropped (its members read the prefix as private tokens): the grouped
// items run on the tensor-memory kernel, whose one-part P needs long items.
// plen[b] = the shared tokens request b skips in its private items.
int prefix_groups(const pkvd_plan_desc& in, const int32_t* seq_lens,
                  const int32_t* prefix_group, const int32_t* prefix_len,
                  std::vector<Group>* groups, std::vector<int32_t>* plen) {
  if (!prefix_group || !prefix_len || !seq_lens || in.batch < 1) return PKVD_EINVAL;
  const int B = in.batch;
  if (in.head_dim != kMlaDk) return PKVD_EUNSUPPORTED;
  if (in.heads < 1 || kMlaTcHeads % in.heads != 0 || in.heads % kMlaHeads != 0)
    return PKVD_EUNSUPPORTED;
  groups->clear();
  plen->assign(B, 0);
  std::vector<int> ids;   // group id of every group seen, kept or dropped
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0) return PKVD_EINVAL;
    const int g = prefix_group[b];
    if (g < 0) continue;
    if (prefix_len[b] < 1 || prefix_len[b] > seq_lens[b]) return PKVD_EINVAL;
    if (b > 0 && prefix_group[b - 1] == g) {
      if (prefix_len[b] != prefix_len[b - 1]) return PKVD_EINVAL;
      if (!groups->empty() && groups->back().first + groups->back().count == b &&
          prefix_group[groups->back().first] == g)
        ++groups->back().count;
    } else {
      for (int o : ids)
        if (o == g) return PKVD_EINVAL;   // members not consecutive
      ids.push_back(g);
      if (prefix_len[b] >= kMlaTcMinContext) groups->push_back({b, 1, prefix_len[b]});
    }
  }
  for (const Group& g : *groups)
    for (int m = 0; m < g.count; ++m) (*plen)[g.first + m] = static_cast<int32_t>(g.len);
  return PKVD_OK;
}

}  // namespace

int prefix_private_desc(const pkvd_plan_desc& in, const int32_t* seq_lens,
                        const int32_t* prefix_group, const int32_t* prefix_len,
                        pkvd_plan_desc* out, int* family) {
  std::vector<Group> groups;
  std::vector<int32_t> plen;
  int rc = prefix_groups(in, seq_lens, prefix_group, prefix_len, &groups, &plen);
  if (rc != PKVD_OK) return rc;
  // normalise on the full lengths (page-table width, scale, pitches), then
  // resolve the variant again on the private lengths
  pkvd_plan_desc nd;
  rc = normalise_desc(in, seq_lens, &nd, family);
  if (rc != PKVD_OK) return rc;
  if (nd.q_len != 1) return PKVD_EUNSUPPORTED;   // one query token per shared-prefix request
  nd.variant = in.variant;
  std::vector<int32_t> rest(in.batch);
  for (int b = 0; b < in.batch; ++b) rest[b] = seq_lens[b] - plen[b];
  return normalise_desc(nd, rest.data(), out, family);
}

int plan_layout_prefix(const pkvd_plan_desc& in, const int32_t* seq_lens,
                       const int32_t* prefix_group, const int32_t* prefix_len,
                       PlanLayout* out) {
  std::vector<Group> groups;
  std::vector<int32_t> plen;
  int rc = prefix_groups(in, seq_lens, prefix_group, prefix_len, &groups, &plen);
  if (rc != PKVD_OK) return rc;
  const int B = in.batch;
  const int per_unit = kMlaTcHeads / in.heads;   // requests whose heads fill 64 rows
  pkvd_plan_desc nd;
  int family = 0;
  rc = prefix_private_desc(in, seq_lens, prefix_group, prefix_len, &nd, &family);
  if (rc != PKVD_OK) return rc;
  nd.num_sms = in.num_sms;
  nd.ctas_per_sm = in.ctas_per_sm;

  // the private tokens: an ordinary plan on the suffix lengths
  std::vector<int32_t> rest(B);
  for (int b = 0; b < B; ++b) rest[b] = seq_lens[b] - plen[b];
  rc = plan_layout(nd, rest.data(), out);
  if (rc != PKVD_OK) return rc;
  PlanLayout& P = *out;
  P.seq_lens.assign(seq_lens, seq_lens + B);

  // prefix splits: one chunk for every group, chosen like the tensor-memory
  // kernel's own splits (one resident block per SM)
  constexpr int blk = kMlaTcBlockTokens;
  const int64_t target = P.desc.num_sms;
  auto items_for = [&](int64_t C) {
    int64_t n = 0;
    for (const Group& g : groups) n += ((g.count + per_unit - 1) / per_unit) * ceil_div(g.len, C);
    return n;
  };
  int64_t maxp = 0;
  for (const Group& g : groups) maxp = std::max(maxp, g.len);
  int64_t Cp = std::max<int64_t>(blk, maxp);
  if (!groups.empty()) {
    int64_t best = -1;
    for (int64_t S = 1; S <= 256; ++S) {
      // no prefix split shorter than kMlaTcMinContext (only a prefix's last
      // split can be, and its weight in the merge is small)
      const int64_t c = std::max<int64_t>(ceil_div(kMlaTcMinContext, blk) * blk,
                                          ceil_div(ceil_div(maxp, S), blk) * blk);
      const int64_t cost = ceil_div(items_for(c), target) * (c + 2 * blk);
      if (best < 0 || cost < best) {
        best = cost;
        Cp = c;
      }
    }
  }
  std::vector<int32_t> sp(B, 0);   // prefix splits of each request
  for (const Group& g : groups)
    for (int m = 0; m < g.count; ++m) sp[g.first + m] = static_cast<int32_t>(ceil_div(g.len, Cp));

  // partial rows of request b: its prefix splits, then its private splits
  std::vector<int32_t> base(B + 1, 0);
  int max_s = 0;
  for (int b = 0; b < B; ++b) {
    const int total = sp[b] + P.splits[b];
    if (total > kMaxSplits) return PKVD_EUNSUPPORTED;
    base[b + 1] = base[b] + total;
    max_s = std::max(max_s, total);
  }
  for (pkvd_work_item& w : P.items) {
    w.partial_row = base[w.request] + sp[w.request] + w.split;
    w.tok_begin += plen[w.request];
    w.tok_end += plen[w.request];
    w.query_pos += plen[w.request];
  }
  for (int b = 0; b < B; ++b) P.splits[b] = sp[b] + P.splits[b];
  P.split_base = base;

  // grouped prefix items, split-major so the units of one group run together
  P.prefix_items.clear();
  int64_t max_sp = 0;
  for (const Group& g : groups) max_sp = std::max(max_sp, ceil_div(g.len, Cp));
  for (int64_t s = 0; s < max_sp; ++s)
    for (const Group& g : groups) {
      if (s * Cp >= g.len) continue;
      for (int u = 0; u * per_unit < g.count; ++u) {
        pkvd_work_item w{};
        w.request = g.first + u * per_unit;
        w.unit = std::min(per_unit, g.count - u * per_unit);
        w.split = static_cast<int32_t>(s);
        w.partial_row = -1;
        w.tok_begin = static_cast<int32_t>(s * Cp);
        w.tok_end = static_cast<int32_t>(std::min<int64_t>(g.len, (s + 1) * Cp));
        w.query_pos = static_cast<int32_t>(g.len - 1);   // every shared token is visible
        w.grouped = 1;
        P.prefix_items.push_back(w);
      }
    }

  pkvd_plan_info& I = P.info;
  I.num_partial_rows = base[B];
  I.max_splits = max_s;
  I.stage2_threads = merge_threads(max_s, P.desc.head_dim_v / I.stage2_tiles);
  I.num_prefix_items = static_cast<int32_t>(P.prefix_items.size());
  I.chunk = 0;
  auto al = [](int64_t x) { return (x + 255) / 256 * 256; };
  const int64_t rows = std::max<int64_t>(I.num_partial_rows, 1);
  const int64_t nitems = static_cast<int64_t>(P.items.size() + P.prefix_items.size());
  I.workspace_bytes = al(std::max<int64_t>(nitems, 1) * static_cast<int64_t>(sizeof(pkvd_work_item))) +
                      al(static_cast<int64_t>(B + 1) * 4) +
                      al(rows * P.desc.heads * P.desc.head_dim_v * 4) + al(rows * P.desc.heads * 4) +
                      al(16);
  return PKVD_OK;
}

// ---------------------------------------------------------------- context parallel

int cp_ranges(int world, int rank, int batch, int page_size, const int32_t* seq_lens,
              int32_t* begin, int32_t* len) {
  if (world < 1 || world > kMaxCpRanks || rank < 0 || rank >= world || batch < 1 ||
      page_size < 1 || !seq_lens || !begin || !len)
    return PKVD_EINVAL;
  for (int b = 0; b < batch; ++b) {
    const int64_t L = seq_lens[b];
    if (L < 0) return PKVD_EINVAL;
    // whole pages per rank, so that every range starts on a page boundary
    const int64_t pages = ceil_div(ceil_div(L, world), page_size);
    const int64_t c = std::max<int64_t>(1, pages) * page_size;
    const int64_t b0 = std::min<int64_t>(L, rank * c);
    const int64_t b1 = std::min<int64_t>(L, (rank + 1) * c);
    begin[b] = static_cast<int32_t>(b0);
    len[b] = static_cast<int32_t>(b1 - b0);
  }
  return PKVD_OK;
}

int cp_shard_desc(const pkvd_plan_desc& in, const int32_t* seq_lens, int world, int rank,
                  pkvd_plan_desc* out, int* family) {
  if (!seq_lens || in.batch < 1) return PKVD_EINVAL;
  std::vector<int32_t> begin(in.batch), len(in.batch);
  int rc = cp_ranges(world, rank, in.batch, in.page_size, seq_lens, begin.data(), len.data());
  if (rc != PKVD_OK) return rc;
  // the full lengths fix the page-table width; the rank's lengths resolve
  // the variant
  pkvd_plan_desc nd;
  rc = normalise_desc(in, seq_lens, &nd, family);
  if (rc != PKVD_OK) return rc;
  if (nd.q_len != 1) return PKVD_EUNSUPPORTED;   // one query token per request
  nd.variant = in.variant;
  return normalise_desc(nd, len.data(), out, family);
}

int plan_layout_cp(const pkvd_plan_desc& in, const int32_t* seq_lens, int world, int rank,
                   PlanLayout* out) {
  pkvd_plan_desc nd;
  int family = 0;
  int rc = cp_shard_desc(in, seq_lens, world, rank, &nd, &family);
  if (rc != PKVD_OK) return rc;
  const int B = in.batch;
  std::vector<int32_t> begin(B), len(B);
  cp_ranges(world, rank, B, in.page_size, seq_lens, begin.data(), len.data());
  rc = plan_layout(nd, len.data(), out);
  if (rc != PKVD_OK) return rc;
  // the items walk absolute token positions of the request's page table
  for (pkvd_work_item& w : out->items) {
    w.tok_begin += begin[w.request];
    w.tok_end += begin[w.request];
    w.query_pos = seq_lens[w.request] - 1;
  }
  return PKVD_OK;
}

}  // namespace pkvd
