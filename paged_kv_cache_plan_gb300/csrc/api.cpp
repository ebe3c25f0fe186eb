// The C ABI of include/pkvd.h: plan creation on the device, the two launches,
// status handling. Argument marshalling only; all arithmetic is in the kernels.
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/pkvd.h"
#include "kernel_configs.h"
#include "kernels.h"
#include "planner.h"

struct pkvd_plan {
  pkvd::PlanLayout layout;
  int device = 0;
  void* dmem = nullptr;
  size_t dbytes = 0;
  pkvd_work_item* d_items = nullptr;
  pkvd_work_item* d_pitems = nullptr;   // grouped shared-prefix items, if any
  int32_t* d_split_base = nullptr;
  float* d_opart = nullptr;
  float* d_lpart = nullptr;
  int32_t* d_status = nullptr;
  pkvd::KernelEntry s1;
  pkvd::KernelEntry s1p;                // kernel of the shared-prefix items
  pkvd::KernelEntry s2;
  int s2_smem = 0;
  float scale_log2 = 0.f;
  // K/V tensor maps of the page-tile path, re-encoded when the pools move
  mutable std::mutex maps_mutex;
  mutable const void* maps_k = nullptr;
  mutable const void* maps_v = nullptr;
  mutable pkvd::KvTensorMaps maps{};
};

namespace {

constexpr double kLog2e = 1.4426950408889634074;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int launch(const pkvd_plan* p, const void* q, const void* k, const void* v,
           const int32_t* page_table, float* out, float* lse, cudaStream_t stream,
           cudaEvent_t ev_begin, cudaEvent_t ev_mid, cudaEvent_t ev_end) {
  if (!p || !out || !lse) return PKVD_EINVAL;
  const pkvd::PlanLayout& L = p->layout;
  const pkvd_plan_desc& d = L.desc;
  const bool any_work = L.info.num_items > 0 || L.info.num_prefix_items > 0;
  if (any_work && (!q || !k || !v || !page_table)) return PKVD_EINVAL;
  if (any_work && (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(page_table)))
    return PKVD_EINVAL;
  if (!aligned16(out) || !aligned16(lse)) return PKVD_EINVAL;

  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) return PKVD_ECUDA;
  if (cur != p->device) return PKVD_EINVAL;

  pkvd::KvTensorMaps maps{};
  if (any_work && p->s1.tiles) {
    std::lock_guard<std::mutex> lock(p->maps_mutex);
    if (p->maps_k != k || p->maps_v != v) {
      const int rc = pkvd::encode_kv_maps(d, k, v, &p->maps);
      if (rc != PKVD_OK) return rc;
      p->maps_k = k;
      p->maps_v = v;
    }
    maps = p->maps;
  }
  if (ev_begin && cudaEventRecord(ev_begin, stream) != cudaSuccess) return PKVD_ECUDA;
  if (any_work) {
    pkvd::Stage1Args a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.page_table = page_table;
    a.items = p->d_items;
    a.split_base = p->d_split_base;
    a.o_part = p->d_opart;
    a.lse_part = p->d_lpart;
    a.lse_stride = L.info.num_partial_rows;
    a.status = p->d_status;
    a.pt_stride = d.max_pages_per_seq;
    a.k_pitch = d.k_row_pitch;
    a.v_pitch = d.v_row_pitch;
    a.num_pool_pages = d.num_pool_pages;
    a.heads = d.heads;
    a.q_len = d.q_len;
    a.kv_heads = d.kv_heads;
    a.page_size = d.page_size;
    a.dv = d.head_dim_v;
    a.scale_log2 = p->scale_log2;
    a.checks = d.checks;
    void* args[] = {&a, &maps};
    if (L.info.num_prefix_items > 0) {
      pkvd::Stage1Args ap = a;
      ap.items = p->d_pitems;
      void* pargs[] = {&ap, &maps};
      if (cudaLaunchKernel(p->s1p.func, dim3(L.info.num_prefix_items), dim3(p->s1p.threads),
                           pargs, static_cast<size_t>(p->s1p.smem), stream) != cudaSuccess)
        return PKVD_ECUDA;
    }
    if (L.info.num_items > 0) {
      // After shared-prefix items the per-request items need nothing they
      // write: programmatic dependent launch lets them take the SMs the
      // prefix grid's last blocks leave idle (they wait for the prefix grid
      // only at their end, so the merge still follows both).
      cudaLaunchConfig_t c1{};
      c1.gridDim = dim3(static_cast<unsigned>(L.info.num_items));
      c1.blockDim = dim3(static_cast<unsigned>(p->s1.threads));
      c1.dynamicSmemBytes = static_cast<size_t>(p->s1.smem);
      c1.stream = stream;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      at[0].val.programmaticStreamSerializationAllowed = 1;
      c1.attrs = at;
      c1.numAttrs = L.info.num_prefix_items > 0 ? 1 : 0;
      if (cudaLaunchKernelExC(&c1, p->s1.func, args) != cudaSuccess) return PKVD_ECUDA;
    }
  }
  if (ev_mid && cudaEventRecord(ev_mid, stream) != cudaSuccess) return PKVD_ECUDA;

  pkvd::Stage2Args m{};
  m.o_part = p->d_opart;
  m.lse_part = p->d_lpart;
  m.lse_stride = L.info.num_partial_rows;
  m.split_base = p->d_split_base;
  m.out = out;
  m.lse = lse;
  m.heads = d.q_len * d.heads;
  m.dv = d.head_dim_v;
  m.tiles = L.info.stage2_tiles;
  void* margs[] = {&m};
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(d.batch * m.heads), static_cast<unsigned>(m.tiles));
  cfg.blockDim = dim3(static_cast<unsigned>(L.info.stage2_threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(p->s2_smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = any_work ? 1 : 0;
  if (cudaLaunchKernelExC(&cfg, p->s2.func, margs) != cudaSuccess) return PKVD_ECUDA;
  if (ev_end && cudaEventRecord(ev_end, stream) != cudaSuccess) return PKVD_ECUDA;
  return PKVD_OK;
}

}  // namespace

extern "C" {

int decode_plan_compute(const pkvd_plan_desc* desc, const int32_t* seq_lens,
                        pkvd_plan_info* info, pkvd_work_item* items, int64_t capacity) {
  if (!desc || !info) return PKVD_EINVAL;
  pkvd::PlanLayout L;
  int rc;
  try {
    rc = pkvd::plan_layout(*desc, seq_lens, &L);
  } catch (const std::bad_alloc&) {
    return PKVD_ENOMEM;
  }
  if (rc != PKVD_OK) return rc;
  *info = L.info;
  if (items) {
    if (capacity < L.info.num_items) return PKVD_EINVAL;
    std::memcpy(items, L.items.data(), L.items.size() * sizeof(pkvd_work_item));
  }
  return PKVD_OK;
}

}  // extern "C"

namespace {

// Plan creation shared by decode_plan_ex, decode_plan_prefix (prefix arrays
// non-null) and decode_plan_cp (cp_world > 0: the token range of rank
// cp_rank).
int make_plan(pkvd_plan** out, const pkvd_plan_desc* desc, const int32_t* seq_lens,
              const int32_t* prefix_group, const int32_t* prefix_len, int cp_world = 0,
              int cp_rank = 0) {
  if (!out || !desc) return PKVD_EINVAL;
  *out = nullptr;
  const bool prefix = prefix_group != nullptr;
  const bool cp = cp_world > 0;
  // the per-request items' description (a shared-prefix plan resolves their
  // variant on the private lengths, a context-parallel plan on its rank's)
  pkvd_plan_desc d;
  int family = 0;
  int rc = prefix ? pkvd::prefix_private_desc(*desc, seq_lens, prefix_group, prefix_len, &d,
                                              &family)
           : cp   ? pkvd::cp_shard_desc(*desc, seq_lens, cp_world, cp_rank, &d, &family)
                  : pkvd::normalise_desc(*desc, seq_lens, &d, &family);
  if (rc != PKVD_OK) return rc;
  // the lengths the items cover (page-tile eligibility depends on them)
  std::vector<int32_t> item_lens(seq_lens, seq_lens + desc->batch);
  if (cp) {
    std::vector<int32_t> begin(desc->batch);
    pkvd::cp_ranges(cp_world, cp_rank, desc->batch, desc->page_size, seq_lens, begin.data(),
                    item_lens.data());
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKVD_ECUDA;
  pkvd::KernelEntry s1, s1p, s2;
  if (!pkvd::stage1_kernel(d, !prefix && pkvd::plan_uses_tiles(d, item_lens.data()), &s1))
    return PKVD_EUNSUPPORTED;
  if (prefix) {
    if (family != PKVD_FAMILY_MLA || !pkvd::mla_tc_kernel(d.dtype, false, &s1p)) return PKVD_EUNSUPPORTED;
    if (cudaFuncSetAttribute(s1p.func, cudaFuncAttributeMaxDynamicSharedMemorySize, s1p.smem) !=
        cudaSuccess)
      return PKVD_ECUDA;
  }
  if (d.num_sms == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PKVD_ECUDA;
    d.num_sms = sms;
  }
  if (cudaFuncSetAttribute(s1.func, cudaFuncAttributeMaxDynamicSharedMemorySize, s1.smem) !=
      cudaSuccess)
    return PKVD_ECUDA;
  // Ask for the largest shared-memory carveout so that several stage-1
  // blocks fit on an SM when their pipelines allow it.
  cudaFuncSetAttribute(s1.func, cudaFuncAttributePreferredSharedMemoryCarveout,
                       cudaSharedmemCarveoutMaxShared);
  cudaGetLastError();
  if (d.ctas_per_sm == 0) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, s1.func, s1.threads,
                                                      static_cast<size_t>(s1.smem)) !=
        cudaSuccess)
      return PKVD_ECUDA;
    if (occ < 1) return PKVD_EUNSUPPORTED;
    d.ctas_per_sm = occ;
  }

  pkvd_plan* p = new (std::nothrow) pkvd_plan;
  if (!p) return PKVD_ENOMEM;
  try {
    rc = prefix ? pkvd::plan_layout_prefix(d, seq_lens, prefix_group, prefix_len, &p->layout)
         : cp   ? pkvd::plan_layout_cp(d, seq_lens, cp_world, cp_rank, &p->layout)
                : pkvd::plan_layout(d, seq_lens, &p->layout);
  } catch (const std::bad_alloc&) {
    rc = PKVD_ENOMEM;
  }
  if (rc != PKVD_OK) {
    delete p;
    return rc;
  }
  p->device = dev;
  const pkvd::PlanLayout& L = p->layout;
  if (!pkvd::stage2_kernel(L.info, L.desc.batch, L.desc.q_len * L.desc.heads,
                           L.desc.head_dim_v, &s2)) {
    delete p;   // the plan's merge shape and the kernel table disagree
    return PKVD_EUNSUPPORTED;
  }
  p->s1 = s1;
  p->s1p = s1p;
  p->s2 = s2;
  p->s2_smem = s2.smem;
  if (cudaFuncSetAttribute(s2.func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           p->s2_smem) != cudaSuccess) {
    delete p;
    return PKVD_ECUDA;
  }
  p->scale_log2 = static_cast<float>(static_cast<double>(L.desc.scale) * kLog2e);

  // one device allocation, carved in 256-byte aligned pieces
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = static_cast<size_t>(std::max(1, L.info.num_partial_rows));
  const size_t n_items = L.items.size() + L.prefix_items.size();
  const size_t b_items = al(std::max<size_t>(n_items, 1) * sizeof(pkvd_work_item));
  const size_t b_split = al(static_cast<size_t>(L.desc.batch + 1) * 4);
  const size_t b_opart = al(rows * L.desc.q_len * L.desc.heads * L.desc.head_dim_v * 4);
  const size_t b_lpart = al(rows * L.desc.q_len * L.desc.heads * 4);
  const size_t b_status = al(16);
  p->dbytes = b_items + b_split + b_opart + b_lpart + b_status;
  if (cudaMalloc(&p->dmem, p->dbytes) != cudaSuccess) {
    cudaGetLastError();
    delete p;
    return PKVD_ENOMEM;
  }
  char* base = static_cast<char*>(p->dmem);
  p->d_items = reinterpret_cast<pkvd_work_item*>(base);
  p->d_pitems = p->d_items + L.items.size();
  p->d_split_base = reinterpret_cast<int32_t*>(base + b_items);
  p->d_opart = reinterpret_cast<float*>(base + b_items + b_split);
  p->d_lpart = reinterpret_cast<float*>(base + b_items + b_split + b_opart);
  p->d_status = reinterpret_cast<int32_t*>(base + b_items + b_split + b_opart + b_lpart);
  bool ok = true;
  if (!L.items.empty())
    ok = ok && cudaMemcpy(p->d_items, L.items.data(), L.items.size() * sizeof(pkvd_work_item),
                          cudaMemcpyHostToDevice) == cudaSuccess;
  if (!L.prefix_items.empty())
    ok = ok && cudaMemcpy(p->d_pitems, L.prefix_items.data(),
                          L.prefix_items.size() * sizeof(pkvd_work_item),
                          cudaMemcpyHostToDevice) == cudaSuccess;
  ok = ok && cudaMemcpy(p->d_split_base, L.split_base.data(), (L.desc.batch + 1) * 4,
                        cudaMemcpyHostToDevice) == cudaSuccess;
  ok = ok && cudaMemset(p->d_status, 0, 16) == cudaSuccess;
  if (!ok) {
    cudaFree(p->dmem);
    delete p;
    return PKVD_ECUDA;
  }
  *out = p;
  return PKVD_OK;
}

}  // namespace

extern "C" {

int decode_plan_ex(pkvd_plan** out, const pkvd_plan_desc* desc, const int32_t* seq_lens) {
  return make_plan(out, desc, seq_lens, nullptr, nullptr);
}

int decode_plan_prefix(pkvd_plan** out, const pkvd_plan_desc* desc, const int32_t* seq_lens,
                       const int32_t* prefix_group, const int32_t* prefix_len) {
  if (!prefix_group || !prefix_len) return PKVD_EINVAL;
  return make_plan(out, desc, seq_lens, prefix_group, prefix_len);
}

int decode_plan_prefix_compute(const pkvd_plan_desc* desc, const int32_t* seq_lens,
                               const int32_t* prefix_group, const int32_t* prefix_len,
                               pkvd_plan_info* info, pkvd_work_item* items, int64_t capacity) {
  if (!desc || !info) return PKVD_EINVAL;
  pkvd::PlanLayout L;
  int rc;
  try {
    rc = pkvd::plan_layout_prefix(*desc, seq_lens, prefix_group, prefix_len, &L);
  } catch (const std::bad_alloc&) {
    return PKVD_ENOMEM;
  }
  if (rc != PKVD_OK) return rc;
  *info = L.info;
  if (items) {
    const size_t n = L.prefix_items.size() + L.items.size();
    if (capacity < static_cast<int64_t>(n)) return PKVD_EINVAL;
    std::memcpy(items, L.prefix_items.data(), L.prefix_items.size() * sizeof(pkvd_work_item));
    std::memcpy(items + L.prefix_items.size(), L.items.data(),
                L.items.size() * sizeof(pkvd_work_item));
  }
  return PKVD_OK;
}

int decode_plan_cp(pkvd_plan** out, const pkvd_plan_desc* desc, const int32_t* seq_lens,
                   int world, int rank) {
  if (world < 1) return PKVD_EINVAL;
  return make_plan(out, desc, seq_lens, nullptr, nullptr, world, rank);
}

int decode_plan_cp_compute(const pkvd_plan_desc* desc, const int32_t* seq_lens, int world,
                           int rank, pkvd_plan_info* info, pkvd_work_item* items,
                           int64_t capacity) {
  if (!desc || !info) return PKVD_EINVAL;
  pkvd::PlanLayout L;
  int rc;
  try {
    rc = pkvd::plan_layout_cp(*desc, seq_lens, world, rank, &L);
  } catch (const std::bad_alloc&) {
    return PKVD_ENOMEM;
  }
  if (rc != PKVD_OK) return rc;
  *info = L.info;
  if (items) {
    if (capacity < L.info.num_items) return PKVD_EINVAL;
    std::memcpy(items, L.items.data(), L.items.size() * sizeof(pkvd_work_item));
  }
  return PKVD_OK;
}

int decode_cp_ranges(int world, int rank, int batch, int page_size, const int32_t* seq_lens,
                     int32_t* begin, int32_t* len) {
  return pkvd::cp_ranges(world, rank, batch, page_size, seq_lens, begin, len);
}

int decode_merge_ranks(int n_ranks, int64_t rows, int dv, const float* o_parts,
                       const float* lse_parts, float* out, float* lse, pkvd_stream_t stream) {
  if (n_ranks < 1 || n_ranks > pkvd::kMaxCpRanks || rows < 0 || rows > 0x7fffffff)
    return PKVD_EINVAL;
  if (dv < 4 || dv > 512 || dv % 4 != 0) return PKVD_EUNSUPPORTED;
  if (rows > 0 && (!o_parts || !lse_parts || !out || !lse)) return PKVD_EINVAL;
  if (rows > 0 && (!aligned16(o_parts) || !aligned16(out) ||
                   (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
                   (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return PKVD_EINVAL;
  return pkvd::launch_merge_ranks(n_ranks, rows, dv, o_parts, lse_parts, out, lse,
                                  reinterpret_cast<cudaStream_t>(stream));
}

int decode_plan(pkvd_plan** out, int batch, int heads, int kv_heads, int head_dim, int page_size,
                const int32_t* seq_lens, int splits) {
  pkvd_plan_desc d{};
  d.batch = batch;
  d.heads = heads;
  d.kv_heads = kv_heads;
  d.head_dim = head_dim;
  d.page_size = page_size;
  d.splits = splits;
  d.dtype = PKVD_BF16;
  return decode_plan_ex(out, &d, seq_lens);
}

int decode_run(const pkvd_plan* plan, const void* q, const void* k_pages, const void* v_pages,
               const int32_t* page_table, float* out, float* lse, pkvd_stream_t stream) {
  return launch(plan, q, k_pages, v_pages, page_table, out, lse,
                reinterpret_cast<cudaStream_t>(stream), nullptr, nullptr, nullptr);
}

int decode_run_timed(const pkvd_plan* plan, const void* q, const void* k_pages,
                     const void* v_pages, const int32_t* page_table, float* out, float* lse,
                     pkvd_stream_t stream, pkvd_event_t ev_begin, pkvd_event_t ev_mid,
                     pkvd_event_t ev_end) {
  return launch(plan, q, k_pages, v_pages, page_table, out, lse,
                reinterpret_cast<cudaStream_t>(stream), reinterpret_cast<cudaEvent_t>(ev_begin),
                reinterpret_cast<cudaEvent_t>(ev_mid), reinterpret_cast<cudaEvent_t>(ev_end));
}

int decode_plan_destroy(pkvd_plan* plan) {
  if (!plan) return PKVD_OK;
  int rc = PKVD_OK;
  int cur = 0;
  if (cudaGetDevice(&cur) == cudaSuccess && cur != plan->device) cudaSetDevice(plan->device);
  if (cudaDeviceSynchronize() != cudaSuccess) rc = PKVD_ECUDA;
  if (plan->dmem && cudaFree(plan->dmem) != cudaSuccess) rc = PKVD_ECUDA;
  if (cur != plan->device) cudaSetDevice(cur);
  delete plan;
  return rc;
}

size_t decode_workspace_bytes(const pkvd_plan* plan) { return plan ? plan->dbytes : 0; }

int decode_plan_query(const pkvd_plan* plan, pkvd_plan_info* info) {
  if (!plan || !info) return PKVD_EINVAL;
  *info = plan->layout.info;
  info->workspace_bytes = static_cast<int64_t>(plan->dbytes);
  return PKVD_OK;
}

int decode_last_device_status(const pkvd_plan* plan, pkvd_stream_t stream) {
  if (!plan) return PKVD_EINVAL;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKVD_ECUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, plan->d_status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return PKVD_ECUDA;
  if (v != 0 && cudaMemset(plan->d_status, 0, 4) != cudaSuccess) return PKVD_ECUDA;
  if (v & 1) return PKVD_ETIMEOUT;
  if (v & 2) return PKVD_EDEVICE_CHECK;
  return PKVD_OK;
}

const char* decode_status_string(int status) {
  switch (status) {
    case PKVD_OK: return "ok";
    case PKVD_EINVAL: return "invalid argument";
    case PKVD_EUNSUPPORTED: return "unsupported shape or dtype";
    case PKVD_ECUDA: return "CUDA runtime error";
    case PKVD_ENOMEM: return "out of memory";
    case PKVD_EDEVICE_CHECK: return "a kernel page-id check failed (an id outside the pool, or shared-prefix pages that differ)";
    case PKVD_ETIMEOUT: return "a kernel pipeline wait timed out";
    default: return "unknown status";
  }
}

}  // extern "C"
