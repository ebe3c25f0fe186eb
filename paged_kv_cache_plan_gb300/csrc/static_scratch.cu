// decode_run_static: one decode op that allocates no device memory.
//
// Some callers cannot call cudaMalloc: a host application that owns every
// byte of device memory through its own pool (an inference server, a game or
// plugin host), or code that runs where allocation is forbidden or would
// stall the stream. decode_plan_ex allocates the work list and the split
// partials, so those callers use this entry point instead. It runs the same
// planner and the same stage-1 and merge kernels, but places every piece of
// scratch -- status word, split table, work list, partial outputs and their
// log-sum-exps -- in the fixed array below, which exists once per device that
// loads the library and stays allocated until the process exits.
//
// Limits and sharing:
//   * the scratch a call needs must fit kStaticScratchBytes (16 MiB); a
//     larger problem is rejected with PKVD_ENOMEM before anything is queued;
//   * every call uses the same array, which keeps the last call's contents;
//     calls queued on one stream run one after the other, but calls that
//     overlap on the GPU (different streams, or different host threads
//     without ordering) race on it;
//   * the first call on a device looks up the array's device address (with
//     that device current);
//   * the work list and split table are copied from host memory that the
//     call owns only while it runs, so the call refuses a stream that is
//     being captured (PKVD_EUNSUPPORTED, nothing queued);
//   * device-side page-id checks and wait timeouts are recorded in the
//     array's status word, cleared at the start of each call;
//     decode_run_static_status reads the last call's word (allocating
//     nothing) and reports it like decode_last_device_status.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <new>

#include "../../include/pkvd.h"
#include "kernel_configs.h"
#include "kernels.h"
#include "planner.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;
constexpr double kLog2eStatic = 1.4426950408889634074;

// The scratch. In host code this name is only a stand-in for the symbol, not
// a device address: host code must go through cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_static_scratch on `dev` (current), looked up once.
int scratch_address(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return PKVD_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return PKVD_ECUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch_addr[dev]);
  return PKVD_OK;
}

bool aligned16_static(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int decode_run_static(const pkvd_plan_desc* desc, const int32_t* seq_lens,
                                 const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* page_table, float* out, float* lse,
                                 pkvd_stream_t stream_handle) {
  if (!desc || !out || !lse) return PKVD_EINVAL;
  const cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
  cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &capturing) != cudaSuccess) return PKVD_ECUDA;
  if (capturing != cudaStreamCaptureStatusNone) return PKVD_EUNSUPPORTED;

  pkvd_plan_desc d;
  int family = 0;
  int rc = pkvd::normalise_desc(*desc, seq_lens, &d, &family);
  if (rc != PKVD_OK) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKVD_ECUDA;
  pkvd::KernelEntry s1, s2;
  if (!pkvd::stage1_kernel(d, pkvd::plan_uses_tiles(d, seq_lens), &s1)) return PKVD_EUNSUPPORTED;
  if (d.num_sms == 0 &&
      cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PKVD_ECUDA;
  if (cudaFuncSetAttribute(s1.func, cudaFuncAttributeMaxDynamicSharedMemorySize, s1.smem) !=
      cudaSuccess)
    return PKVD_ECUDA;
  cudaFuncSetAttribute(s1.func, cudaFuncAttributePreferredSharedMemoryCarveout,
                       cudaSharedmemCarveoutMaxShared);
  cudaGetLastError();
  if (d.ctas_per_sm == 0) {
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, s1.func, s1.threads,
                                                      static_cast<size_t>(s1.smem)) !=
            cudaSuccess ||
        occ < 1)
      return PKVD_ECUDA;
    d.ctas_per_sm = occ;
  }

  pkvd::PlanLayout L;
  try {
    rc = pkvd::plan_layout(d, seq_lens, &L);
  } catch (const std::bad_alloc&) {
    return PKVD_ENOMEM;
  }
  if (rc != PKVD_OK) return rc;
  if (!pkvd::stage2_kernel(L.info, L.desc.batch, L.desc.q_len * L.desc.heads,
                           L.desc.head_dim_v, &s2))
    return PKVD_EUNSUPPORTED;   // the plan's merge shape and the kernel table disagree
  const bool any_work = L.info.num_items > 0;
  if (any_work && (!q || !k_pages || !v_pages || !page_table)) return PKVD_EINVAL;
  if (any_work && (!aligned16_static(q) || !aligned16_static(k_pages) ||
                   !aligned16_static(v_pages) || !aligned16_static(page_table)))
    return PKVD_EINVAL;
  if (!aligned16_static(out) || !aligned16_static(lse)) return PKVD_EINVAL;

  // Carve the array: status | split table | work list | partial lse | partial outputs.
  auto al = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = static_cast<size_t>(std::max(1, L.info.num_partial_rows));
  const size_t b_status = al(16);
  const size_t b_split = al(static_cast<size_t>(L.desc.batch + 1) * 4);
  const size_t b_items = al(std::max<size_t>(L.items.size(), 1) * sizeof(pkvd_work_item));
  const size_t b_lpart = al(rows * L.desc.q_len * L.desc.heads * 4);
  const size_t b_opart = al(rows * L.desc.q_len * L.desc.heads * L.desc.head_dim_v * 4);
  if (b_status + b_split + b_items + b_lpart + b_opart > kStaticScratchBytes)
    return PKVD_ENOMEM;

  unsigned char* base = nullptr;
  rc = scratch_address(dev, &base);
  if (rc != PKVD_OK) return rc;
  int32_t* d_status = reinterpret_cast<int32_t*>(base);
  int32_t* d_split = reinterpret_cast<int32_t*>(base + b_status);
  pkvd_work_item* d_items = reinterpret_cast<pkvd_work_item*>(base + b_status + b_split);
  float* d_lpart = reinterpret_cast<float*>(base + b_status + b_split + b_items);
  float* d_opart = reinterpret_cast<float*>(base + b_status + b_split + b_items + b_lpart);

  // The status word must start at zero; the tables are rewritten every call
  // (copies from pageable host memory are staged before these calls return).
  if (cudaMemsetAsync(d_status, 0, 16, stream) != cudaSuccess) return PKVD_ECUDA;
  if (cudaMemcpyAsync(d_split, L.split_base.data(), (L.desc.batch + 1) * sizeof(int32_t),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return PKVD_ECUDA;
  if (any_work && cudaMemcpyAsync(d_items, L.items.data(),
                                  L.items.size() * sizeof(pkvd_work_item),
                                  cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return PKVD_ECUDA;

  if (any_work) {
    pkvd::Stage1Args a{};
    a.q = q;
    a.k = k_pages;
    a.v = v_pages;
    a.page_table = page_table;
    a.items = d_items;
    a.split_base = d_split;
    a.o_part = d_opart;
    a.lse_part = d_lpart;
    a.lse_stride = L.info.num_partial_rows;
    a.status = d_status;
    a.pt_stride = L.desc.max_pages_per_seq;
    a.k_pitch = L.desc.k_row_pitch;
    a.v_pitch = L.desc.v_row_pitch;
    a.num_pool_pages = L.desc.num_pool_pages;
    a.heads = L.desc.heads;
    a.q_len = L.desc.q_len;
    a.kv_heads = L.desc.kv_heads;
    a.page_size = L.desc.page_size;
    a.dv = L.desc.head_dim_v;
    a.scale_log2 = static_cast<float>(static_cast<double>(L.desc.scale) * kLog2eStatic);
    a.checks = L.desc.checks;
    pkvd::KvTensorMaps maps{};
    if (s1.tiles) {
      rc = pkvd::encode_kv_maps(L.desc, k_pages, v_pages, &maps);
      if (rc != PKVD_OK) return rc;
    }
    void* args[] = {&a, &maps};
    if (cudaLaunchKernel(s1.func, dim3(L.info.num_items), dim3(s1.threads), args,
                         static_cast<size_t>(s1.smem), stream) != cudaSuccess)
      return PKVD_ECUDA;
  }
  pkvd::Stage2Args m{};
  m.o_part = d_opart;
  m.lse_part = d_lpart;
  m.lse_stride = L.info.num_partial_rows;
  m.split_base = d_split;
  m.out = out;
  m.lse = lse;
  m.heads = L.desc.q_len * L.desc.heads;
  m.dv = L.desc.head_dim_v;
  m.tiles = L.info.stage2_tiles;
  void* margs[] = {&m};
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(L.desc.batch * m.heads),
                     static_cast<unsigned>(m.tiles));
  cfg.blockDim = dim3(static_cast<unsigned>(L.info.stage2_threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(s2.smem);
  if (cudaFuncSetAttribute(s2.func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(cfg.dynamicSmemBytes)) != cudaSuccess)
    return PKVD_ECUDA;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = any_work ? 1 : 0;
  if (cudaLaunchKernelExC(&cfg, s2.func, margs) != cudaSuccess) return PKVD_ECUDA;
  return PKVD_OK;
}

extern "C" int decode_run_static_status(pkvd_stream_t stream_handle) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKVD_ECUDA;
  unsigned char* base = nullptr;
  int rc = scratch_address(dev, &base);
  if (rc != PKVD_OK) return rc;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream_handle)) != cudaSuccess)
    return PKVD_ECUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, base, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return PKVD_ECUDA;
  if (v != 0 && cudaMemset(base, 0, sizeof(v)) != cudaSuccess) return PKVD_ECUDA;
  if (v & 1) return PKVD_ETIMEOUT;
  if (v & 2) return PKVD_EDEVICE_CHECK;
  return PKVD_OK;
}
