// Host side of the launches shared by the planned and the allocation-free
// entry points: stage-1 kernel lookup and the K/V tensor maps of the
// page-tile path.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "kernel_configs.h"
#include "kernels.h"

namespace pkvd {

bool stage1_kernel(const pkvd_plan_desc& d, bool tiles, KernelEntry* e) {
  // a GQA item covers the q_len x group (query token, head) rows of a KV head
  const int q_len = d.q_len > 0 ? d.q_len : 1;
  const int group = d.heads / d.kv_heads;
  const bool causal = q_len > 1;
  switch (d.variant) {
    case PKVD_VARIANT_GQA_FMA:
      return !causal && gqa_fma_kernel(d.dtype, d.head_dim, group, tiles, e);
    case PKVD_VARIANT_GQA_MMA:
      return gqa_mma_kernel(d.dtype, d.head_dim, q_len * group, tiles, causal, e);
    case PKVD_VARIANT_MLA_MMA: return !tiles && mla_mma_kernel(d.dtype, causal, e);
    case PKVD_VARIANT_MLA_TC: return !tiles && mla_tc_kernel(d.dtype, causal, e);
    default: return false;
  }
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

int encode_one(PFN_cuTensorMapEncodeTiled_v12000 fn, const pkvd_plan_desc& d, const void* base,
               int64_t pitch_elems, int cols, CUtensorMap* out) {
  // rows of the pool viewed as [pages * kv_heads * page_size, pitch]
  const uint64_t rows = d.num_pool_pages > 0
                            ? static_cast<uint64_t>(d.num_pool_pages) * d.kv_heads * d.page_size
                            : 0x7fffffffull;
  if (rows > 0x7fffffffull) return PKVD_EUNSUPPORTED;   // row coordinates are int32
  cuuint64_t gdim[3] = {64, rows, static_cast<cuuint64_t>(cols / 64)};
  cuuint64_t gstride[2] = {static_cast<cuuint64_t>(pitch_elems) * 2, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kGqaBlockTokens),
                       static_cast<cuuint32_t>(cols / 64)};
  cuuint32_t estride[3] = {1, 1, 1};
  const CUresult r =
      fn(out, d.dtype == PKVD_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
         3, const_cast<void*>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKVD_OK : PKVD_ECUDA;
}

}  // namespace

int encode_tiled_map(int dtype, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box, CUtensorMap* out) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return PKVD_ECUDA;
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bx[5], estride[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bx[i] = box[i];
    estride[i] = 1;
    if (i > 0) gstride[i - 1] = strides[i - 1];
  }
  const CUresult r =
      fn(out, dtype == PKVD_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
         static_cast<cuuint32_t>(rank), const_cast<void*>(base), gdim, gstride, bx, estride,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKVD_OK : PKVD_ECUDA;
}

int encode_kv_maps(const pkvd_plan_desc& d, const void* k, const void* v, KvTensorMaps* out) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return PKVD_ECUDA;
  std::memset(out, 0, sizeof(*out));
  int rc = encode_one(fn, d, k, d.k_row_pitch, d.head_dim, &out->k);
  if (rc == PKVD_OK) rc = encode_one(fn, d, v, d.v_row_pitch, d.head_dim_v, &out->v);
  return rc;
}

}  // namespace pkvd
