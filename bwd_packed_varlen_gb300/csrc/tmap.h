// Host-side construction of TMA tensor maps for THD tensors.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace teattn {

// cuTensorMapEncodeTiled, resolved once through the runtime (no -lcuda needed).
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

// 3-D map over a contiguous [rows, heads, d] 16-bit tensor, dims ordered
// (d, heads, rows). One load fetches a box of 64 columns x 1 head x 128 rows
// into shared memory with the 128-byte swizzle; columns >= d and rows >= `rows`
// read as zero.
inline bool make_tmap_thd(CUtensorMap* map, const void* base, int rows, int heads, int d,
                          bool bf16, int box_rows = 128) {
  auto enc = tmap_encoder();
  if (!enc) return false;
  cuuint64_t gdim[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(rows > 0 ? rows : 1)};
  cuuint64_t gstride[2] = {static_cast<cuuint64_t>(d) * 2,
                           static_cast<cuuint64_t>(heads) * static_cast<cuuint64_t>(d) * 2};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   3, const_cast<void*>(base), gdim, gstride, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace teattn
