// Host-side construction of TMA tensor maps for token-major attention tensors.
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

// 4-D map over a contiguous 16-bit tensor of `rows` token rows of `heads` x d,
// dims ordered (d, heads, batch entry, token). `nb` is 1 for the packed layout
// [rows, heads, d] (token coordinate = row) and the batch size for the
// sequence-major layout [rows / nb, nb, heads, d] (token i of sequence b at row
// i * nb + b). One load fetches 64 columns x 1 head x 1 batch entry x box_rows
// tokens into shared memory with the 128-byte swizzle; columns >= d and tokens
// past the extent read as zero.
inline bool make_tmap_tokens(CUtensorMap* map, const void* base, int rows, int nb, int heads,
                             int d, bool bf16, int box_rows = 128) {
  auto enc = tmap_encoder();
  if (!enc || nb < 1) return false;
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(heads) * static_cast<cuuint64_t>(d) * 2;
  const int nt = rows / nb;
  cuuint64_t gdim[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(nb), static_cast<cuuint64_t>(nt > 0 ? nt : 1)};
  cuuint64_t gstride[3] = {static_cast<cuuint64_t>(d) * 2, row_bytes, row_bytes * nb};
  cuuint32_t box[4] = {64, 1, 1, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   4, const_cast<void*>(base), gdim, gstride, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace teattn
