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

// 4-D map over a contiguous tensor of `rows` token rows of `heads` x d elements,
// dims ordered (d, heads, batch entry, token). `nb` is 1 for the packed layout
// [rows, heads, d] (token coordinate = row) and the batch size for the
// sequence-major layout [rows / nb, nb, heads, d] (token i of sequence b at row
// i * nb + b). One load fetches 128 bytes of columns (64 16-bit or 128 8-bit
// elements) x 1 head x 1 batch entry x box_rows tokens into shared memory with the
// 128-byte swizzle; columns >= d and tokens past the extent read as zero.
inline bool make_tmap_tokens_typed(CUtensorMap* map, const void* base, int rows, int nb, int heads,
                                   int d, CUtensorMapDataType type, int elem_bytes, int box_rows) {
  auto enc = tmap_encoder();
  if (!enc || nb < 1) return false;
  const cuuint64_t row_bytes =
      static_cast<cuuint64_t>(heads) * static_cast<cuuint64_t>(d) * static_cast<cuuint64_t>(elem_bytes);
  const int nt = rows / nb;
  cuuint64_t gdim[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(nb), static_cast<cuuint64_t>(nt > 0 ? nt : 1)};
  cuuint64_t gstride[3] = {static_cast<cuuint64_t>(d) * elem_bytes, row_bytes, row_bytes * nb};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / elem_bytes), 1, 1,
                       static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, type, 4, const_cast<void*>(base), gdim, gstride, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 16-bit (bf16 or fp16) tensors.
inline bool make_tmap_tokens(CUtensorMap* map, const void* base, int rows, int nb, int heads,
                             int d, bool bf16, int box_rows = 128) {
  return make_tmap_tokens_typed(map, base, rows, nb, heads, d,
                                bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                                2, box_rows);
}

// 8-bit (e4m3) tensors, moved as raw bytes.
inline bool make_tmap_tokens_u8(CUtensorMap* map, const void* base, int rows, int nb, int heads,
                                int d, int box_rows = 128) {
  return make_tmap_tokens_typed(map, base, rows, nb, heads, d, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                                box_rows);
}

}  // namespace teattn
