// tma_host.h -- host-side creation of TMA tensor maps (driver entry point
// obtained through the runtime, so the library links no driver stub).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace mla {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Tensor map over a paged latent cache [num_blocks][page_size][576] bf16 with a
// box of 64 columns (128 bytes, 128-byte swizzle) x min(page_size, 64) rows x 1
// page.  Returns false on failure.
inline bool make_kv_tensor_map(CUtensorMap* map, const void* kv, int64_t num_blocks, int32_t page_size) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {576, (cuuint64_t)page_size, (cuuint64_t)num_blocks};
  const cuuint64_t strides[2] = {576 * 2, (cuuint64_t)page_size * 576 * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)(page_size < 64 ? page_size : 64), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(kv), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Tensor maps over an FP8 E4M3 cache [num_blocks][page_size][576] bytes, for
// rows of min(page_size, 64): the wide map reads 128 columns (one 128-byte
// swizzled box: the source of two bf16 64-dim chunks), the tail map the last
// 64 columns (512..575, unswizzled 64-byte rows).
inline bool make_kv8_tensor_maps(CUtensorMap* wide, CUtensorMap* tail, const void* kv, int64_t num_blocks,
                                 int32_t page_size) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {576, (cuuint64_t)page_size, (cuuint64_t)num_blocks};
  const cuuint64_t strides[2] = {576, (cuuint64_t)page_size * 576};
  const cuuint32_t rows = (cuuint32_t)(page_size < 64 ? page_size : 64);
  const cuuint32_t box_w[3] = {128, rows, 1}, box_t[3] = {64, rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(wide, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(kv), dims, strides, box_w, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS &&
         enc(tail, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(kv), dims, strides, box_t, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map over a query part (q_nope or q_pe) viewed as [rows][width] bf16
// with a row stride of `stride` elements (a multiple of 8), box of 64 rows x
// 64 columns (128 bytes, 128-byte swizzle), with a unit outer dimension so
// the 3-D TMA wrapper serves it.  Rows past the end read as zero.
inline bool make_query_tensor_map(CUtensorMap* map, const void* q, int64_t rows, int32_t width, int64_t stride) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc || rows < 1) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)width, (cuuint64_t)rows, 1};
  const cuuint64_t strides[2] = {(cuuint64_t)stride * 2, (cuuint64_t)stride * 2 * (cuuint64_t)rows};
  const cuuint32_t box[3] = {64, 64, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace mla
