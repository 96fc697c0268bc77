// Host-side TMA tensor-map encoding (driver entry point fetched at run time,
// so the library loads on machines without a CUDA driver).
#include <cudaTypedefs.h>
#include <cuda.h>
#include <mutex>

#include "tmap.h"

namespace mla {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
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

bool make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t ld_elems, uint32_t box_cols, uint32_t box_rows, bool weights) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld_elems * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  weights ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static bool encode_pool(CUtensorMap* tm, const void* base, cuuint32_t rank, const cuuint64_t* dims,
                        const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_pool_blocks(CUtensorMap* tm, const void* base, uint64_t rows, uint32_t box_rows,
                           uint32_t nb) {
  const cuuint64_t dims[3] = {64, rows, 9};
  const cuuint64_t strides[2] = {1152, 128};
  const cuuint32_t box[3] = {64, box_rows, nb};
  return encode_pool(tm, base, 3, dims, strides, box);
}

bool make_tmap_pool_slabs(CUtensorMap* tm, const void* base, uint64_t rows, uint32_t nb) {
  const cuuint64_t dims[4] = {64, 32, 9, rows / 32};
  const cuuint64_t strides[3] = {1152, 128, 32 * 1152};
  const cuuint32_t box[4] = {64, 32, nb, 2};
  return encode_pool(tm, base, 4, dims, strides, box);
}

bool make_tmap_u8_2d(CUtensorMap* tm, const void* base, uint64_t rows, uint64_t row_bytes,
                     uint32_t box_bytes, uint32_t box_rows, bool swizzle128) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_bytes, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mla
