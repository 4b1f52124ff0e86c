#include "tma.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace mt {

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
cudaError_t g_err = cudaSuccess;
std::once_flag g_once;

void init() {
  cudaDriverEntryPointQueryResult q{};
  void* fn = nullptr;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
    g_err = (e != cudaSuccess) ? e : cudaErrorSymbolNotFound;
    return;
  }
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
}  // namespace

cudaError_t tma_init() {
  std::call_once(g_once, init);
  return g_err;
}

bool tma_map_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, int64_t ld, uint32_t box_cols,
                uint32_t box_rows) {
  if (tma_init() != cudaSuccess) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tma_map_slices(CUtensorMap* map, const void* base, uint64_t rows, uint64_t batch, int64_t ld, int64_t bstride,
                    uint32_t box_slices, uint32_t box_rows) {
  if (tma_init() != cudaSuccess || ld % 64) return false;
  cuuint64_t dims[4] = {64, rows, static_cast<cuuint64_t>(ld / 64), batch};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(ld) * 2, 128, static_cast<cuuint64_t>(bstride) * 2};
  cuuint32_t box[4] = {64, box_rows, box_slices, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mt
