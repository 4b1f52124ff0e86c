// Host-side TMA tensor-map encoding (driver entry point looked up once through the runtime,
// so the library does not link libcuda directly).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace mt {

// cudaSuccess once the driver's cuTensorMapEncodeTiled has been found.
cudaError_t tma_init();
// Row-major bf16 matrix of `rows` x `cols` (row stride `ld` elements); box box_cols x box_rows,
// 128-byte swizzle, zero fill out of bounds.
bool tma_map_2d(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, int64_t ld, uint32_t box_cols,
                uint32_t box_rows);
// bf16 tensor [d2][d1][d0] with strides (elements) s1 for d1 and s2 for d2; box b0 x b1 x 1.
bool tma_map_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, int64_t s1, int64_t s2,
                uint32_t b0, uint32_t b1);

}  // namespace mt
