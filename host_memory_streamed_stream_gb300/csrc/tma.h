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
// bf16 row-major [batch][rows][ld] (batch stride `bstride` elements, ld a multiple of 64) seen
// as a 4-D tensor (64 columns, rows, ld / 64 slices, batch) whose third dimension steps 64
// columns (128 bytes). One box (64, box_rows, box_slices, 1) at coordinates (0, row, col / 64, b)
// loads box_rows rows of box_slices consecutive 64-column slices in one operation, laid out in
// shared memory slice after slice, each [box_rows][64] with the 128-byte swizzle. TMA issue cost
// is mostly per box and per 128-byte row, so one box per head-dim tile instead of one per slice
// roughly doubles the load rate of 64-row tiles.
bool tma_map_slices(CUtensorMap* map, const void* base, uint64_t rows, uint64_t batch, int64_t ld, int64_t bstride,
                    uint32_t box_slices, uint32_t box_rows);
}  // namespace mt
