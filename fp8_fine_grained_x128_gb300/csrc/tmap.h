// tmap.h -- host-side construction of 2-D TMA tensor maps (128-byte swizzle)
// shared by the GEMM kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace fp8fg {

// Tensor map over a row-major [rows][inner] matrix (row stride in bytes),
// boxes of box_inner x box_rows elements, 128-byte swizzle, zero fill
// outside the matrix.  false if the driver's encoder is unavailable or
// rejects the arguments (base / stride alignment, box size).
bool make_map_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *ptr, uint64_t inner, uint64_t rows,
                 uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapL2promotion l2);

}  // namespace fp8fg
